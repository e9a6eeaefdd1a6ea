"""Seeded synthetic inputs for the attention backward-over-backward workloads.

This module only draws random numbers and holds the named workload shapes.  It
contains none of the method's arithmetic, so both the CUDA path and the fp64
CPU oracle take their inputs from here without sharing any computation.

Recipe (the pages benchmark an isolated attention layer on synthetic tensors):

* one CPU ``torch.Generator`` seeded with ``seed`` (a CUDA one, same recipe,
  for the edge-case shapes with hundreds of thousands of heads, whose CPU
  draw would take minutes);
* draws in the fixed order Q, K, V, dO, U_Q, U_K, U_V, each of shape
  ``[B, H, N, d]`` (contiguous, row-major); rectangular workloads draw the
  key-side tensors K, V, U_K, U_V with ``Nk`` rows (the same draw order);
* ``dist="unit"``: all seven tensors ~ N(0, 1) (the tiny fp32 workload);
* ``dist="scaled"``: Q, K, V ~ N(0, 1) / d**0.25 so that Q K^T has unit
  variance; dO, U_Q, U_K, U_V ~ N(0, 1);
* grouped-query workloads draw K, V, U_K, U_V with ``Hkv`` heads (the
  same draw order);
* ``peaked_k_rows``: for every (b, h) pick floor(0.05 N_k) distinct key rows
  with the same generator (after the seven draws) and multiply them by 4,
  which makes some softmax rows peaked;
* ``stress``: Q, K ~ N(0, 1) (unscaled), so the scaled scores tau Q K^T have
  unit variance and the x4 key rows are truly peaked;
* bf16 workloads round the fp32 draws to bf16 (round to nearest even) as the
  last step; the oracle then reads the bf16 values exactly, as fp64.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

NAMES = ("Q", "K", "V", "dO", "UQ", "UK", "UV")
KV_NAMES = ("K", "V", "UK", "UV")


@dataclass(frozen=True)
class Workload:
    """A named problem shape: batch B, heads H, query rows N, head dim d
    (key rows Nk and key/value heads Hkv where they differ)."""

    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str  # "f32" or "bf16"
    dist: str = "scaled"  # "unit" or "scaled"
    peaked_k_rows: bool = False
    stress: bool = False
    seed: int = 0
    causal: bool = False
    Hkv: int = 0  # key/value heads (grouped-query attention); 0 means H
    Nk: int = 0  # key rows (rectangular attention); 0 means N

    @property
    def kv_heads(self) -> int:
        return self.Hkv if self.Hkv else self.H

    @property
    def kv_len(self) -> int:
        return self.Nk if self.Nk else self.N

    @property
    def pairs(self) -> int:
        """(query, key) pairs the softmax sees per head: N Nk, or under the
        causal mask (key j visible from query i when j <= i) the count of
        pairs with j <= i."""
        n, nk = self.N, self.kv_len
        if not self.causal:
            return n * nk
        m = min(n, nk)
        return m * (m + 1) // 2 + (n - m) * nk

    @property
    def tau(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """Fixed GEMM list of both passes: 19 GEMMs of 2 d flops per visible
        (query, key) pair, i.e. 38 N^2 d per head without a mask."""
        return 38.0 * self.pairs * self.d * self.B * self.H


# The five workloads of the isolated-layer benchmark (non-causal).
TINY_F32 = Workload("tiny_f32_B1_H1_N128_d64", 1, 1, 128, 64, "f32", dist="unit")
GPT2_LAYER = Workload("gpt2_layer_B4_H12_N1024_d64", 4, 12, 1024, 64, "bf16")
MID_LENGTH = Workload("mid_B1_H12_N8192_d64", 1, 12, 8192, 64, "bf16")
MID_LENGTH_PEAKED = Workload("mid_peaked_B1_H12_N8192_d64", 1, 12, 8192, 64, "bf16",
                             peaked_k_rows=True)
MID_LENGTH_STRESS = Workload("mid_stress_B1_H12_N8192_d64", 1, 12, 8192, 64, "bf16",
                             peaked_k_rows=True, stress=True)
LONG_CONTEXT = Workload("long_B1_H4_N65536_d64", 1, 4, 65536, 64, "bf16")
EXTREME_D64 = Workload("extreme_B1_H1_N262144_d64", 1, 1, 262144, 64, "bf16")
EXTREME_D128 = Workload("extreme_B1_H1_N131072_d128", 1, 1, 131072, 128, "bf16")

# Causal shapes of the pages' isolated-layer timing table (B=4, H=12, bf16).
CAUSAL_N4096 = Workload("causal_B4_H12_N4096_d64", 4, 12, 4096, 64, "bf16", causal=True)
CAUSAL_N8192 = Workload("causal_B4_H12_N8192_d64", 4, 12, 8192, 64, "bf16", causal=True)
CAUSAL_N16384 = Workload("causal_B4_H12_N16384_d64", 4, 12, 16384, 64, "bf16", causal=True)
CAUSAL_N16384_D128 = Workload("causal_B4_H12_N16384_d128", 4, 12, 16384, 128, "bf16",
                              causal=True)
CAUSAL_N32768_D128 = Workload("causal_B4_H12_N32768_d128", 4, 12, 32768, 128, "bf16",
                              causal=True)
CAUSAL_N65536_D128 = Workload("causal_B4_H12_N65536_d128", 4, 12, 65536, 128, "bf16",
                              causal=True)
# Grouped-query attention: 12 query heads share 4 key/value heads (and a
# multi-query variant with one shared head).
GQA_N8192 = Workload("gqa_B1_H12_Hkv4_N8192_d64", 1, 12, 8192, 64, "bf16", Hkv=4)
MQA_N8192 = Workload("mqa_B1_H12_Hkv1_N8192_d64", 1, 12, 8192, 64, "bf16", Hkv=1)
# Rectangular attention: fewer queries than keys and the reverse.
RECT_Q4096_K16384 = Workload("rect_B1_H8_Nq4096_Nk16384_d64", 1, 8, 4096, 64, "bf16", Nk=16384)
RECT_Q16384_K4096 = Workload("rect_B1_H8_Nq16384_Nk4096_d64", 1, 8, 16384, 64, "bf16", Nk=4096)
# Long query streams against a few key blocks: pass 2's loop as long as in the
# long-context and extreme workloads (1024 / 4096 query tiles per key block),
# with few enough keys that the oracle covers every key column.
LONGLOOP_D64 = Workload("longloop_B1_H4_Nq65536_Nk256_d64", 1, 4, 65536, 64, "bf16", Nk=256)
LONGLOOP_EXTREME_D64 = Workload("longloop_B1_H1_Nq262144_Nk512_d64", 1, 1, 262144, 64, "bf16",
                                Nk=512)
LONGLOOP_D128 = Workload("longloop_B1_H1_Nq131072_Nk256_d128", 1, 1, 131072, 128, "bf16",
                         Nk=256)
# The rest of the throughput-vs-length curve (d = 64, non-causal): N = 2048 .. 32768.
CURVE_N2048 = Workload("curve_B4_H12_N2048_d64", 4, 12, 2048, 64, "bf16")
CURVE_N4096 = Workload("curve_B2_H12_N4096_d64", 2, 12, 4096, 64, "bf16")
CURVE_N16384 = Workload("curve_B1_H8_N16384_d64", 1, 8, 16384, 64, "bf16")
CURVE_N32768 = Workload("curve_B1_H4_N32768_d64", 1, 4, 32768, 64, "bf16")
# A mid-size case for detailed profiles: inputs (~0.3 GB) larger than L2.
PROFILE = Workload("profile_B1_H8_N32768_d64", 1, 8, 32768, 64, "bf16")
# d = 128 kernels under ncu: one head (no head-group streams), inputs 176 MiB > L2.
PROFILE_D128 = Workload("profile_B1_H1_N98304_d128", 1, 1, 98304, 128, "bf16")

WORKLOADS = {w.name: w for w in (TINY_F32, GPT2_LAYER, MID_LENGTH, MID_LENGTH_PEAKED,
                                 MID_LENGTH_STRESS, LONG_CONTEXT, EXTREME_D64, EXTREME_D128,
                                 CAUSAL_N4096, CAUSAL_N8192, CAUSAL_N16384, CAUSAL_N16384_D128,
                                 CAUSAL_N32768_D128, CAUSAL_N65536_D128, GQA_N8192,
                                 MQA_N8192,
                                 RECT_Q4096_K16384, RECT_Q16384_K4096, LONGLOOP_D64,
                                 LONGLOOP_EXTREME_D64, LONGLOOP_D128, PROFILE, PROFILE_D128,
                                 CURVE_N2048, CURVE_N4096, CURVE_N16384, CURVE_N32768)}


def make_inputs(w: Workload, device: str = "cpu") -> dict[str, torch.Tensor]:
    """Draw the seven input tensors of ``w`` (on the CPU by default).

    Returns fp32 tensors for ``dtype="f32"`` and bf16 tensors for
    ``dtype="bf16"``, all contiguous: ``[B, H, N, d]`` for Q, dO, U_Q and
    ``[B, Hkv, Nk, d]`` for K, V, U_K, U_V.  ``device="cuda"`` draws the same
    recipe with a CUDA generator (other values than the CPU draw, same
    distribution), for shapes whose CPU draw would take minutes; the oracle
    then reads the drawn values back.
    """
    if device != "cpu" and w.peaked_k_rows:
        raise ValueError("peaked key rows are drawn on the CPU only")
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    shape = (w.B, w.H, w.N, w.d)
    kv_shape = (w.B, w.kv_heads, w.kv_len, w.d)  # K, V, U_K, U_V (grouped-query, rectangular)
    out = {}
    for name in NAMES:
        out[name] = torch.randn(kv_shape if name in KV_NAMES else shape, generator=g,
                                dtype=torch.float32, device=device)
    if w.dist == "scaled":
        s = w.d ** -0.25
        for name in ("Q", "K", "V"):
            if w.stress and name in ("Q", "K"):
                continue
            out[name].mul_(s)
    elif w.dist != "unit":
        raise ValueError(f"unknown dist {w.dist!r}")
    if w.peaked_k_rows:
        n_peak = int(math.floor(0.05 * w.kv_len))
        for b in range(w.B):
            for h in range(w.kv_heads):
                idx = torch.randperm(w.kv_len, generator=g)[:n_peak]
                out["K"][b, h, idx, :] *= 4.0
    if w.dtype == "bf16":
        out = {k: v.to(torch.bfloat16) for k, v in out.items()}
    elif w.dtype != "f32":
        raise ValueError(f"unknown dtype {w.dtype!r}")
    return out


def small_workload(B: int, H: int, N: int, d: int, dtype: str, seed: int = 0,
                   dist: str | None = None, **kw) -> Workload:
    """An ad-hoc shape for parity and edge-case tests."""
    if dist is None:
        dist = "unit" if dtype == "f32" else "scaled"
    nk = f"_Nk{kw['Nk']}" if kw.get("Nk") else ""
    return Workload(f"adhoc_B{B}_H{H}_N{N}{nk}_d{d}_{dtype}", B, H, N, d, dtype, dist=dist,
                    seed=seed, **kw)


def as_float64_numpy(t: torch.Tensor):
    """Exact fp64 copy (bf16 and fp32 values are representable in fp64)."""
    return t.detach().to("cpu").to(torch.float64).numpy()
