"""Shared helpers of the parity tests: run the CUDA path through the C ABI on
seeded inputs and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

from exact_second_order_gb300 import flashbob as fb
from exact_second_order_gb300.inputs import KV_NAMES, NAMES, as_float64_numpy, make_inputs
from oracle import bob as orc

# Gates: relative Frobenius error on every output.
TOL = {"f32": 1e-4, "bf16": 2e-2}
MAT_KEYS = ("dQt", "dKt", "dVt", "ddOt")
ROW_KEYS = ("alpha", "E")

# Achieved errors of this session, (check, output, error) in the order the
# tests ran; written as JSON lines to $FLASHBOB_PARITY_LOG at the end of the
# session (tests/conftest.py) so that the margins under the gates are kept.
RECORDED: list[tuple[str, str, float]] = []


def record(check: str, errs: dict) -> dict:
    for k, v in errs.items():
        RECORDED.append((check, k, float(v)))
    return errs


def rel_fro(got, ref) -> float:
    """Relative Frobenius error; where the exact result is zero (the oracle's
    norm is at rounding level, e.g. d~Q, d~K, d~V at N = 1) the error is the
    largest absolute deviation instead."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(got - ref)
    if den <= 1e-10 * np.sqrt(max(ref.size, 1)):
        return float(np.abs(got - ref).max()) if ref.size else 0.0
    return num / den


def run_cuda(w, stream=None, fill_nan=True):
    """Inputs of workload ``w`` (CPU tensors) and the device results of
    flashbob_prep + flashbob_bob."""
    x = make_inputs(w)
    dev = {k: v.cuda() for k, v in x.items()}
    O, L, D = fb.prep(dev["Q"], dev["K"], dev["V"], dev["dO"], w.tau, causal=w.causal,
                      stream=stream)
    out = fb.alloc_bob_outputs(dev["Q"], fill=float("nan") if fill_nan else None, K=dev["K"])
    fb.bob(dev["Q"], dev["K"], dev["V"], O, dev["dO"], L, D, dev["UQ"], dev["UK"], dev["UV"],
           w.tau, out=out, causal=w.causal, stream=stream)
    torch.cuda.synchronize()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    return x, dev, {"O": O, "L": L, "D": D}, out


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def oracle_inputs(x):
    return [as_float64_numpy(x[k]) for k in NAMES]


def full_oracle_errors(w, x, state, out, heads=None):
    """Relative Frobenius errors of every output against the full oracle, on
    all (b, h) query heads or the listed ones; d~K and d~V are compared on
    the key/value heads those query heads use (grouped-query attention: a
    shared head's reference sums every query head of its group)."""
    args = oracle_inputs(x)
    Q, K, V, dO, UQ, UK, UV = args
    G = w.H // w.kv_heads
    qheads = heads if heads is not None else [(b, h) for b in range(w.B) for h in range(w.H)]
    kvheads = sorted({(b, h // G) for b, h in qheads})
    ref_q = {k: {} for k in ("dQt", "ddOt", "alpha", "E", "L", "D")}
    ref_k = {"dKt": {}, "dVt": {}}
    for b, g in kvheads:
        hs = slice(g * G, (g + 1) * G)
        r = orc.bob_gqa(Q[b, hs], K[b, g:g + 1], V[b, g:g + 1], dO[b, hs], UQ[b, hs],
                        UK[b, g:g + 1], UV[b, g:g + 1], w.tau, w.causal)
        for k in ref_q:
            for i in range(G):
                ref_q[k][(b, g * G + i)] = r[k][i]
        for k in ref_k:
            ref_k[k][(b, g)] = r[k][0]
    errs = {}
    for k in ("dQt", "ddOt", "alpha", "E"):
        errs[k] = rel_fro(np.stack([to_np(out[k][b, h]) for b, h in qheads]),
                          np.stack([ref_q[k][(b, h)] for b, h in qheads]))
    for k in ("dKt", "dVt"):
        errs[k] = rel_fro(np.stack([to_np(out[k][b, g]) for b, g in kvheads]),
                          np.stack([ref_k[k][(b, g)] for b, g in kvheads]))
    for k in ("L", "D"):
        errs[k] = rel_fro(np.stack([to_np(state[k][b, h]) for b, h in qheads]),
                          np.stack([ref_q[k][(b, h)] for b, h in qheads]))
    if heads is None:
        O = np.stack([np.stack([orc.prep(Q[b, h], K[b, h // G], V[b, h // G], dO[b, h], w.tau,
                                         w.causal)[0] for h in range(w.H)])
                      for b in range(w.B)])
        errs["O"] = rel_fro(to_np(state["O"]), O)
    return errs


def sampled_row_errors(w, x, out, state, n_rows=256, seed=1234, heads=None):
    """Row outputs of ``n_rows`` seeded rows per listed head against
    ``oracle.bob_rows`` (O(N d) per row)."""
    rng = np.random.default_rng(seed)
    B, H, N, d = w.B, w.H, w.N, w.d
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    got = {k: [] for k in ("dQt", "ddOt", "alpha", "E", "L", "D")}
    ref = {k: [] for k in got}
    for b, h in heads:
        rows = np.sort(rng.choice(N, size=min(n_rows, N), replace=False))
        g = h // (w.H // w.kv_heads)  # shared key/value head
        args = [as_float64_numpy(x[k][b, g if k in KV_NAMES else h]) for k in NAMES]
        r = orc.bob_rows(*args, w.tau, rows, causal=w.causal)
        for k in got:
            src = out[k] if k in out else state[k]
            got[k].append(to_np(src[b, h][rows]))
            ref[k].append(r[k])
    return {k: rel_fro(np.concatenate(got[k]), np.concatenate(ref[k])) for k in got}


def sampled_col_errors(w, x, out, kv_heads, n_cols=128, seed=4321):
    """d~K and d~V of ``n_cols`` seeded key columns of each listed key/value
    head (b, g) against the column-form oracle, element by element.  The
    oracle's own row scalars (L, D, alpha, E of every row of every query head
    of the group; plain C, fp64) feed ``oracle.bob_cols_group``: nothing the
    CUDA path computed is used."""
    from oracle import crows
    rng = np.random.default_rng(seed)
    G = w.H // w.kv_heads
    got = {"dKt": [], "dVt": []}
    ref = {"dKt": [], "dVt": []}
    for b, g in kv_heads:
        cols = np.sort(rng.choice(w.kv_len, size=min(n_cols, w.kv_len), replace=False))
        kv = [as_float64_numpy(x[k][b, g]) for k in ("K", "V", "UK", "UV")]
        hs = range(g * G, (g + 1) * G)
        qs = {k: np.stack([as_float64_numpy(x[k][b, h]) for h in hs]) for k in ("Q", "dO", "UQ")}
        scal = [crows.row_scalars(qs["Q"][i], kv[0], kv[1], qs["dO"][i], qs["UQ"][i], kv[2],
                                  kv[3], w.tau, w.causal) for i in range(G)]
        r = orc.bob_cols_group(qs["Q"], kv[0], kv[1], qs["dO"], qs["UQ"], kv[2], kv[3], w.tau,
                               cols, w.causal, scalars=scal)
        for k in got:
            got[k].append(to_np(out[k][b, g][cols]))
            ref[k].append(r[k])
    return {k: rel_fro(np.concatenate(got[k]), np.concatenate(ref[k])) for k in got}


def column_sum_residuals(out):
    """|sum_j d~K_j| and |sum_j d~V_j| relative to the column norms: both sums
    vanish exactly (Phi is invariant under K -> K + 1 c^T, V -> V + 1 c^T)."""
    res = {}
    for k in ("dKt", "dVt"):
        a = out[k].double()
        s = a.sum(dim=2)  # [B, H, d]
        scale = a.pow(2).sum(dim=2).sqrt()
        res[k] = float((s.norm() / scale.norm()).item())
    return res
