"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle.

Small shapes: every output against the full oracle, element by element
(relative Frobenius error).  Full workload sizes: seeded rows of every head
against the per-row oracle (alpha, E, d~Q, d~dO, L, D) and seeded key
columns against the column-form oracle (d~K, d~V, with the oracle's own row
scalars of every row), plus the exact column-sum invariants of d~K and d~V,
NaN-poisoned outputs (every element written) and the memory check.  Long
query streams against a few key blocks run pass 2's full-length loop under
the full oracle.  Every achieved error is recorded (tests/helpers.py).
"""
import os

import numpy as np
import pytest
import torch

from exact_second_order_gb300 import flashbob as fb
from exact_second_order_gb300 import inputs as wl
from tests.helpers import (MAT_KEYS, ROW_KEYS, TOL, column_sum_residuals, full_oracle_errors,
                           record, run_cuda, sampled_col_errors, sampled_row_errors)

pytestmark = pytest.mark.gpu


def _assert_all_written(out):
    for k, t in out.items():
        assert not torch.isnan(t).any().item(), f"{k} has unwritten (NaN) elements"


def _check_full(w, heads=None):
    x, dev, state, out = run_cuda(w)
    _assert_all_written(out)
    errs = record(f"{w.name} full", full_oracle_errors(w, x, state, out, heads=heads))
    tol = TOL[w.dtype]
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{w.name}: {bad} (all: {errs})"
    return errs


def test_tiny_f32_workload_full_oracle():
    errs = _check_full(wl.TINY_F32)
    assert max(errs.values()) < 1e-4


@pytest.mark.parametrize("N", [1, 2, 7, 31, 33, 65, 129, 300])
@pytest.mark.parametrize("d", [64, 128, 5, 100])
def test_f32_ragged_shapes(N, d):
    _check_full(wl.small_workload(1, 2, N, d, "f32", seed=N + d))


def test_f32_batch_heads():
    _check_full(wl.small_workload(2, 3, 97, 64, "f32", seed=3))


@pytest.mark.parametrize("N", [1, 7, 32, 127, 128, 129, 300, 1000])
@pytest.mark.parametrize("d", [64, 128, 96])
def test_bf16_ragged_shapes(N, d):
    _check_full(wl.small_workload(1, 2, N, d, "bf16", seed=N + d))


def test_bf16_peaked_and_stress_small():
    _check_full(wl.small_workload(1, 2, 700, 64, "bf16", seed=9, peaked_k_rows=True))
    _check_full(wl.small_workload(1, 2, 700, 64, "bf16", seed=9, peaked_k_rows=True,
                                  stress=True))


def test_gpt2_layer_workload_full_oracle():
    _check_full(wl.GPT2_LAYER)


@pytest.mark.parametrize("w", [wl.MID_LENGTH, wl.MID_LENGTH_PEAKED, wl.MID_LENGTH_STRESS],
                         ids=lambda w: w.name)
def test_mid_length_workloads(w):
    x, dev, state, out = run_cuda(w)
    _assert_all_written(out)
    errs = record(f"{w.name} rows", sampled_row_errors(w, x, out, state))
    assert max(errs.values()) <= TOL["bf16"], errs
    cols = record(f"{w.name} cols", sampled_col_errors(
        w, x, out, [(0, g) for g in range(w.kv_heads)], n_cols=64))
    assert max(cols.values()) <= TOL["bf16"], cols
    res = column_sum_residuals(out)
    assert max(res.values()) <= TOL["bf16"], res
    # full oracle on one head covers every element of that head
    full = record(f"{w.name} full head", full_oracle_errors(w, x, state, out, heads=[(0, 0)]))
    assert max(full.values()) <= TOL["bf16"], full


def _memory_checked_run(w):
    torch.cuda.synchronize()
    x = wl.make_inputs(w)
    dev = {k: v.cuda() for k, v in x.items()}
    O, L, D = fb.prep(dev["Q"], dev["K"], dev["V"], dev["dO"], w.tau, causal=w.causal)
    out = fb.alloc_bob_outputs(dev["Q"], fill=float("nan"), K=dev["K"])
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    before_alloc = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    fb.bob(dev["Q"], dev["K"], dev["V"], O, dev["dO"], L, D, dev["UQ"], dev["UK"], dev["UV"],
           w.tau, out=out, causal=w.causal)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert torch.cuda.max_memory_allocated() - before_alloc <= 64 << 20
    assert free_before - free_after <= 64 << 20
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    return x, dev, {"O": O, "L": L, "D": D}, out


@pytest.mark.parametrize("w", [wl.LONG_CONTEXT, wl.EXTREME_D64, wl.EXTREME_D128],
                         ids=lambda w: w.name)
def test_long_workloads_sampled_rows_columns_and_memory(w):
    x, dev, state, out = _memory_checked_run(w)
    _assert_all_written(out)
    heads = [(0, h) for h in range(w.H)]
    errs = record(f"{w.name} rows", sampled_row_errors(
        w, x, out, state, n_rows=256 if w.H == 1 else 64, heads=heads))
    assert max(errs.values()) <= TOL["bf16"], errs
    res = record(f"{w.name} column sums", column_sum_residuals(out))
    assert max(res.values()) <= TOL["bf16"], res
    # d~K, d~V element by element on seeded key columns: the oracle needs
    # every row's scalars (O(N^2 d) per head on the host), so the longest
    # sequences take minutes and are opted into with FLASHBOB_FULL_COLUMNS=1.
    if w is wl.LONG_CONTEXT or os.environ.get("FLASHBOB_FULL_COLUMNS") == "1":
        kv = [(0, g) for g in range(w.kv_heads)] if w is not wl.LONG_CONTEXT else [(0, 0), (0, 3)]
        cols = record(f"{w.name} cols", sampled_col_errors(w, x, out, kv, n_cols=128))
        assert max(cols.values()) <= TOL["bf16"], cols


# Pass 2 at its full-size loop length: a query stream as long as the long
# workloads' (1024, 4096 and 4096 tiles per key block) against a few key
# blocks, so that every d~K, d~V column and sampled rows go through the
# oracle in seconds.
@pytest.mark.parametrize("w", [wl.LONGLOOP_D64, wl.LONGLOOP_EXTREME_D64, wl.LONGLOOP_D128],
                         ids=lambda w: w.name)
def test_long_query_streams_every_column(w):
    x, dev, state, out = run_cuda(w)
    _assert_all_written(out)
    cols = record(f"{w.name} all cols", sampled_col_errors(
        w, x, out, [(0, g) for g in range(w.kv_heads)], n_cols=w.kv_len))
    assert max(cols.values()) <= TOL["bf16"], cols
    errs = record(f"{w.name} rows", sampled_row_errors(
        w, x, out, state, n_rows=512, heads=[(0, h) for h in range(w.H)]))
    assert max(errs.values()) <= TOL["bf16"], errs


def test_stream_argument_is_honoured():
    w = wl.small_workload(1, 2, 200, 64, "bf16", seed=5)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        x, dev, state, out = run_cuda(w, stream=s)
    errs = full_oracle_errors(w, x, state, out)
    assert max(errs.values()) <= TOL["bf16"], errs


def test_repeated_calls_are_deterministic():
    w = wl.small_workload(1, 3, 333, 64, "bf16", seed=6)
    _, dev, state, out1 = run_cuda(w)
    out2 = fb.bob(dev["Q"], dev["K"], dev["V"], state["O"], dev["dO"], state["L"], state["D"],
                  dev["UQ"], dev["UK"], dev["UV"], w.tau)
    torch.cuda.synchronize()
    for k in MAT_KEYS + ROW_KEYS:
        assert torch.equal(out1[k], out2[k]), k


def test_bad_arguments_return_codes_and_launch_nothing():
    w = wl.small_workload(1, 1, 64, 64, "bf16")
    x, dev, state, out = run_cuda(w)
    before = {k: v.clone() for k, v in out.items()}
    with pytest.raises(fb.FlashbobError) as e:
        fb.bob(dev["Q"], dev["K"], dev["V"], state["O"], dev["dO"], state["L"], state["D"],
               dev["UQ"], dev["UK"], dev["UV"], float("nan"), out=out)
    assert e.value.status == fb.FLASHBOB_ERR_INVALID_ARG
    torch.cuda.synchronize()
    for k in out:
        assert torch.equal(out[k], before[k]) or torch.isnan(before[k]).all()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    np.testing.assert_equal(fb.flashbob_status_string(0), "FLASHBOB_OK")


def test_binding_checks_every_tensor_before_the_call():
    # Shape, dtype, layout and device of every tensor are checked in the
    # binding (the C ABI sees only pointers and sizes); a rejected call
    # launches nothing.
    w = wl.small_workload(1, 2, 64, 64, "bf16", seed=8)
    x, dev, state, out = run_cuda(w)
    before = {k: v.clone() for k, v in out.items()}
    args = dict(dev, O=state["O"], L=state["L"], D=state["D"])

    def call(**over):
        a = dict(args, **over)
        fb.bob(a["Q"], a["K"], a["V"], a["O"], a["dO"], a["L"], a["D"], a["UQ"], a["UK"],
               a["UV"], w.tau, out=out)

    with pytest.raises(ValueError, match="shape"):
        call(K=dev["K"][..., :32].contiguous())                 # wrong head dim
    with pytest.raises(ValueError, match="shape"):
        call(L=state["L"][:, :1].contiguous())                  # wrong head count
    with pytest.raises(TypeError, match="float32"):
        call(K=dev["K"].float())                                # inputs of mixed dtypes
    with pytest.raises(TypeError, match="float32"):
        call(O=state["O"].bfloat16())                           # row state not fp32
    with pytest.raises(ValueError, match="contiguous"):
        call(V=dev["V"].transpose(2, 3).contiguous().transpose(2, 3))   # column-major V
    with pytest.raises(ValueError, match="CUDA tensor"):
        call(UQ=dev["UQ"].cpu())
    torch.cuda.synchronize()
    for k in out:
        assert torch.equal(out[k], before[k]), k
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK


# --------------------------------------------------------------------------
# Causal mask (the setting of the pages' timing tables)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N", [1, 5, 32, 127, 128, 129, 300, 700])
@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (64, "f32"), (96, "bf16"), (128, "bf16")])
def test_causal_small_shapes(N, d, dtype):
    _check_full(wl.small_workload(1, 2, N, d, dtype, seed=N + d, causal=True))


def test_causal_pages_shape_sampled_rows():
    w = wl.CAUSAL_N4096
    x, dev, state, out = run_cuda(w)
    _assert_all_written(out)
    heads = [(0, 0), (1, 5), (3, 11)]
    errs = record(f"{w.name} rows", sampled_row_errors(w, x, out, state, n_rows=128,
                                                       heads=heads))
    assert max(errs.values()) <= TOL["bf16"], errs
    cols = record(f"{w.name} cols", sampled_col_errors(w, x, out, heads, n_cols=128))
    assert max(cols.values()) <= TOL["bf16"], cols
    res = column_sum_residuals(out)
    assert max(res.values()) <= TOL["bf16"], res
    full = record(f"{w.name} full head", full_oracle_errors(w, x, state, out, heads=[(2, 7)]))
    assert max(full.values()) <= TOL["bf16"], full


# --------------------------------------------------------------------------
# Grouped-query / multi-query attention (shared key/value heads)
# --------------------------------------------------------------------------

# Small grids split each group over a cluster of S CTAs (S = 2, 4, 2, 3, 8
# for these head counts), so these shapes also cover the cluster-wide sum.
@pytest.mark.parametrize("H,Hkv", [(4, 2), (4, 1), (6, 3), (6, 2), (8, 1)])
@pytest.mark.parametrize("N", [1, 65, 300])
@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("f32", 64), ("bf16", 96), ("bf16", 128)])
def test_gqa_small_shapes(H, Hkv, N, dtype, d):
    _check_full(wl.small_workload(2, H, N, d, dtype, seed=N + H, Hkv=Hkv))


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_causal_bf16(causal):
    _check_full(wl.small_workload(1, 4, 333, 64, "bf16", seed=8, Hkv=2, causal=causal))


@pytest.mark.parametrize("w", [wl.GQA_N8192, wl.MQA_N8192], ids=lambda w: w.name)
def test_gqa_workloads_sampled_rows(w):
    x, dev, state, out = run_cuda(w)
    _assert_all_written(out)
    heads = [(0, 0), (0, 5), (0, 11)]
    errs = record(f"{w.name} rows", sampled_row_errors(w, x, out, state, n_rows=128,
                                                       heads=heads))
    assert max(errs.values()) <= TOL["bf16"], errs
    cols = record(f"{w.name} cols", sampled_col_errors(
        w, x, out, [(0, g) for g in range(w.kv_heads)], n_cols=64))
    assert max(cols.values()) <= TOL["bf16"], cols
    res = column_sum_residuals(out)
    assert max(res.values()) <= TOL["bf16"], res
    full = record(f"{w.name} full group", full_oracle_errors(w, x, state, out, heads=[(0, 0)]))
    assert max(full.values()) <= TOL["bf16"], full


# --------------------------------------------------------------------------
# Rectangular attention (N_q query rows, N_k key rows)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,Nk", [(1, 300), (65, 7), (129, 300), (300, 129), (200, 1)])
@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("f32", 64), ("bf16", 96), ("bf16", 128)])
def test_rectangular_small_shapes(N, Nk, dtype, d, causal):
    # causal with Nk >= Nq + 128 leaves whole key blocks that no query sees
    _check_full(wl.small_workload(1, 2, N, d, dtype, seed=N + Nk, Nk=Nk, causal=causal))


@pytest.mark.parametrize("causal", [False, True])
def test_rectangular_gqa_bf16(causal):
    _check_full(wl.small_workload(2, 4, 200, 64, "bf16", seed=12, Hkv=2, Nk=333, causal=causal))


@pytest.mark.parametrize("w", [wl.RECT_Q4096_K16384, wl.RECT_Q16384_K4096], ids=lambda w: w.name)
def test_rectangular_workloads_sampled_rows(w):
    x, dev, state, out = run_cuda(w)
    _assert_all_written(out)
    heads = [(0, 0), (0, 7)]
    errs = record(f"{w.name} rows", sampled_row_errors(w, x, out, state, n_rows=128,
                                                       heads=heads))
    assert max(errs.values()) <= TOL["bf16"], errs
    cols = record(f"{w.name} cols", sampled_col_errors(w, x, out, heads, n_cols=128))
    assert max(cols.values()) <= TOL["bf16"], cols
    res = column_sum_residuals(out)
    assert max(res.values()) <= TOL["bf16"], res
    full = record(f"{w.name} full head", full_oracle_errors(w, x, state, out, heads=[(0, 3)]))
    assert max(full.values()) <= TOL["bf16"], full


# Maximum head counts: B * H = 5 * 65535 query heads, more than four times
# the grid's y extent, so the heads cannot be cut into four head-group slices
# of at most 65535 and the call runs whole on the caller's stream (d = 64,
# and grouped-query d = 128).  Inputs are drawn on the device (the CPU draw
# of 3e8 values takes minutes); key/value groups sampled across the whole
# range of heads go through the full oracle.
MAX_HEADS = [wl.small_workload(5, 65535, 3, 64, "bf16", seed=31),
             wl.small_workload(5, 65535, 3, 128, "bf16", seed=32, Hkv=13107)]


def _group_subproblem(w, x, state, out, groups):
    """Key/value groups (b, g) of a large call as a workload of their own:
    batch i = group i, with its H / Hkv query heads and one key/value head."""
    G = w.H // w.kv_heads
    sub = wl.small_workload(len(groups), G, w.N, w.d, w.dtype, seed=w.seed, Hkv=1,
                            causal=w.causal)

    def q(t):
        return torch.stack([t[b, g * G:(g + 1) * G] for b, g in groups])

    def kv(t):
        return torch.stack([t[b, g:g + 1] for b, g in groups])

    xs = {k: (kv(v) if k in wl.KV_NAMES else q(v)) for k, v in x.items()}
    st = {k: q(v) for k, v in state.items()}
    os_ = {k: (kv(v) if k in ("dKt", "dVt") else q(v)) for k, v in out.items()}
    return sub, xs, st, os_


@pytest.mark.parametrize("w", MAX_HEADS, ids=lambda w: w.name)
def test_maximum_head_counts(w):
    assert fb.flashbob_bob_launches(w.B, w.H, w.kv_heads, w.N, w.kv_len, w.d,
                                    fb.FLASHBOB_BF16) == (3 if w.d == 128 else 2)
    x = wl.make_inputs(w, device="cuda")
    O, L, D = fb.prep(x["Q"], x["K"], x["V"], x["dO"], w.tau, causal=w.causal)
    out = fb.alloc_bob_outputs(x["Q"], fill=float("nan"), K=x["K"])
    fb.bob(x["Q"], x["K"], x["V"], O, x["dO"], L, D, x["UQ"], x["UK"], x["UV"], w.tau,
           out=out, causal=w.causal)
    torch.cuda.synchronize()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    _assert_all_written(out)
    n = w.kv_heads
    groups = [(0, 0), (0, n - 1), (1, n // 3), (2, n // 2), (3, 2 * n // 3), (4, n - 2),
              (4, n - 1)]
    sub, xs, st, os_ = _group_subproblem(w, x, {"O": O, "L": L, "D": D}, out, groups)
    errs = record(f"{w.name} sampled groups", full_oracle_errors(sub, xs, st, os_))
    assert max(errs.values()) <= TOL["bf16"], errs
    del x, O, L, D, out
    torch.cuda.empty_cache()


# --------------------------------------------------------------------------
# Head dim 128 on the tensor cores
# --------------------------------------------------------------------------

def test_d128_runs_the_tensor_core_tiles():
    t = fb.flashbob_bob_tile_sizes(128, fb.FLASHBOB_BF16)
    assert (t["Br1"], t["Bc1"], t["Br2"], t["Bc2"]) == (128, 32, 32, 128)


@pytest.mark.parametrize("w", [wl.small_workload(1, 2, 700, 128, "bf16", seed=21,
                                                 peaked_k_rows=True, stress=True),
                               wl.small_workload(2, 6, 1000, 128, "bf16", seed=22, Hkv=2,
                                                 causal=True),
                               wl.small_workload(1, 3, 777, 128, "bf16", seed=23, Nk=1300)],
                         ids=lambda w: w.name)
def test_d128_stress_gqa_causal_rectangular(w):
    _check_full(w)


def test_d128_mid_length_sampled_rows():
    w = wl.Workload("mid_B1_H4_N8192_d128", 1, 4, 8192, 128, "bf16", causal=True)
    x, dev, state, out = run_cuda(w)
    _assert_all_written(out)
    errs = record(f"{w.name} rows", sampled_row_errors(w, x, out, state, n_rows=128,
                                                       heads=[(0, 0), (0, 3)]))
    assert max(errs.values()) <= TOL["bf16"], errs
    cols = record(f"{w.name} cols", sampled_col_errors(w, x, out, [(0, 0), (0, 3)], n_cols=128))
    assert max(cols.values()) <= TOL["bf16"], cols
    res = column_sum_residuals(out)
    assert max(res.values()) <= TOL["bf16"], res
    full = record(f"{w.name} full head", full_oracle_errors(w, x, state, out, heads=[(0, 1)]))
    assert max(full.values()) <= TOL["bf16"], full


# --------------------------------------------------------------------------
# Failure detection: a bounded wait that runs out is reported, not hung
# --------------------------------------------------------------------------

def test_bounded_wait_gives_up_and_reports_timeout():
    import time
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    t0 = time.perf_counter()
    fb.flashbob_check_wait_timeout()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_ERR_TIMEOUT  # synchronises
    assert time.perf_counter() - t0 >= 1.5  # the 2 s limit, not an early exit
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK  # the report clears the word
    # the context is still usable
    _check_full(wl.small_workload(1, 2, 150, 64, "bf16", seed=31))


# --------------------------------------------------------------------------
# Prep: the running row maximum is raised mid-sequence
# --------------------------------------------------------------------------

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_prep_when_later_keys_dominate(d, causal):
    """Keys past position 640 are scaled up ×3 (scores of variance ~9 against
    ~0.01 before), so most rows' softmax maximum jumps by far more than
    2^8 after the first tiles and prep must rescale its running sums and
    accumulators; O, L, D, and the BoB built on them, against the oracle."""
    from exact_second_order_gb300.inputs import NAMES, as_float64_numpy
    w = wl.small_workload(1, 2, 1500, d, "bf16", seed=40 + d, dist="unit", causal=causal)
    x = wl.make_inputs(w)
    scale = torch.full((w.N, 1), 0.1)
    scale[640:] = 3.0
    x["K"] = (x["K"].float() * scale).to(torch.bfloat16)
    dev = {k: v.cuda() for k, v in x.items()}
    O, L, D = fb.prep(dev["Q"], dev["K"], dev["V"], dev["dO"], w.tau, causal=causal)
    out = fb.bob(dev["Q"], dev["K"], dev["V"], O, dev["dO"], L, D, dev["UQ"], dev["UK"],
                 dev["UV"], w.tau, causal=causal)
    torch.cuda.synchronize()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    from tests.helpers import rel_fro, to_np
    from oracle import bob as orc
    errs = {}
    for h in range(w.H):
        a = [as_float64_numpy(x[k][0, h]) for k in NAMES]
        o, l, dd = orc.prep(*a[:4], w.tau, causal)
        r = orc.bob(*a, w.tau, causal)
        for k, got, ref in (("O", O, o), ("L", L, l), ("D", D, dd)):
            errs[f"{k}{h}"] = rel_fro(to_np(got[0, h]), ref)
        for k in ("dQt", "dKt", "dVt", "ddOt", "alpha", "E"):
            errs[f"{k}{h}"] = rel_fro(to_np(out[k][0, h]), r[k])
    record(f"prep rescale d{d} causal={causal}", errs)
    assert max(errs.values()) <= TOL["bf16"], errs
