"""GPU parity of flashbob_attention_jvp (through the C ABI) against the fp64
oracle's attention_jvp: O' and L' along the tangents (U_Q, U_K, U_V)."""
import numpy as np
import pytest
import torch

from exact_second_order_gb300 import flashbob as fb
from exact_second_order_gb300 import inputs as wl
from exact_second_order_gb300.inputs import KV_NAMES, NAMES, as_float64_numpy
from oracle import bob as orc
from tests.helpers import TOL, rel_fro, to_np

pytestmark = pytest.mark.gpu


def _run_jvp(w):
    x = wl.make_inputs(w)
    dev = {k: v.cuda() for k, v in x.items()}
    O, L, D = fb.prep(dev["Q"], dev["K"], dev["V"], None, w.tau, causal=w.causal)
    assert D is None
    Od = torch.full_like(O, float("nan"))
    Ld = torch.full_like(L, float("nan"))
    fb.flashbob_attention_jvp(dev["Q"], dev["K"], dev["V"], O, L, dev["UQ"], dev["UK"],
                              dev["UV"], w.tau, Od, Ld, causal=w.causal)
    torch.cuda.synchronize()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    assert not torch.isnan(Od).any().item() and not torch.isnan(Ld).any().item()
    return x, dev, O, L, Od, Ld


def _full_errors(w, x, O, L, Od, Ld):
    arr = {k: as_float64_numpy(x[k]) for k in NAMES}
    G = w.H // w.kv_heads
    ref = {"O": [], "L": [], "Od": [], "Ld": []}
    for b in range(w.B):
        for h in range(w.H):
            g = h // G
            r = orc.attention_jvp(arr["Q"][b, h], arr["K"][b, g], arr["V"][b, g],
                                  arr["UQ"][b, h], arr["UK"][b, g], arr["UV"][b, g], w.tau,
                                  w.causal)
            for k, v in zip(("O", "L", "Od", "Ld"), r):
                ref[k].append(v)
    got = {"O": to_np(O), "L": to_np(L), "Od": to_np(Od), "Ld": to_np(Ld)}
    return {k: rel_fro(got[k].reshape(len(ref[k]), -1),
                       np.stack(ref[k]).reshape(len(ref[k]), -1)) for k in ref}


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,Nk,H,Hkv", [(1, 1, 2, 2), (129, 129, 2, 2), (300, 77, 4, 2),
                                        (65, 300, 3, 1), (1000, 1000, 1, 1),
                                        # one whole 64-key tile; seven whole tiles, so
                                        # every ring of the key stream wraps
                                        (64, 64, 2, 2), (200, 448, 2, 1)])
@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("f32", 64), ("bf16", 96), ("bf16", 128)])
def test_jvp_small_shapes_full_oracle(N, Nk, H, Hkv, dtype, d, causal):
    w = wl.small_workload(1, H, N, d, dtype, seed=N + Nk + H, Hkv=Hkv, Nk=Nk, causal=causal)
    x, dev, O, L, Od, Ld = _run_jvp(w)
    errs = _full_errors(w, x, O, L, Od, Ld)
    tol = TOL[dtype]
    assert max(errs.values()) <= tol, errs


def test_forward_only_prep_matches_full_prep():
    w = wl.small_workload(2, 3, 333, 64, "bf16", seed=4, causal=True)
    x = wl.make_inputs(w)
    dev = {k: v.cuda() for k, v in x.items()}
    O1, L1, _ = fb.prep(dev["Q"], dev["K"], dev["V"], dev["dO"], w.tau, causal=True)
    O2, L2, D2 = fb.prep(dev["Q"], dev["K"], dev["V"], None, w.tau, causal=True)
    torch.cuda.synchronize()
    assert D2 is None
    assert torch.equal(O1, O2) and torch.equal(L1, L2)


@pytest.mark.parametrize("w", [wl.MID_LENGTH, wl.GQA_N8192, wl.RECT_Q4096_K16384,
                               wl.Workload("jvp_B1_H4_N8192_d128", 1, 4, 8192, 128, "bf16",
                                           causal=True)],
                         ids=lambda w: w.name)
def test_jvp_workloads_sampled_rows(w):
    """Rows of O' and L' against the row form of the oracle (its alpha and
    d~dO, which equal L' and O' for any dO)."""
    x, dev, O, L, Od, Ld = _run_jvp(w)
    rng = np.random.default_rng(99)
    G = w.H // w.kv_heads
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for h in (0, w.H - 1):
        rows = np.sort(rng.choice(w.N, size=64, replace=False))
        args = [as_float64_numpy(x[k][0, h // G if k in KV_NAMES else h]) for k in NAMES]
        r = orc.bob_rows(*args, w.tau, rows, causal=w.causal)
        got_o.append(to_np(Od[0, h][rows]))
        got_l.append(to_np(Ld[0, h][rows]))
        ref_o.append(r["ddOt"])
        ref_l.append(r["alpha"])
    assert rel_fro(np.concatenate(got_o), np.concatenate(ref_o)) <= TOL["bf16"]
    assert rel_fro(np.concatenate(got_l), np.concatenate(ref_l)) <= TOL["bf16"]
