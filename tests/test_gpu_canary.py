"""Out-of-bounds write checks: every output the C ABI writes sits at the front
of a larger device buffer whose tail holds a sentinel; after the call the
tails must be intact (nothing written past an output) and the fronts fully
written (NaN-poisoned before the call)."""
import math

import pytest
import torch

from exact_second_order_gb300 import flashbob as fb
from exact_second_order_gb300 import inputs as wl

pytestmark = pytest.mark.gpu

SENTINEL = 12345.678
PAD = 4099  # floats past the end of each output (not a multiple of any tile)


class Canaried:
    """fp32 views at the front of sentinel-padded buffers."""

    def __init__(self):
        self.bufs = []

    def __call__(self, *shape):
        n = math.prod(shape)
        buf = torch.full((n + PAD,), SENTINEL, dtype=torch.float32, device="cuda")
        buf[:n] = float("nan")
        self.bufs.append((buf, n))
        return buf[:n].view(*shape)

    def check(self):
        torch.cuda.synchronize()
        for buf, n in self.bufs:
            assert torch.all(buf[n:] == SENTINEL).item(), "write past the end of an output"
            assert not torch.isnan(buf[:n]).any().item(), "an output element was not written"


@pytest.mark.parametrize("w", [
    wl.small_workload(1, 2, 129, 64, "bf16", seed=1),
    wl.small_workload(2, 4, 300, 64, "bf16", seed=2, Hkv=2, Nk=77, causal=True),
    wl.small_workload(1, 6, 333, 64, "bf16", seed=3, Hkv=2),
    wl.small_workload(1, 2, 200, 128, "bf16", seed=4, causal=True),
    wl.small_workload(2, 4, 150, 128, "bf16", seed=5, Hkv=1, Nk=400),
    wl.small_workload(1, 2, 65, 100, "f32", seed=6, causal=True),
], ids=lambda w: w.name + ("_causal" if w.causal else ""))
def test_prep_bob_and_jvp_write_nothing_past_their_outputs(w):
    x = wl.make_inputs(w)
    dev = {k: v.cuda() for k, v in x.items()}
    B, H, Nq, d = dev["Q"].shape
    Hkv, Nk = dev["K"].shape[1], dev["K"].shape[2]
    c = Canaried()
    O, L, D = c(B, H, Nq, d), c(B, H, Nq), c(B, H, Nq)
    fb.flashbob_prep(dev["Q"], dev["K"], dev["V"], dev["dO"], O, L, D, w.tau, causal=w.causal)
    out = {"dQt": c(B, H, Nq, d), "ddOt": c(B, H, Nq, d), "dKt": c(B, Hkv, Nk, d),
           "dVt": c(B, Hkv, Nk, d), "alpha": c(B, H, Nq), "E": c(B, H, Nq)}
    fb.flashbob_bob(dev["Q"], dev["K"], dev["V"], O, dev["dO"], L, D, dev["UQ"], dev["UK"],
                    dev["UV"], w.tau, out["dQt"], out["dKt"], out["dVt"], out["ddOt"],
                    out["alpha"], out["E"], causal=w.causal)
    Od, Ld = c(B, H, Nq, d), c(B, H, Nq)
    fb.flashbob_attention_jvp(dev["Q"], dev["K"], dev["V"], O, L, dev["UQ"], dev["UK"],
                              dev["UV"], w.tau, Od, Ld, causal=w.causal)
    c.check()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
