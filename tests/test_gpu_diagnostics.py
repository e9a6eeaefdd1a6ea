"""The tensor-core issue-rate diagnostic (flashbob_mma_cycles): it runs,
returns a positive cost for every shape, and the cost grows with N where the
math dominates (N = 256 takes about twice N = 128)."""
import pytest

from exact_second_order_gb300 import flashbob as fb

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("a_in_tmem", [False, True])
def test_mma_cycles_shapes(a_in_tmem):
    c = {n: fb.flashbob_mma_cycles(n, a_in_tmem) for n in (32, 64, 128, 256)}
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    assert all(v > 0 for v in c.values()), c
    assert 1.6 <= c[256] / c[128] <= 2.4, c
    assert c[32] <= c[64] * 1.05 and c[64] <= c[128] * 1.05, c
