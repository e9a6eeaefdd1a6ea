"""The bench's host-side pieces on CPU: the oracle sample behind
`cpu_baseline` and the reference arm, and the workload keys that both arms'
lines carry (so that their configs compare equal)."""
import bench
from exact_second_order_gb300 import inputs as wl


def test_oracle_sample_and_baseline_record():
    w = wl.small_workload(1, 2, 256, 64, "bf16", seed=3)
    x = wl.make_inputs(w)
    smp = bench.oracle_sample(w, x, 0.3)
    assert smp["rows"] > 0 and smp["cols"] > 0 and smp["t_rows"] > 0 and smp["t_cols"] > 0
    base = bench.oracle_baseline(w, smp)
    assert base["kind"] == "oracle" and base["unit"] == bench.UNIT
    assert base["value"] > 0 and base["cores"] >= 1 and base["sample"]
    assert base["seconds_per_row"] > 0 and base["seconds_per_column"] > 0
    # the extrapolation covers every row and every key column of every head
    full = w.B * (w.H * w.N * base["seconds_per_row"] + w.H * w.kv_len * base["seconds_per_column"])
    assert abs(base["extrapolated_full_call_s"] - full) <= 1e-9 * full


def test_both_arms_carry_the_same_workload_keys():
    for w in (wl.LONG_CONTEXT, wl.GQA_N8192, wl.RECT_Q4096_K16384, wl.CAUSAL_N4096):
        c = bench.config_dict(w)
        assert c["workload"] == w.name and c["Hkv"] == w.kv_heads and c["Nk"] == w.kv_len
        assert set(c) == {"workload", "B", "H", "Hkv", "N", "Nk", "d", "causal", "tau",
                          "flop_convention"}
    assert bench.DEFAULT_WORKLOAD == wl.LONG_CONTEXT.name
