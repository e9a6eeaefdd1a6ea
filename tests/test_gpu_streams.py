"""The head-group streams of flashbob_bob (a call with several key/value
heads and more than two waves of pass-1 CTAs runs each group's pass 1 ->
pass 2 chain on an internal stream): the results equal those of the two
passes called one after the other on one stream, bit for bit, and the call
stays ordered within the caller's stream (a later kernel on that stream sees
every output)."""
import pytest
import torch

from exact_second_order_gb300 import flashbob as fb
from exact_second_order_gb300 import inputs as wl

pytestmark = pytest.mark.gpu

CASES = [
    wl.small_workload(1, 4, 16384, 64, "bf16", seed=11),                 # 4 groups, 512 CTAs
    wl.small_workload(2, 3, 8192, 64, "bf16", seed=12, causal=True),     # 6 groups, causal
    wl.small_workload(1, 8, 16384, 64, "bf16", seed=13, Hkv=2),          # GQA: 2 groups of 4
    wl.small_workload(1, 4, 16384, 128, "bf16", seed=14, Nk=12288),      # d = 128, rectangular
    wl.small_workload(1, 6, 16384, 128, "bf16", seed=15, causal=True),   # d = 128, 6 groups
]


def _run(w, split):
    x = wl.make_inputs(w)
    d = {k: v.cuda() for k, v in x.items()}
    O, L, D = fb.prep(d["Q"], d["K"], d["V"], d["dO"], w.tau, causal=w.causal)
    out = fb.alloc_bob_outputs(d["Q"], fill=float("nan"), K=d["K"])
    st = torch.cuda.current_stream()
    if split:
        fb.flashbob_bob(d["Q"], d["K"], d["V"], O, d["dO"], L, D, d["UQ"], d["UK"], d["UV"],
                        w.tau, out["dQt"], out["dKt"], out["dVt"], out["ddOt"], out["alpha"],
                        out["E"], causal=w.causal, stream=st)
    else:
        fb.flashbob_bob_pass1(d["Q"], d["K"], d["V"], O, d["dO"], L, D, d["UQ"], d["UK"],
                              d["UV"], w.tau, out["dQt"], out["ddOt"], out["alpha"], out["E"],
                              causal=w.causal, stream=st)
        fb.flashbob_bob_pass2(d["Q"], d["K"], d["V"], d["dO"], L, D, out["alpha"], out["E"],
                              d["UQ"], d["UK"], d["UV"], w.tau, out["dKt"], out["dVt"],
                              causal=w.causal, stream=st)
    # Read on the caller's stream right behind the call, before any device
    # synchronisation: a kernel queued there must see every output.
    sums = {k: torch.nan_to_num(v, nan=1e30).double().sum() for k, v in out.items()}
    torch.cuda.synchronize()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    return out, {k: v.item() for k, v in sums.items()}


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_head_group_streams_match_one_stream_bit_for_bit(w):
    launches = fb.flashbob_bob_launches(w.B, w.H, w.kv_heads, w.N, w.kv_len, w.d,
                                        fb.FLASHBOB_BF16)
    groups = w.B * w.kv_heads
    assert launches == (3 if w.d == 128 else 2) * min(4, groups), launches
    split, split_sums = _run(w, True)
    ref, _ = _run(w, False)
    for k in ref:
        assert not torch.isnan(split[k]).any().item(), f"{k}: unwritten elements"
        assert torch.equal(split[k], ref[k]), f"{k} differs from the one-stream passes"
        # the stream-ordered reduction saw the finished outputs
        assert split_sums[k] == pytest.approx(ref[k].double().sum().item(), rel=0, abs=0)


def test_small_calls_stay_on_the_callers_stream():
    # one wave of pass-1 CTAs, or one head group: no internal streams
    assert fb.flashbob_bob_launches(1, 4, 4, 1024, 1024, 64, fb.FLASHBOB_BF16) == 2
    assert fb.flashbob_bob_launches(1, 12, 1, 65536, 65536, 64, fb.FLASHBOB_BF16) == 2
    assert fb.flashbob_bob_launches(1, 4, 4, 65536, 65536, 64, fb.FLASHBOB_F32) == 2


@pytest.mark.parametrize("w", [CASES[0], CASES[3]], ids=[CASES[0].name, CASES[3].name])
def test_head_group_streams_under_cuda_graph_capture(w):
    # A captured flashbob_bob stays on the capturing stream (the shared
    # internal streams are never drawn into a capture): the replay's outputs
    # equal a direct call's (which runs the head groups on the internal
    # streams) bit for bit, and a replay with changed inputs (same buffers)
    # tracks them.
    x = wl.make_inputs(w)
    d = {k: v.cuda() for k, v in x.items()}
    O, L, D = fb.prep(d["Q"], d["K"], d["V"], d["dO"], w.tau, causal=w.causal)
    ref = fb.bob(d["Q"], d["K"], d["V"], O, d["dO"], L, D, d["UQ"], d["UK"], d["UV"], w.tau,
                 causal=w.causal)
    out = fb.alloc_bob_outputs(d["Q"], fill=float("nan"), K=d["K"])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm the library's caches outside the capture
        fb.bob(d["Q"], d["K"], d["V"], O, d["dO"], L, D, d["UQ"], d["UK"], d["UV"], w.tau,
               out=out, causal=w.causal, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for t in out.values():
        t.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fb.bob(d["Q"], d["K"], d["V"], O, d["dO"], L, D, d["UQ"], d["UK"], d["UV"], w.tau,
               out=out, causal=w.causal, stream=torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    for k in ref:
        assert torch.equal(out[k], ref[k]), f"{k}: graph replay differs from the direct call"
    # new tangents in the same buffers: the replay follows them
    d["UV"].mul_(2)
    ref2 = fb.bob(d["Q"], d["K"], d["V"], O, d["dO"], L, D, d["UQ"], d["UK"], d["UV"], w.tau,
                  causal=w.causal)
    g.replay()
    torch.cuda.synchronize()
    for k in ref2:
        assert torch.equal(out[k], ref2[k]), f"{k}: replay after an input change differs"


def test_direct_call_while_another_thread_captures():
    # One thread opens a capture (thread-local mode) and records a call; before
    # it closes the capture, the main thread makes a direct call of a size that
    # runs head groups on the internal streams.  The direct call runs and is
    # exact (no capture holds the internal streams), and the graph recorded
    # meanwhile replays exactly.
    import threading
    w = CASES[0]
    x = wl.make_inputs(w)
    d = {k: v.cuda() for k, v in x.items()}
    O, L, D = fb.prep(d["Q"], d["K"], d["V"], d["dO"], w.tau, causal=w.causal)
    ref = fb.bob(d["Q"], d["K"], d["V"], O, d["dO"], L, D, d["UQ"], d["UK"], d["UV"], w.tau,
                 causal=w.causal)
    out_g = fb.alloc_bob_outputs(d["Q"], fill=float("nan"), K=d["K"])
    out_d = fb.alloc_bob_outputs(d["Q"], fill=float("nan"), K=d["K"])
    s_main = torch.cuda.Stream()
    torch.cuda.synchronize()
    recorded, direct_done = threading.Event(), threading.Event()
    errors = []
    g = torch.cuda.CUDAGraph()

    def capturer():
        try:
            torch.cuda.set_device(0)
            cap = torch.cuda.Stream()
            with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
                fb.bob(d["Q"], d["K"], d["V"], O, d["dO"], L, D, d["UQ"], d["UK"], d["UV"],
                       w.tau, out=out_g, causal=w.causal, stream=cap)
                recorded.set()
                if not direct_done.wait(timeout=120):
                    raise TimeoutError("the direct call did not finish")
        except Exception as e:  # reported below, on the main thread
            errors.append(e)
        finally:
            recorded.set()

    t = threading.Thread(target=capturer)
    t.start()
    assert recorded.wait(timeout=120)
    try:
        if not errors:
            fb.bob(d["Q"], d["K"], d["V"], O, d["dO"], L, D, d["UQ"], d["UK"], d["UV"], w.tau,
                   out=out_d, causal=w.causal, stream=s_main)
            s_main.synchronize()
    finally:
        direct_done.set()
        t.join(timeout=120)
    assert not t.is_alive()
    assert not errors, errors
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    for k in ref:
        assert torch.equal(out_d[k], ref[k]), f"{k}: the direct call differs"
    g.replay()
    torch.cuda.synchronize()
    for k in ref:
        assert torch.equal(out_g[k], ref[k]), f"{k}: the replay differs"


def test_concurrent_calls_from_two_host_threads():
    # ctypes releases the interpreter lock, so two host threads enqueue
    # flashbob_bob calls at once, each on its own stream; the library
    # serialises the use of its internal streams and events, and every result
    # equals the one-thread result bit for bit.
    import threading
    w = CASES[0]
    x = wl.make_inputs(w)
    d = {k: v.cuda() for k, v in x.items()}
    O, L, D = fb.prep(d["Q"], d["K"], d["V"], d["dO"], w.tau, causal=w.causal)
    ref = fb.bob(d["Q"], d["K"], d["V"], O, d["dO"], L, D, d["UQ"], d["UK"], d["UV"], w.tau,
                 causal=w.causal)
    torch.cuda.synchronize()
    outs = [[fb.alloc_bob_outputs(d["Q"], fill=float("nan"), K=d["K"]) for _ in range(3)]
            for _ in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    errors = []

    def worker(i):
        try:
            torch.cuda.set_device(0)
            for out in outs[i]:
                fb.bob(d["Q"], d["K"], d["V"], O, d["dO"], L, D, d["UQ"], d["UK"], d["UV"],
                       w.tau, out=out, causal=w.causal, stream=streams[i])
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    for per_thread in outs:
        for out in per_thread:
            for k in ref:
                assert torch.equal(out[k], ref[k]), k
