"""C-ABI checks that need no GPU: the library loads, exports every entry
point the header declares, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

from exact_second_order_gb300 import flashbob as fb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def lib():
    if not os.path.exists(fb.LIB_PATH):
        from exact_second_order_gb300.build import build
        build()
    return fb.load_library()


def declared_entry_points():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(flashbob_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for n in ("flashbob_prep", "flashbob_bob", "flashbob_bob_pass1", "flashbob_bob_pass2",
              "flashbob_bob_tile_sizes",
              "flashbob_last_device_error", "flashbob_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_entry_points():
        assert hasattr(lib, name), name
        assert name in fb._SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    assert fb.flashbob_status_string(0) == "FLASHBOB_OK"
    assert fb.flashbob_status_string(5) == "FLASHBOB_ERR_TIMEOUT"
    assert fb.flashbob_status_string(99) == "FLASHBOB_UNKNOWN_STATUS"


def test_tile_sizes(lib):
    t = fb.flashbob_bob_tile_sizes(64, fb.FLASHBOB_F32)
    assert t["Br1"] > 0 and t["Bc2"] > 0 and t["smem_bytes_pass1"] > 0
    t = fb.flashbob_bob_tile_sizes(64, fb.FLASHBOB_BF16)
    assert t["smem_bytes_pass1"] <= 232448 and t["smem_bytes_pass2"] <= 232448
    t = fb.flashbob_bob_tile_sizes(128, fb.FLASHBOB_BF16)
    assert t["smem_bytes_pass1"] <= 232448
    for bad in (0, -1, 129):
        assert lib.flashbob_bob_tile_sizes(bad, 0, None, None, None, None, None, None) == \
            fb.FLASHBOB_ERR_UNSUPPORTED
    assert lib.flashbob_bob_tile_sizes(64, 7, None, None, None, None, None, None) == \
        fb.FLASHBOB_ERR_INVALID_ARG


def _bob_raw(lib, ptrs, tau=0.125, B=1, H=1, N=8, d=64, dtype=0, causal=0, Hkv=None, Nk=None):
    Hkv = H if Hkv is None else Hkv
    Nk = N if Nk is None else Nk
    return lib.flashbob_bob(*ptrs[:10], tau, *ptrs[10:], B, H, Hkv, N, Nk, d, causal, dtype,
                            None)


def _fake_ptrs(n=16, stride=1 << 20, base=1 << 32):
    # distinct, 16-byte aligned, non-overlapping addresses; never dereferenced
    return [base + i * stride for i in range(n)]


def test_bob_rejects_bad_arguments_on_the_host(lib):
    ok = _fake_ptrs()
    E = fb
    # null pointer
    for i in range(16):
        p = list(ok)
        p[i] = None
        assert _bob_raw(lib, p) == E.FLASHBOB_ERR_INVALID_ARG
    # sizes and tau
    for kw in ({"B": 0}, {"H": -1}, {"N": 0}, {"Nk": 0}, {"Nk": -3}, {"d": 0}, {"tau": 0.0},
               {"tau": -1.0},
               {"tau": float("nan")}, {"tau": float("inf")}, {"dtype": 3}, {"causal": 2},
               {"causal": -1}, {"Hkv": 0}, {"H": 4, "Hkv": 3}, {"H": 2, "Hkv": 4}):
        assert _bob_raw(lib, ok, **kw) == E.FLASHBOB_ERR_INVALID_ARG, kw
    assert _bob_raw(lib, ok, d=129) == E.FLASHBOB_ERR_UNSUPPORTED
    assert _bob_raw(lib, ok, H=70000) == E.FLASHBOB_ERR_UNSUPPORTED
    # B * H must fit the kernels' 32-bit (batch, head) index
    assert _bob_raw(lib, ok, B=32769, H=65535) == E.FLASHBOB_ERR_UNSUPPORTED
    # misaligned pointer
    for i in range(16):
        p = list(ok)
        p[i] += 8
        assert _bob_raw(lib, p) == E.FLASHBOB_ERR_MISALIGNED
    # an output overlapping an input, and two overlapping outputs
    p = list(ok)
    p[10] = p[0] + 16
    assert _bob_raw(lib, p) == E.FLASHBOB_ERR_INVALID_ARG
    p = list(ok)
    p[11] = p[10]
    assert _bob_raw(lib, p) == E.FLASHBOB_ERR_INVALID_ARG


def test_bob_sizes_key_side_buffers_by_nk_and_hkv(lib):
    """The overlap check sizes K, V, U_K, U_V, d~K, d~V with Hkv heads of Nk
    rows and the query-side buffers with H heads of Nq rows."""
    ok = _fake_ptrs()
    # d~K starts 2 KiB into K: inside K's 4 KiB at Nk = 16 (fp32, d = 64),
    # outside it if K were sized with Nq = 1 rows.
    p = list(ok)
    p[11] = p[1] + 2048
    assert _bob_raw(lib, p, N=1, Nk=16) == fb.FLASHBOB_ERR_INVALID_ARG
    # d~Q starts 2 KiB into Q: inside Q's 4 KiB at Nq = 16.
    p = list(ok)
    p[10] = p[0] + 2048
    assert _bob_raw(lib, p, N=16, Nk=1) == fb.FLASHBOB_ERR_INVALID_ARG


def test_prep_rejects_bad_arguments_on_the_host(lib):
    ok = _fake_ptrs(7)

    def call(p=ok, B=1, H=1, N=8, d=64, tau=0.125, dtype=0, causal=0, Hkv=None, Nk=None):
        Hkv = H if Hkv is None else Hkv
        Nk = N if Nk is None else Nk
        return lib.flashbob_prep(*p, B, H, Hkv, N, Nk, d, tau, causal, dtype, None)
    for i in range(7):
        p = list(ok)
        p[i] = None
        assert call(p) == fb.FLASHBOB_ERR_INVALID_ARG
        p = list(ok)
        p[i] += 4
        assert call(p) == fb.FLASHBOB_ERR_MISALIGNED
    assert call(N=0) == fb.FLASHBOB_ERR_INVALID_ARG
    assert call(Nk=0) == fb.FLASHBOB_ERR_INVALID_ARG
    assert call(tau=float("nan")) == fb.FLASHBOB_ERR_INVALID_ARG
    assert call(d=200) == fb.FLASHBOB_ERR_UNSUPPORTED
    assert call(B=32769, H=65535) == fb.FLASHBOB_ERR_UNSUPPORTED
    assert call(causal=3) == fb.FLASHBOB_ERR_INVALID_ARG
    assert call(H=6, Hkv=4) == fb.FLASHBOB_ERR_INVALID_ARG
    p = list(ok)
    p[4] = p[3]
    assert call(p) == fb.FLASHBOB_ERR_INVALID_ARG


def test_binding_fails_loudly_without_the_library(tmp_path):
    saved = fb._lib
    fb._lib = None
    try:
        with pytest.raises(ImportError):
            fb.load_library(str(tmp_path / "missing.so"))
    finally:
        fb._lib = saved


def test_binding_rejects_host_tensors_and_bad_ranks():
    # The C ABI takes device pointers only; the binding refuses host tensors
    # (and tensors that are not [B, heads, rows, d]) before any call.
    import torch
    x = {k: torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16) for k in
         ("Q", "K", "V", "dO", "UQ", "UK", "UV")}
    O = torch.zeros(1, 2, 8, 64)
    L = torch.zeros(1, 2, 8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fb.flashbob_prep(x["Q"], x["K"], x["V"], x["dO"], O, L, L.clone(), 0.125)
    out = {k: torch.zeros(1, 2, 8, 64) for k in ("dQt", "dKt", "dVt", "ddOt")}
    with pytest.raises(ValueError, match="CUDA tensor"):
        fb.flashbob_bob(x["Q"], x["K"], x["V"], O, x["dO"], L, L, x["UQ"], x["UK"], x["UV"],
                        0.125, out["dQt"], out["dKt"], out["dVt"], out["ddOt"], L, L)
    with pytest.raises(ValueError, match="4-d"):
        fb.flashbob_attention_jvp(x["Q"][0], x["K"], x["V"], O, L, x["UQ"], x["UK"], x["UV"],
                                  0.125, O, L)


def test_pass_entry_points_reject_bad_arguments_on_the_host(lib):
    ok = _fake_ptrs()
    sizes = (1, 1, 1, 8, 8, 64, 0, 0, None)  # B, H, Hkv, Nq, Nk, d, causal, dtype, stream
    p1 = ok[:15]
    bad = list(p1)
    bad[3] = None  # O
    assert lib.flashbob_bob_pass1(*bad[:10], 0.125, *bad[10:14], *sizes) == \
        fb.FLASHBOB_ERR_INVALID_ARG
    bad = list(p1)
    bad[10] = bad[4]  # d~Q over dO
    assert lib.flashbob_bob_pass1(*bad[:10], 0.125, *bad[10:14], *sizes) == \
        fb.FLASHBOB_ERR_INVALID_ARG
    p2 = ok[:13]
    bad = list(p2)
    bad[6] = None  # alpha
    assert lib.flashbob_bob_pass2(*bad[:11], 0.125, *bad[11:13], *sizes) == \
        fb.FLASHBOB_ERR_INVALID_ARG
    bad = list(p2)
    bad[11] = bad[6]  # d~K over alpha
    assert lib.flashbob_bob_pass2(*bad[:11], 0.125, *bad[11:13], *sizes) == \
        fb.FLASHBOB_ERR_INVALID_ARG
    bad = list(p2)
    bad[12] += 4
    assert lib.flashbob_bob_pass2(*bad[:11], 0.125, *bad[11:13], *sizes) == \
        fb.FLASHBOB_ERR_MISALIGNED


def test_jvp_and_forward_only_prep_reject_bad_arguments_on_the_host(lib):
    ok = _fake_ptrs(10)
    sizes = (1, 2, 1, 8, 8, 64, 0, 0, None)  # B, H, Hkv, Nq, Nk, d, causal, dtype, stream

    def jvp(p, tau=0.125, sz=sizes):
        return lib.flashbob_attention_jvp(*p[:8], tau, *p[8:], *sz)
    for i in range(10):
        p = list(ok)
        p[i] = None
        assert jvp(p) == fb.FLASHBOB_ERR_INVALID_ARG
        p = list(ok)
        p[i] += 8
        assert jvp(p) == fb.FLASHBOB_ERR_MISALIGNED
    assert jvp(ok, tau=float("nan")) == fb.FLASHBOB_ERR_INVALID_ARG
    assert jvp(ok, sz=(1, 3, 2, 8, 8, 64, 0, 0, None)) == fb.FLASHBOB_ERR_INVALID_ARG
    assert jvp(ok, sz=(1, 2, 1, 8, 0, 64, 0, 0, None)) == fb.FLASHBOB_ERR_INVALID_ARG
    assert jvp(ok, sz=(1, 2, 1, 8, 8, 64, 2, 0, None)) == fb.FLASHBOB_ERR_INVALID_ARG
    p = list(ok)
    p[8] = p[3] + 16  # O' over O
    assert jvp(p) == fb.FLASHBOB_ERR_INVALID_ARG
    p = list(ok)
    p[9] = p[8]  # L' over O'
    assert jvp(p) == fb.FLASHBOB_ERR_INVALID_ARG
    # prep: dO and D are both given or both null
    q = _fake_ptrs(7)
    for i in (3, 6):
        p = list(q)
        p[i] = None
        assert lib.flashbob_prep(*p, 1, 1, 1, 8, 8, 64, 0.125, 0, 0, None) == \
            fb.FLASHBOB_ERR_INVALID_ARG


def test_launch_count_query_checks_its_arguments(lib):
    n = ctypes.c_int(-1)
    # fp32 runs the two CUDA-core launches whatever the sizes
    assert lib.flashbob_bob_launches(1, 4, 4, 65536, 65536, 64, fb.FLASHBOB_F32,
                                     ctypes.byref(n)) == fb.FLASHBOB_OK
    assert n.value == 2
    for bad in ((0, 4, 4, 8, 8, 64), (1, 4, 3, 8, 8, 64), (1, 4, 4, 0, 8, 64),
                (1, 4, 4, 8, 8, 129)):
        assert lib.flashbob_bob_launches(*bad, fb.FLASHBOB_BF16, ctypes.byref(n)) != \
            fb.FLASHBOB_OK, bad
    assert lib.flashbob_bob_launches(1, 4, 4, 8, 8, 64, 7, ctypes.byref(n)) == \
        fb.FLASHBOB_ERR_INVALID_ARG
    assert lib.flashbob_bob_launches(1, 4, 4, 8, 8, 64, fb.FLASHBOB_BF16, None) == \
        fb.FLASHBOB_ERR_INVALID_ARG


def test_mma_cycles_rejects_bad_shapes_before_any_launch(lib):
    c = ctypes.c_double()
    for n in (0, 8, 24, 272, -16):
        assert lib.flashbob_mma_cycles(n, 0, None, ctypes.byref(c)) == \
            fb.FLASHBOB_ERR_INVALID_ARG, n
    assert lib.flashbob_mma_cycles(64, 1, None, None) == fb.FLASHBOB_ERR_INVALID_ARG
