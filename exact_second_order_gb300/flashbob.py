"""Python binding of libflashbob (argument marshalling only).

The functions carry the C names of ``include/flashbob.h``.  Tensors are
PyTorch CUDA tensors used only as device memory; every step of the
computation runs in the library's kernels.  Loading fails loudly when the
library has not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libflashbob.so")

FLASHBOB_OK = 0
FLASHBOB_ERR_INVALID_ARG = 1
FLASHBOB_ERR_UNSUPPORTED = 2
FLASHBOB_ERR_MISALIGNED = 3
FLASHBOB_ERR_CUDA = 4
FLASHBOB_ERR_TIMEOUT = 5
FLASHBOB_F32 = 0
FLASHBOB_BF16 = 1

# Every entry point the header declares, with its ctypes signature.
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SIGNATURES = {
    "flashbob_prep": ([_P] * 7 + [_I] * 6 + [_F, _I, _I, _P], _I),
    "flashbob_bob": ([_P] * 10 + [_F] + [_P] * 6 + [_I] * 8 + [_P], _I),
    "flashbob_bob_pass1": ([_P] * 10 + [_F] + [_P] * 4 + [_I] * 8 + [_P], _I),
    "flashbob_bob_pass2": ([_P] * 11 + [_F] + [_P] * 2 + [_I] * 8 + [_P], _I),
    "flashbob_attention_jvp": ([_P] * 8 + [_F] + [_P] * 2 + [_I] * 8 + [_P], _I),
    "flashbob_bob_launches": ([_I] * 7 + [ctypes.POINTER(_I)], _I),
    "flashbob_bob_tile_sizes": ([_I, _I] + [ctypes.POINTER(_I)] * 4
                                + [ctypes.POINTER(ctypes.c_size_t)] * 2, _I),
    "flashbob_last_device_error": ([], _I),
    "flashbob_check_wait_timeout": ([_P], _I),
    "flashbob_mma_cycles": ([_I, _I, _P, ctypes.POINTER(ctypes.c_double)], _I),
    "flashbob_status_string": ([_I], ctypes.c_char_p),
}

_lib = None


class FlashbobError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {flashbob_status_string(status)}")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libflashbob.so (once) and declare the signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with exact_second_order_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (args, res) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return FLASHBOB_F32
    if t.dtype == torch.bfloat16:
        return FLASHBOB_BF16
    raise TypeError(f"unsupported input dtype {t.dtype}")


def _stream_handle(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _check(where: str, Q, K, spec) -> None:
    """The C ABI sees only pointers and sizes, so the binding checks what the
    header fixes for each tensor before handing its pointer on: a CUDA tensor
    on Q's device, contiguous (row-major), with the shape and dtype of its
    role.  ``spec`` lists (name, tensor, role, dtype) with role "q"
    ([B, H, N_q, d]), "k" ([B, H_kv, N_k, d]) or "row" ([B, H, N_q]) and
    dtype "in" (the inputs' common dtype, Q's) or "f32"; None tensors are
    skipped (the ABI decides which may be NULL)."""
    import torch
    for name, t in (("Q", Q), ("K", K)):
        if not isinstance(t, torch.Tensor) or t.dim() != 4:
            raise ValueError(f"{where}: {name} must be a 4-d tensor [B, heads, rows, d]")
    B, H, Nq, d = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    shapes = {"q": (B, H, Nq, d), "k": (B, Hkv, Nk, d), "row": (B, H, Nq)}
    for name, t, role, dt in spec:
        if t is None:
            continue
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.device != Q.device:
            raise ValueError(f"{where}: {name} must be a CUDA tensor on {Q.device}")
        if tuple(t.shape) != shapes[role]:
            raise ValueError(f"{where}: {name} has shape {tuple(t.shape)}, "
                             f"expected {shapes[role]}")
        want = Q.dtype if dt == "in" else torch.float32
        if t.dtype != want:
            raise TypeError(f"{where}: {name} is {t.dtype}, expected {want}")
        if not t.is_contiguous():
            raise ValueError(f"{where}: {name} must be contiguous")


def _input_specs(Q, K, V, dO, UQ, UK, UV):
    """Check list of the seven inputs of the BoB calls (one common dtype)."""
    return [("Q", Q, "q", "in"), ("K", K, "k", "in"), ("V", V, "k", "in"),
            ("dO", dO, "q", "in"), ("UQ", UQ, "q", "in"), ("UK", UK, "k", "in"),
            ("UV", UV, "k", "in")]


def _device(t):
    """The CUDA device context of tensor ``t``: the library works on the
    current device, so every call runs with its tensors' device current."""
    import torch
    return torch.cuda.device(t.device)


def flashbob_status_string(status: int) -> str:
    return load_library().flashbob_status_string(status).decode()


def flashbob_prep(Q, K, V, dO, O, L, D, tau: float, causal: bool = False, stream=None) -> None:
    """O, L, D of [B, H, Nq, d] queries and [B, Hkv, Nk, d] keys/values
    (see flashbob_prep in the header); dO = D = None computes O and L only."""
    _check("flashbob_prep", Q, K, [("Q", Q, "q", "in"), ("K", K, "k", "in"),
                                    ("V", V, "k", "in"), ("dO", dO, "q", "in"),
                                    ("O", O, "q", "f32"), ("L", L, "row", "f32"),
                                    ("D", D, "row", "f32")])
    B, H, Nq, d = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    with _device(Q):
        st = load_library().flashbob_prep(
            _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(O), _ptr(L), _ptr(D), B, H, Hkv, Nq, Nk,
            d, float(tau), int(causal), _dtype_code(Q), _stream_handle(stream))
    if st != FLASHBOB_OK:
        raise FlashbobError(st, "flashbob_prep")


def flashbob_bob(Q, K, V, O, dO, L, D, UQ, UK, UV, tau: float, dQt, dKt, dVt, ddOt, alpha, E,
                 causal: bool = False, stream=None) -> None:
    """d~Q, d~K, d~V, d~dO, alpha, E (see flashbob_bob in the header)."""
    _check("flashbob_bob", Q, K, _input_specs(Q, K, V, dO, UQ, UK, UV) + [
        ("O", O, "q", "f32"), ("L", L, "row", "f32"), ("D", D, "row", "f32"),
        ("dQt", dQt, "q", "f32"), ("dKt", dKt, "k", "f32"), ("dVt", dVt, "k", "f32"),
        ("ddOt", ddOt, "q", "f32"), ("alpha", alpha, "row", "f32"), ("E", E, "row", "f32")])
    B, H, Nq, d = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    with _device(Q):
        st = load_library().flashbob_bob(
            _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(L), _ptr(D), _ptr(UQ),
            _ptr(UK), _ptr(UV), float(tau), _ptr(dQt), _ptr(dKt), _ptr(dVt), _ptr(ddOt),
            _ptr(alpha), _ptr(E), B, H, Hkv, Nq, Nk, d, int(causal), _dtype_code(Q),
            _stream_handle(stream))
    if st != FLASHBOB_OK:
        raise FlashbobError(st, "flashbob_bob")


def flashbob_bob_pass1(Q, K, V, O, dO, L, D, UQ, UK, UV, tau: float, dQt, ddOt, alpha, E,
                       causal: bool = False, stream=None) -> None:
    """Pass 1 only: d~Q, d~dO, alpha, E (see flashbob_bob_pass1 in the header)."""
    _check("flashbob_bob_pass1", Q, K, _input_specs(Q, K, V, dO, UQ, UK, UV) + [
        ("O", O, "q", "f32"), ("L", L, "row", "f32"), ("D", D, "row", "f32"),
        ("dQt", dQt, "q", "f32"), ("ddOt", ddOt, "q", "f32"), ("alpha", alpha, "row", "f32"),
        ("E", E, "row", "f32")])
    B, H, Nq, d = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    with _device(Q):
        st = load_library().flashbob_bob_pass1(
            _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(L), _ptr(D), _ptr(UQ),
            _ptr(UK), _ptr(UV), float(tau), _ptr(dQt), _ptr(ddOt), _ptr(alpha), _ptr(E), B, H,
            Hkv, Nq, Nk, d, int(causal), _dtype_code(Q), _stream_handle(stream))
    if st != FLASHBOB_OK:
        raise FlashbobError(st, "flashbob_bob_pass1")


def flashbob_bob_pass2(Q, K, V, dO, L, D, alpha, E, UQ, UK, UV, tau: float, dKt, dVt,
                       causal: bool = False, stream=None) -> None:
    """Pass 2 only: d~K, d~V from pass 1's alpha, E (see flashbob_bob_pass2)."""
    _check("flashbob_bob_pass2", Q, K, _input_specs(Q, K, V, dO, UQ, UK, UV) + [
        ("L", L, "row", "f32"), ("D", D, "row", "f32"), ("alpha", alpha, "row", "f32"),
        ("E", E, "row", "f32"), ("dKt", dKt, "k", "f32"), ("dVt", dVt, "k", "f32")])
    B, H, Nq, d = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    with _device(Q):
        st = load_library().flashbob_bob_pass2(
            _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(L), _ptr(D), _ptr(alpha), _ptr(E),
            _ptr(UQ), _ptr(UK), _ptr(UV), float(tau), _ptr(dKt), _ptr(dVt), B, H, Hkv, Nq, Nk,
            d, int(causal), _dtype_code(Q), _stream_handle(stream))
    if st != FLASHBOB_OK:
        raise FlashbobError(st, "flashbob_bob_pass2")


def flashbob_attention_jvp(Q, K, V, O, L, UQ, UK, UV, tau: float, Od, Ld,
                           causal: bool = False, stream=None) -> None:
    """O' and L' along the tangents (U_Q, U_K, U_V) (see flashbob_attention_jvp)."""
    _check("flashbob_attention_jvp", Q, K, [
        ("Q", Q, "q", "in"), ("K", K, "k", "in"), ("V", V, "k", "in"), ("UQ", UQ, "q", "in"),
        ("UK", UK, "k", "in"), ("UV", UV, "k", "in"), ("O", O, "q", "f32"),
        ("L", L, "row", "f32"), ("Od", Od, "q", "f32"), ("Ld", Ld, "row", "f32")])
    B, H, Nq, d = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    with _device(Q):
        st = load_library().flashbob_attention_jvp(
            _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(L), _ptr(UQ), _ptr(UK), _ptr(UV),
            float(tau), _ptr(Od), _ptr(Ld), B, H, Hkv, Nq, Nk, d, int(causal), _dtype_code(Q),
            _stream_handle(stream))
    if st != FLASHBOB_OK:
        raise FlashbobError(st, "flashbob_attention_jvp")


def flashbob_bob_launches(B: int, H: int, Hkv: int, Nq: int, Nk: int, d: int,
                          in_dtype: int) -> int:
    """Kernel launches of one flashbob_bob call with these sizes."""
    n = ctypes.c_int()
    st = load_library().flashbob_bob_launches(B, H, Hkv, Nq, Nk, d, in_dtype, ctypes.byref(n))
    if st != FLASHBOB_OK:
        raise FlashbobError(st, "flashbob_bob_launches")
    return n.value


def flashbob_bob_tile_sizes(d: int, in_dtype: int) -> dict:
    """Tiles and dynamic shared memory of flashbob_bob for (d, in_dtype)."""
    v = [ctypes.c_int() for _ in range(4)]
    s = [ctypes.c_size_t() for _ in range(2)]
    st = load_library().flashbob_bob_tile_sizes(d, in_dtype, *(ctypes.byref(x) for x in v),
                                                *(ctypes.byref(x) for x in s))
    if st != FLASHBOB_OK:
        raise FlashbobError(st, "flashbob_bob_tile_sizes")
    return {"Br1": v[0].value, "Bc1": v[1].value, "Br2": v[2].value, "Bc2": v[3].value,
            "smem_bytes_pass1": s[0].value, "smem_bytes_pass2": s[1].value}


def flashbob_check_wait_timeout(stream=None) -> None:
    """Launch the diagnostic whose bounded wait runs out (see the header)."""
    st = load_library().flashbob_check_wait_timeout(_stream_handle(stream))
    if st != FLASHBOB_OK:
        raise FlashbobError(st, "flashbob_check_wait_timeout")


def flashbob_mma_cycles(n: int, a_in_tmem: bool, stream=None) -> float:
    """SM cycles per tcgen05.mma of M = 128, N = n, K = 16 (see the header)."""
    c = ctypes.c_double()
    st = load_library().flashbob_mma_cycles(n, int(a_in_tmem), _stream_handle(stream),
                                             ctypes.byref(c))
    if st != FLASHBOB_OK:
        raise FlashbobError(st, "flashbob_mma_cycles")
    return c.value


def flashbob_last_device_error() -> int:
    """Status of the device error word (synchronises the device, then clears)."""
    return load_library().flashbob_last_device_error()


# ---------------------------------------------------------------------------
# Convenience wrappers: allocate the outputs with torch, then call the ABI.
# ---------------------------------------------------------------------------

def prep(Q, K, V, dO, tau: float, causal: bool = False, stream=None):
    """Allocate O, L, D on Q's device and run flashbob_prep (dO = None: the
    forward only, D is returned as None)."""
    import torch
    B, H, Nq, d = Q.shape
    O = torch.empty((B, H, Nq, d), dtype=torch.float32, device=Q.device)
    L = torch.empty((B, H, Nq), dtype=torch.float32, device=Q.device)
    D = None if dO is None else torch.empty((B, H, Nq), dtype=torch.float32, device=Q.device)
    flashbob_prep(Q, K, V, dO, O, L, D, tau, causal, stream)
    return O, L, D


def attention_jvp(Q, K, V, UQ, UK, UV, tau: float, causal: bool = False, O=None, L=None,
                  stream=None):
    """O, L (from flashbob_prep when not given) and the tangents O', L'."""
    import torch
    if O is None or L is None:
        O, L, _ = prep(Q, K, V, None, tau, causal, stream)
    Od = torch.empty_like(O)
    Ld = torch.empty_like(L)
    flashbob_attention_jvp(Q, K, V, O, L, UQ, UK, UV, tau, Od, Ld, causal, stream)
    return O, L, Od, Ld


def alloc_bob_outputs(Q, fill: float | None = None, K=None) -> dict:
    """fp32 output buffers of flashbob_bob (optionally filled, e.g. with NaN);
    d~K and d~V take K's head count and length (grouped-query, rectangular
    attention) when K is given."""
    import torch
    B, H, Nq, d = Q.shape
    Hkv, Nk = (K.shape[1], K.shape[2]) if K is not None else (H, Nq)
    out = {k: torch.empty((B, H, Nq, d), dtype=torch.float32, device=Q.device)
           for k in ("dQt", "ddOt")}
    out.update({k: torch.empty((B, Hkv, Nk, d), dtype=torch.float32, device=Q.device)
                for k in ("dKt", "dVt")})
    out.update({k: torch.empty((B, H, Nq), dtype=torch.float32, device=Q.device)
                for k in ("alpha", "E")})
    if fill is not None:
        for t in out.values():
            t.fill_(fill)
    return out


def bob(Q, K, V, O, dO, L, D, UQ, UK, UV, tau: float, out: dict | None = None,
        causal: bool = False, stream=None):
    """Run flashbob_bob into ``out`` (allocated when None); returns the dict."""
    if out is None:
        out = alloc_bob_outputs(Q, K=K)
    flashbob_bob(Q, K, V, O, dO, L, D, UQ, UK, UV, tau, out["dQt"], out["dKt"], out["dVt"],
                 out["ddOt"], out["alpha"], out["E"], causal, stream)
    return out
