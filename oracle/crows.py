"""ctypes binding of the plain-C row-scalar oracle (``oracle/rowscal.c``).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``.  ``row_scalars``
returns the same L, D, alpha, E as ``oracle.bob.row_scalars`` (fp64, same
definitions), fast enough for one (batch, head) of a 64K-262K sequence in
the GPU tests' time budget.  The library is compiled with gcc on first use
(or by ``build()``) into ``oracle/_build/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "rowscal.c")
LIB = os.path.join(HERE, "_build", "liboracle_rows.so")

_lib = None


def build() -> str:
    """Compile rowscal.c (gcc, OpenMP, no fast-math: IEEE fp64 throughout;
    a multiply-add may be fused where the machine has an FMA instruction)."""
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O3", "-fopenmp", "-fPIC", "-shared", "-o", tmp, SRC, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"gcc failed on {SRC}:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
            build()
        lib = ctypes.CDLL(LIB)
        f = lib.oracle_row_scalars
        P = ctypes.c_void_p
        f.argtypes = [P] * 7 + [ctypes.c_int] * 3 + [ctypes.c_double, ctypes.c_int] + [P] * 4
        f.restype = ctypes.c_int
        _lib = lib
    return _lib


def row_scalars(Q, K, V, dO, UQ, UK, UV, tau, causal=False):
    """L, D, alpha, E of every query row of one (batch, head).

    Q, dO, UQ: [N_q, d]; K, V, UK, UV: [N_k, d]; any real dtype whose values
    are exact in fp32 (the bf16 and fp32 inputs of the workloads)."""
    lib = _load()
    arrs = [np.ascontiguousarray(np.asarray(x, dtype=np.float32)) for x in
            (Q, K, V, dO, UQ, UK, UV)]
    for x, src in zip(arrs, (Q, K, V, dO, UQ, UK, UV)):
        if not np.array_equal(x.astype(np.float64), np.asarray(src, dtype=np.float64)):
            raise ValueError("inputs must be exactly representable in fp32")
    Nq, d = arrs[0].shape
    Nk = arrs[1].shape[0]
    out = {k: np.empty(Nq, dtype=np.float64) for k in ("L", "D", "alpha", "E")}
    rc = lib.oracle_row_scalars(*[x.ctypes.data for x in arrs], Nq, Nk, d, float(tau),
                                1 if causal else 0,
                                *[out[k].ctypes.data for k in ("L", "D", "alpha", "E")])
    if rc != 0:
        raise RuntimeError(f"oracle_row_scalars failed ({rc})")
    return out
