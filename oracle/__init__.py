"""CPU oracle of the MLA paged decode step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import, call, link or run anything in this package.  The
GPU library never imports it, and it never imports the GPU library: the two
share nothing but the seeded input generators.

Contents:
  * ``mla_oracle``   -- plain fp64 NumPy definition of every step;
  * ``brute``        -- pure-Python scalar loops of the same, for tiny inputs;
  * ``mla_oracle_c.c`` -- plain fp64 C restatement (OpenMP over requests),
    the timed CPU baseline; built by :func:`build_c` with gcc.

Parity status: every function is pinned by CPU tests (``tests/test_oracle.py``)
against closed forms, invariants, library routines and the brute force.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
C_SRC = os.path.join(_HERE, "mla_oracle_c.c")
C_LIB = os.path.join(_HERE, "_build", "libmla_oracle_c.so")


def build_c(force: bool = False) -> str:
    """Compile the C oracle to a shared library (gcc, OpenMP, portable
    flags: the same source builds on x86_64 and aarch64)."""
    if not force and os.path.exists(C_LIB) and os.path.getmtime(C_LIB) >= os.path.getmtime(C_SRC):
        return C_LIB
    os.makedirs(os.path.dirname(C_LIB), exist_ok=True)
    tmp = C_LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, C_SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, C_LIB)
    return C_LIB


_lib = None


def load_c():
    """ctypes handle of the C oracle (built on first use)."""
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_c())
        lib.mla_oracle_decode_step.restype = ctypes.c_int
        lib.mla_oracle_decode_step.argtypes = [
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
            ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
        lib.mla_oracle_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def decode_step_c(q_bits, kv_codes, pages, indptr, scale, kv_scale, heads, qlen,
                  w_uv_bits, gate_bits, requests=None, threads=0):
    """Run the C oracle on numpy inputs; returns (latent, lse, out) float64
    arrays of the full [S, ...] shapes (rows of requests not computed stay
    NaN)."""
    import numpy as np

    lib = load_c()
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    kv = np.ascontiguousarray(kv_codes, dtype=np.uint8)
    pages = np.ascontiguousarray(pages, dtype=np.int32)
    indptr = np.ascontiguousarray(indptr, dtype=np.int32)
    w = np.ascontiguousarray(w_uv_bits, dtype=np.uint16)
    g = np.ascontiguousarray(gate_bits, dtype=np.uint16)
    R = len(indptr) - 1
    S = R * qlen
    latent = np.full((S, heads, 512), np.nan)
    lse = np.full((S, heads), np.nan)
    out = np.full((S, heads * 128), np.nan)
    req = None if requests is None else np.ascontiguousarray(requests, dtype=np.int32)
    p = lambda a: None if a is None else a.ctypes.data  # noqa: E731
    rc = lib.mla_oracle_decode_step(
        p(q), q.shape[1] * q.shape[2], p(kv), p(pages), p(indptr), R, qlen, heads,
        float(scale), float(kv_scale), p(w), p(g), p(latent), p(lse), p(out), p(req),
        0 if req is None else len(req), int(threads))
    if rc != 0:
        raise MemoryError("C oracle failed to allocate")
    return latent, lse, out
