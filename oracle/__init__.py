"""CPU oracle for the ragged MXFP8 weight-gradient grouped GEMM.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. It shares no code
with the CUDA library (``moe_ragged_contraction_gb300``) and never imports it.

Source of the arithmetic ("Ragged MXFP8 Weight Gradients: A FlyDSL Grouped GEMM
on MI355X", section 1 and section 5.5; "Group-GEMM in XLA", Part 3,
"Contracting"):

    out[g, n, k] = bf16_rne( sum over tokens t in [offs[g-1], offs[g]) of
                     e4m3(A[n,t]) 2^(sA[n,t/32]-127) * e4m3(B[k,t]) 2^(sB[k,t/32]-127) )

computed in fp64 by ``oracle.c`` (plain triple loop, token order) and rounded
to bf16 in one step. ``grouped_gemm`` is the non-contracting form in MXFP8
("Group-GEMM in XLA", Part 1, "The Ragged-Dot Operation"; the forward and
data-gradient products of the same expert layer):

    out[t, n] = bf16_rne( sum over k of e4m3(X[t,k]) 2^(sX[t,k/32]-127) *
                          e4m3(W[g,n,k]) 2^(sW[g,n,k/32]-127) ),  g = group of row t,

rows past offs[E-1] zero. ``ragged_dot.py`` holds the generic fp64 ragged-dot forms
(non-contracting and contracting) used to pin the worked example of the XLA
page.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (exact rational brute force, hand-computed
values, library decode tables, dense-GEMM special cases, the sum invariant and
the worked example).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc into ``liboracle.so`` (in-tree)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I = ctypes.c_int
        L = ctypes.c_int64
        lib.oracle_dec_e4m3.argtypes = [ctypes.c_uint8]
        lib.oracle_dec_e4m3.restype = ctypes.c_double
        lib.oracle_dec_e8m0.argtypes = [ctypes.c_uint8]
        lib.oracle_dec_e8m0.restype = ctypes.c_double
        lib.oracle_bf16_rne.argtypes = [ctypes.c_double]
        lib.oracle_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_wgrad.argtypes = [P, P, P, P, P, I, I, I, L, P, P, P, I]
        lib.oracle_wgrad.restype = I
        lib.oracle_wgrad_points.argtypes = [P, P, P, P, P, I, I, I, L, P, P, P, L, P, P, P, I]
        lib.oracle_wgrad_points.restype = I
        lib.oracle_grouped_gemm.argtypes = [P, P, P, P, P, I, L, I, I, P, P, L, P, P, P, I]
        lib.oracle_grouped_gemm.restype = I
        lib.oracle_quantize_tokenwise.argtypes = [P, L, L, P, P, I]
        lib.oracle_quantize_tokenwise.restype = I
        _lib = lib
        return lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def dec_e4m3(b: int) -> float:
    return _load().oracle_dec_e4m3(int(b))


def dec_e8m0(b: int) -> float:
    return _load().oracle_dec_e8m0(int(b))


def bf16_rne(x: float) -> int:
    """fp64 -> bf16 bit pattern, round to nearest even."""
    return int(_load().oracle_bf16_rne(float(x)))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp64 values (exact)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def wgrad(A, sA, B, sB, offs, E, N, K, M, want_acc=False, nthreads=None):
    """Full output. Returns bf16 bits [E,N,K] (uint16); with ``want_acc`` also
    the fp64 sums and the fp64 sums of |a*b| (both [E,N,K])."""
    lib = _load()
    A = _c(A, np.uint8); sA = _c(sA, np.uint8)
    B = _c(B, np.uint8); sB = _c(sB, np.uint8)
    offs = _c(offs, np.int32)
    assert A.size == N * M and B.size == K * M
    assert sA.size == N * (M // 32) and sB.size == K * (M // 32) and offs.size == E
    out = np.empty((E, N, K), dtype=np.uint16)
    acc = np.empty((E, N, K), dtype=np.float64) if want_acc else None
    aacc = np.empty((E, N, K), dtype=np.float64) if want_acc else None
    rc = lib.oracle_wgrad(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(offs), E, N, K, M,
                          _ptr(out), _ptr(acc) if want_acc else None,
                          _ptr(aacc) if want_acc else None,
                          nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_wgrad: invalid arguments or offsets")
    return (out, acc, aacc) if want_acc else out


def wgrad_points(A, sA, B, sB, offs, E, N, K, M, g, n, k, want_acc=False, nthreads=None):
    """Selected elements (g[i], n[i], k[i]). Returns bf16 bits [P] (and fp64
    sums and sums of |a*b| with ``want_acc``)."""
    lib = _load()
    A = _c(A, np.uint8); sA = _c(sA, np.uint8)
    B = _c(B, np.uint8); sB = _c(sB, np.uint8)
    offs = _c(offs, np.int32)
    g = _c(g, np.int32); n = _c(n, np.int32); k = _c(k, np.int32)
    P = g.size
    assert n.size == P and k.size == P
    out = np.empty(P, dtype=np.uint16)
    acc = np.empty(P, dtype=np.float64)
    aacc = np.empty(P, dtype=np.float64)
    rc = lib.oracle_wgrad_points(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(offs), E, N, K, M,
                                 _ptr(g), _ptr(n), _ptr(k), P, _ptr(out), _ptr(acc), _ptr(aacc),
                                 nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_wgrad_points: invalid arguments, offsets or indices")
    return (out, acc, aacc) if want_acc else out


def grouped_gemm(X, sX, W, sW, offs, E, M, N, K, points=None, want_acc=False, nthreads=None):
    """Non-contracting ragged dot in MXFP8: out[t, n] for every row t of group
    g = sum_k x(t, k) w(g, n, k); X [M,K], sX [M,K/32], W [E,N,K], sW
    [E,N,K/32]; rows past offs[E-1] are zero. Returns bf16 bits [M,N] (or [P]
    for ``points`` = (t, n) index arrays), with ``want_acc`` also the fp64 sums
    and the fp64 sums of |x*w|."""
    lib = _load()
    X = _c(X, np.uint8); sX = _c(sX, np.uint8)
    W = _c(W, np.uint8); sW = _c(sW, np.uint8)
    offs = _c(offs, np.int32)
    assert X.size == M * K and sX.size == M * (K // 32)
    assert W.size == E * N * K and sW.size == E * N * (K // 32) and offs.size == E
    if points is None:
        shape = (M, N)
        pt = pn = None
        P = 0
    else:
        pt = _c(points[0], np.int64); pn = _c(points[1], np.int64)
        assert pt.size == pn.size
        P = pt.size
        shape = (P,)
    out = np.empty(shape, dtype=np.uint16)
    acc = np.empty(shape, dtype=np.float64) if want_acc else None
    aacc = np.empty(shape, dtype=np.float64) if want_acc else None
    rc = lib.oracle_grouped_gemm(_ptr(X), _ptr(sX), _ptr(W), _ptr(sW), _ptr(offs), E, M, N, K,
                                 _ptr(pt) if pt is not None else None, _ptr(pn) if pn is not None else None, P,
                                 _ptr(out), _ptr(acc) if want_acc else None, _ptr(aacc) if want_acc else None,
                                 nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_grouped_gemm: invalid arguments, offsets or points")
    return (out, acc, aacc) if want_acc else out


def quantize_tokenwise(x, nthreads=None):
    """x fp32 [R,M] -> (q E4M3 bytes [R,M], s E8M0 bytes [R,M/32])."""
    lib = _load()
    x = _c(x, np.float32)
    R, M = x.shape
    q = np.empty((R, M), dtype=np.uint8)
    s = np.empty((R, M // 32), dtype=np.uint8)
    rc = lib.oracle_quantize_tokenwise(_ptr(x), R, M, _ptr(q), _ptr(s), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_quantize_tokenwise: M must be a multiple of 32")
    return q, s


def decode_operand(q, s):
    """Dequantise an operand (exact in fp64): q [R,M] E4M3, s [R,M/32] E8M0."""
    lut = np.array([dec_e4m3(i) for i in range(256)], dtype=np.float64)
    slut = np.array([dec_e8m0(i) for i in range(256)], dtype=np.float64)
    q = np.asarray(q, dtype=np.uint8)
    s = np.asarray(s, dtype=np.uint8)
    return lut[q] * np.repeat(slut[s], 32, axis=1)
