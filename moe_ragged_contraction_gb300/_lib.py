"""ctypes binding of ``libmxfp8_wgrad.so`` (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels; this module
only turns torch tensors into device pointers, sizes and the current stream.
There is no fallback: if the library is missing or fails to load, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

OK = 0
EINVAL = -1
EALIGN = -2
ECUDA = -3
EUNSUPPORTED = -4
ENOWS = -5

DEV_OFFS_UNSORTED = 1
DEV_OFFS_RANGE = 2
DEV_OFFS_ALIGN = 4
DEV_WAIT_TIMEOUT = 8


class Mxfp8Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


def lib_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load the in-tree CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise ImportError(
                f"CUDA library {path} is missing: build it with "
                "`python -m moe_ragged_contraction_gb300.build` (or __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        P, I, L, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        lib.mxfp8_wgrad_grouped.argtypes = [P, P, P, P, P, I, I, I, L, P, P]
        lib.mxfp8_wgrad_grouped.restype = I
        lib.mxfp8_wgrad_workspace_bytes.argtypes = [I, I, I, L]
        lib.mxfp8_wgrad_workspace_bytes.restype = Z
        lib.mxfp8_wgrad_grouped_ws.argtypes = [P, P, P, P, P, I, I, I, L, P, P, Z, P]
        lib.mxfp8_wgrad_grouped_ws.restype = I
        lib.mxfp8_quantize_tokenwise.argtypes = [P, I, L, P, P, P]
        lib.mxfp8_quantize_tokenwise.restype = I
        lib.mxfp8_grouped_gemm.argtypes = [P, P, P, P, P, I, L, I, I, P, P]
        lib.mxfp8_grouped_gemm.restype = I
        lib.mxfp8_quantize_transpose_bf16.argtypes = [P, L, I, P, P, P]
        lib.mxfp8_quantize_transpose_bf16.restype = I
        lib.mxfp8_quantize_transpose_bf16_sf.argtypes = [P, L, I, I, P, P, P, P]
        lib.mxfp8_quantize_transpose_bf16_sf.restype = I
        lib.mxfp8_sf_blocks_bytes.argtypes = [I, L, I]
        lib.mxfp8_sf_blocks_bytes.restype = Z
        lib.mxfp8_wgrad_grouped_sf.argtypes = [P, P, P, P, P, I, I, I, L, I, I, P, P]
        lib.mxfp8_wgrad_grouped_sf.restype = I
        lib.mxfp8_last_error.argtypes = []
        lib.mxfp8_last_error.restype = ctypes.c_char_p
        lib.mxfp8_device_status.argtypes = [ctypes.POINTER(ctypes.c_int32), I]
        lib.mxfp8_device_status.restype = I
        lib.mxfp8_wgrad_set_timing_events.argtypes = [P, P]
        lib.mxfp8_wgrad_set_timing_events.restype = I
        lib.mxfp8_wgrad_set_tile_orientation.argtypes = [I]
        lib.mxfp8_wgrad_set_tile_orientation.restype = I
        IP = ctypes.POINTER(ctypes.c_int)
        lib.mxfp8_wgrad_set_tile_rows.argtypes = [I]
        lib.mxfp8_wgrad_set_tile_rows.restype = I
        lib.mxfp8_wgrad_set_epilogue_store.argtypes = [I]
        lib.mxfp8_wgrad_set_epilogue_store.restype = I
        lib.mxfp8_wgrad_tile_config.argtypes = [I, I, I, L, IP, IP, IP, IP]
        lib.mxfp8_wgrad_tile_config.restype = I
        lib.mxfp8_grouped_gemm_tile_config.argtypes = [I, I, I, L, IP, IP, IP]
        lib.mxfp8_grouped_gemm_tile_config.restype = I
        _lib = lib
        return lib


def check(rc: int) -> None:
    if rc != OK:
        msg = load().mxfp8_last_error().decode(errors="replace")
        raise Mxfp8Error(rc, msg)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _expect(t, dtype, name, device=True):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def wgrad_grouped(A, sA, B, sB, offs, out=None, workspace=None, stream=None):
    """dW[g] = dY[g]^T X[g] for every expert (see include/mxfp8_wgrad.h).

    A: uint8 [N, M] (E4M3), sA: uint8 [N, M/32] (E8M0), B: uint8 [K, M],
    sB: uint8 [K, M/32], offs: int32 [E] inclusive group ends (device).
    Returns (or fills) ``out``: bf16 [E, N, K].
    """
    import torch

    for t, dt, nm in ((A, torch.uint8, "A"), (sA, torch.uint8, "sA"), (B, torch.uint8, "B"),
                      (sB, torch.uint8, "sB"), (offs, torch.int32, "offs")):
        _expect(t, dt, nm)
    N, M = A.shape
    K, M2 = B.shape
    E = offs.numel()
    if M2 != M or tuple(sA.shape) != (N, M // 32) or tuple(sB.shape) != (K, M // 32):
        raise ValueError("inconsistent operand / scale shapes")
    if out is None:
        out = torch.empty((E, N, K), dtype=torch.bfloat16, device=A.device)
    _expect(out, torch.bfloat16, "out")
    if tuple(out.shape) != (E, N, K):
        raise ValueError(f"out must be [{E}, {N}, {K}]")
    lib = load()
    if workspace is None:
        rc = lib.mxfp8_wgrad_grouped(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(offs), E, N, K, M,
                                     _ptr(out), _stream(stream))
    else:
        _expect(workspace, torch.uint8, "workspace")
        rc = lib.mxfp8_wgrad_grouped_ws(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(offs), E, N, K, M,
                                        _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    check(rc)
    return out


def grouped_gemm(X, sX, W, sW, offs, out=None, stream=None):
    """Grouped GEMM with ragged rows (see include/mxfp8_wgrad.h):
    out[t] = x[t] . W[g(t)]^T for the rows t of group g.

    X: uint8 [M, K] (E4M3), sX: uint8 [M, K/32], W: uint8 [E, N, K],
    sW: uint8 [E, N, K/32], offs: int32 [E] inclusive group ends (device).
    Returns (or fills) ``out``: bf16 [M, N].
    """
    import torch

    for t, dt, nm in ((X, torch.uint8, "X"), (sX, torch.uint8, "sX"), (W, torch.uint8, "W"),
                      (sW, torch.uint8, "sW"), (offs, torch.int32, "offs")):
        _expect(t, dt, nm)
    M, K = X.shape
    E, N, K2 = W.shape
    if K2 != K or tuple(sX.shape) != (M, K // 32) or tuple(sW.shape) != (E, N, K // 32) or offs.numel() != E:
        raise ValueError("inconsistent operand / scale / offset shapes")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    _expect(out, torch.bfloat16, "out")
    if tuple(out.shape) != (M, N):
        raise ValueError(f"out must be [{M}, {N}]")
    check(load().mxfp8_grouped_gemm(_ptr(X), _ptr(sX), _ptr(W), _ptr(sW), _ptr(offs), E, M, N, K, _ptr(out),
                                    _stream(stream)))
    return out


def workspace_bytes(E: int, N: int, K: int, M: int) -> int:
    return int(load().mxfp8_wgrad_workspace_bytes(E, N, K, M))


ORIENT_AUTO, ORIENT_NK, ORIENT_KN = 0, 1, 2


def set_tile_orientation(mode: int) -> None:
    """Process-wide tile orientation: 0 automatic, 1 (256-row side on A), 2 (on B)."""
    check(load().mxfp8_wgrad_set_tile_orientation(int(mode)))


def set_tile_rows(tn: int) -> None:
    """Process-wide N-side tile width: 0 for the modelled choice, else a multiple of 16 in [16, 448]."""
    check(load().mxfp8_wgrad_set_tile_rows(int(tn)))


STORE_AUTO, STORE_DIRECT = 0, 1


def set_epilogue_store(mode: int) -> None:
    """Process-wide epilogue stores: 0 TMA stores where their staging fits, 1 direct stores only."""
    check(load().mxfp8_wgrad_set_epilogue_store(int(mode)))


def tile_config(E: int, N: int, K: int, M: int) -> dict:
    """Tiling the current settings give for E experts, an [N, K] output and M tokens."""
    v = [ctypes.c_int(0) for _ in range(4)]
    check(load().mxfp8_wgrad_tile_config(E, N, K, M, *(ctypes.byref(x) for x in v)))
    kn, tn, tm, tnn = (int(x.value) for x in v)
    return {"kn": kn, "tn": tn, "tiles_m": tm, "tiles_n": tnn}


def grouped_gemm_tile_config(E: int, N: int, K: int, M: int) -> dict:
    """Tiling the grouped GEMM would use for X [M, K] and W [E, N, K] under the current settings."""
    v = [ctypes.c_int(0) for _ in range(3)]
    check(load().mxfp8_grouped_gemm_tile_config(E, N, K, M, *(ctypes.byref(x) for x in v)))
    tn, tm, tnn = (int(x.value) for x in v)
    return {"tn": tn, "tiles_m_max": tm, "tiles_n": tnn}


def quantize_tokenwise(x, q=None, s=None, stream=None):
    """Tokenwise MXFP8 quantiser: x fp32 [R, M] -> (q uint8 [R, M], s uint8 [R, M/32])."""
    import torch

    _expect(x, torch.float32, "x")
    R, M = x.shape
    if q is None:
        q = torch.empty((R, M), dtype=torch.uint8, device=x.device)
    if s is None:
        s = torch.empty((R, M // 32), dtype=torch.uint8, device=x.device)
    _expect(q, torch.uint8, "q")
    _expect(s, torch.uint8, "s")
    check(load().mxfp8_quantize_tokenwise(_ptr(x), R, M, _ptr(q), _ptr(s), _stream(stream)))
    return q, s


def quantize_transpose_bf16(x, q=None, s=None, stream=None):
    """Fused quantise-and-transpose: x bf16 [M, R] (token-major) ->
    (q uint8 [R, M] E4M3, token axis contiguous; s uint8 [R, M/32] E8M0)."""
    import torch

    _expect(x, torch.bfloat16, "x")
    M, R = x.shape
    if q is None:
        q = torch.empty((R, M), dtype=torch.uint8, device=x.device)
    if s is None:
        s = torch.empty((R, M // 32), dtype=torch.uint8, device=x.device)
    _expect(q, torch.uint8, "q")
    _expect(s, torch.uint8, "s")
    if tuple(q.shape) != (R, M) or tuple(s.shape) != (R, M // 32):
        raise ValueError(f"q must be [{R}, {M}] and s [{R}, {M // 32}]")
    check(load().mxfp8_quantize_transpose_bf16(_ptr(x), M, R, _ptr(q), _ptr(s), _stream(stream)))
    return q, s


def sf_blocks_bytes(R: int, M: int, tile_rows: int) -> int:
    """Bytes of the scale-factor blocks of an [R, M] operand cut into tiles of tile_rows rows (0 if invalid)."""
    return int(load().mxfp8_sf_blocks_bytes(R, M, tile_rows))


def quantize_transpose_bf16_sf(x, tile_rows, q=None, sf=None, s=None, stream=None):
    """Fused quantise-and-transpose writing the scales as tcgen05 scale-factor
    blocks for tiles of ``tile_rows`` rows (see include/mxfp8_wgrad.h):
    x bf16 [M, R] -> (q uint8 [R, M] E4M3, sf uint8 [sf_blocks_bytes(R, M, tile_rows)],
    s uint8 [R, M/32] or None when not asked for)."""
    import torch

    _expect(x, torch.bfloat16, "x")
    M, R = x.shape
    nbytes = sf_blocks_bytes(R, M, tile_rows)
    if nbytes == 0:
        raise ValueError(f"invalid sizes R={R}, M={M}, tile_rows={tile_rows}")
    if q is None:
        q = torch.empty((R, M), dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty((nbytes,), dtype=torch.uint8, device=x.device)
    _expect(q, torch.uint8, "q")
    _expect(sf, torch.uint8, "sf")
    if s is not None:
        _expect(s, torch.uint8, "s")
        if tuple(s.shape) != (R, M // 32):
            raise ValueError(f"s must be [{R}, {M // 32}]")
    if tuple(q.shape) != (R, M) or sf.numel() < nbytes:
        raise ValueError(f"q must be [{R}, {M}] and sf hold {nbytes} bytes")
    check(load().mxfp8_quantize_transpose_bf16_sf(_ptr(x), M, R, int(tile_rows), _ptr(q), _ptr(s), _ptr(sf),
                                                  _stream(stream)))
    return q, sf, s


def wgrad_grouped_sf(A, sfA, B, sfB, offs, kn, tn, out=None, stream=None):
    """The weight gradient with scales given as scale-factor blocks laid out
    for the tiling (kn, tn) (see include/mxfp8_wgrad.h): sfA for tiles of
    (tn if kn else 256) rows of A, sfB for tiles of (256 if kn else tn) rows of B.
    A: uint8 [N, M], B: uint8 [K, M], offs: int32 [E]. Returns (or fills) out bf16 [E, N, K]."""
    import torch

    for t, dt, nm in ((A, torch.uint8, "A"), (sfA, torch.uint8, "sfA"), (B, torch.uint8, "B"),
                      (sfB, torch.uint8, "sfB"), (offs, torch.int32, "offs")):
        _expect(t, dt, nm)
    N, M = A.shape
    K, M2 = B.shape
    E = offs.numel()
    rows_a, rows_b = (int(tn), 256) if kn else (256, int(tn))
    if M2 != M or sfA.numel() < sf_blocks_bytes(N, M, rows_a) or sfB.numel() < sf_blocks_bytes(K, M, rows_b):
        raise ValueError("inconsistent operand / scale-factor block sizes")
    if out is None:
        out = torch.empty((E, N, K), dtype=torch.bfloat16, device=A.device)
    _expect(out, torch.bfloat16, "out")
    if tuple(out.shape) != (E, N, K):
        raise ValueError(f"out must be [{E}, {N}, {K}]")
    check(load().mxfp8_wgrad_grouped_sf(_ptr(A), _ptr(sfA), _ptr(B), _ptr(sfB), _ptr(offs), E, N, K, M, int(kn),
                                        int(tn), _ptr(out), _stream(stream)))
    return out


def device_status(clear: bool = True) -> int:
    """Device status word (DEV_* bits); synchronises the current device."""
    v = ctypes.c_int32(0)
    check(load().mxfp8_device_status(ctypes.byref(v), 1 if clear else 0))
    return int(v.value)


def set_timing_events(ev_before, ev_after) -> None:
    """Record torch.cuda.Event pair around the main kernel of the next call."""
    b = ctypes.c_void_p(ev_before.cuda_event) if ev_before is not None else None
    a = ctypes.c_void_p(ev_after.cuda_event) if ev_after is not None else None
    check(load().mxfp8_wgrad_set_timing_events(b, a))
