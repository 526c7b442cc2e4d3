"""CPU-side checks of the C ABI: the library builds for sm_103a, loads without
a GPU, exports every function include/*.h declares, and rejects invalid
arguments on the host (no compute call is made here)."""
import ctypes
import glob
import os
import re

import pytest

import moe_ragged_contraction_gb300 as mx
from moe_ragged_contraction_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mx.build()
    return mx.load()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(mxfp8_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("mxfp8_wgrad_grouped", "mxfp8_quantize_tokenwise", "mxfp8_wgrad_grouped_ws",
              "mxfp8_wgrad_workspace_bytes", "mxfp8_last_error", "mxfp8_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_workspace_bytes(lib):
    f = lib.mxfp8_wgrad_workspace_bytes
    assert f(0, 128, 256, 1024) == 0
    assert f(4, 128, 256, 1000) == 0  # M % 32 != 0
    assert f(4, 128, 256, 1024) > 0
    # grows with tokens, rows and columns
    assert f(8, 1408, 2048, 65536) > f(8, 1408, 2048, 32768) > f(8, 128, 2048, 32768)


P = 0x10000  # 16-byte aligned fake address: never dereferenced on these paths


def call(lib, A=P, sA=P, B=P, sB=P, offs=P, E=4, N=128, K=256, M=1024, out=P):
    return lib.mxfp8_wgrad_grouped(A, sA, B, sB, offs, E, N, K, M, out, None)


@pytest.mark.parametrize("kw,code", [
    (dict(E=-1), _lib.EINVAL), (dict(E=100000), _lib.EINVAL), (dict(N=0), _lib.EINVAL),
    (dict(K=0), _lib.EINVAL), (dict(M=1000), _lib.EINVAL), (dict(M=0), _lib.EINVAL),
    (dict(A=None), _lib.EINVAL), (dict(offs=None), _lib.EINVAL), (dict(out=None), _lib.EINVAL),
    (dict(A=P + 8), _lib.EALIGN), (dict(out=P + 4), _lib.EALIGN), (dict(K=260), _lib.EALIGN),
])
def test_host_validation(lib, kw, code):
    assert call(lib, **kw) == code
    assert len(lib.mxfp8_last_error()) > 0


def test_empty_expert_count_is_noop(lib):
    assert call(lib, E=0, A=None, sA=None, B=None, sB=None, offs=None, out=None) == _lib.OK


def test_ws_variant_checks_size(lib):
    need = lib.mxfp8_wgrad_workspace_bytes(4, 128, 256, 1024)
    rc = lib.mxfp8_wgrad_grouped_ws(P, P, P, P, P, 4, 128, 256, 1024, P, P, need - 1, None)
    assert rc == _lib.ENOWS
    rc = lib.mxfp8_wgrad_grouped_ws(P, P, P, P, P, 4, 128, 256, 1024, P, P + 16, need, None)
    assert rc == _lib.EALIGN  # workspace needs 256-byte alignment


def test_quantize_validation(lib):
    q = lib.mxfp8_quantize_tokenwise
    assert q(P, 0, 1024, P, P, None) == _lib.EINVAL
    assert q(P, 4, 1000, P, P, None) == _lib.EINVAL
    assert q(None, 4, 1024, P, P, None) == _lib.EINVAL
    assert q(P + 4, 4, 1024, P, P, None) == _lib.EALIGN


def test_timing_events_pairing(lib):
    assert lib.mxfp8_wgrad_set_timing_events(ctypes.c_void_p(P), None) == _lib.EINVAL
    assert lib.mxfp8_wgrad_set_timing_events(None, None) == _lib.OK


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib._build, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(ImportError):
        _lib.load()


def test_tile_config_choice(lib):
    """Host-side tiling: the automatic mode follows the kernel's cost model
    (bytes per step against MMA cycles, padding, tile count); either
    orientation and any admissible tile width can be forced; invalid settings
    fail."""
    try:
        mx.set_tile_orientation(0)
        mx.set_tile_rows(0)
        # 16B expert shape: K = 2048 = 8 x 256 on the 256 side (B), N = 1408 = 4 x 352
        # (two MMAs, TMA stores of the transposed chunks): no padding on either side
        assert mx.tile_config(8, 1408, 2048, 32768) == {"kn": 1, "tn": 352, "tiles_m": 8, "tiles_n": 4}
        assert mx.tile_config(8, 1408, 2048, 196608) == {"kn": 1, "tn": 352, "tiles_m": 8, "tiles_n": 4}
        # 671B up/gate: K = 7168 = 16 x 448 with the 256 side on A (N = 4096)
        assert mx.tile_config(32, 4096, 7168, 262144) == {"kn": 0, "tn": 448, "tiles_m": 16, "tiles_n": 16}
        # 671B down: K = 2048 = 8 x 256 on the 256 side (B), N = 7168 = 16 x 448, every
        # transposed chunk staged for a TMA store; forced onto A, 5 tiles of 416 (1.6% padding)
        assert mx.tile_config(32, 7168, 2048, 524288) == {"kn": 1, "tn": 448, "tiles_m": 8, "tiles_n": 16}
        mx.set_tile_orientation(1)
        assert mx.tile_config(32, 7168, 2048, 524288) == {"kn": 0, "tn": 416, "tiles_m": 28, "tiles_n": 5}
        mx.set_tile_orientation(0)
        # many experts with 32 tokens each: bound by writing the output; the widest
        # tiles whose chunks are all written by staged TMA stores
        assert mx.tile_config(512, 512, 2048, 16384) == {"kn": 0, "tn": 448, "tiles_m": 2, "tiles_n": 5}
        mx.set_tile_orientation(1)
        assert mx.tile_config(8, 1408, 2048, 32768) == {"kn": 0, "tn": 416, "tiles_m": 6, "tiles_n": 5}
        mx.set_tile_rows(256)
        assert mx.tile_config(8, 1408, 2048, 32768) == {"kn": 0, "tn": 256, "tiles_m": 6, "tiles_n": 8}
        mx.set_tile_orientation(2)
        mx.set_tile_rows(176)
        assert mx.tile_config(8, 1408, 2048, 32768) == {"kn": 1, "tn": 176, "tiles_m": 8, "tiles_n": 8}
        for bad in (3, -1):
            with pytest.raises(mx.Mxfp8Error):
                mx.set_tile_orientation(bad)
        for bad in (8, 24, 464, -16):
            with pytest.raises(mx.Mxfp8Error):
                mx.set_tile_rows(bad)
        with pytest.raises(mx.Mxfp8Error):
            mx.tile_config(4, 0, 8, 1024)
    finally:
        mx.set_tile_orientation(0)
        mx.set_tile_rows(0)


def test_tile_config_covers_output(lib):
    """Whatever the model picks, tn is a multiple of 16 in [16, 448] and the
    tiles cover both output axes."""
    import numpy as np
    rng = np.random.default_rng(5)
    try:
        for mode in (0, 1, 2):
            mx.set_tile_orientation(mode)
            for _ in range(40):
                N = int(rng.integers(1, 9000))
                K = 8 * int(rng.integers(1, 1200))
                E = int(rng.integers(1, 300))
                M = 32 * int(rng.integers(1, 20000))
                cfg = mx.tile_config(E, N, K, M)
                tn = cfg["tn"]
                assert tn % 16 == 0 and 16 <= tn <= 448
                if mode:
                    assert cfg["kn"] == mode - 1
                rows_m, rows_n = (K, N) if cfg["kn"] else (N, K)
                assert cfg["tiles_m"] == -(-rows_m // 256)
                assert cfg["tiles_n"] == -(-rows_n // tn)
    finally:
        mx.set_tile_orientation(0)


def test_workspace_covers_both_orientations(lib):
    """The workspace size is the larger of the two orientations' needs: the
    plan, then 2 scale blocks per 256-row tile and ceil(tn/128) per tn-row tile,
    each for the K-step bound ceil(M/128) + E."""
    E, N, K, M = 8, 1408, 2048, 196608
    ts = -(-M // 128) + E
    plan = -(-4 * (8 + 5 * E) // 1024) * 1024
    need = []
    try:
        for mode in (1, 2):
            mx.set_tile_orientation(mode)
            c = mx.tile_config(E, N, K, M)
            need.append(plan + (c["tiles_m"] * 2 + c["tiles_n"] * -(-c["tn"] // 128)) * ts * 512)
    finally:
        mx.set_tile_orientation(0)
    assert lib.mxfp8_wgrad_workspace_bytes(E, N, K, M) == max(need)


def test_quantize_transpose_validation(lib):
    q = lib.mxfp8_quantize_transpose_bf16
    q.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert q(P, 1024, 0, P, P, None) == _lib.EINVAL       # R < 1
    assert q(P, 1000, 64, P, P, None) == _lib.EINVAL      # M % 32 != 0
    assert q(None, 1024, 64, P, P, None) == _lib.EINVAL   # null x
    assert q(P + 1, 1024, 64, P, P, None) == _lib.EALIGN  # x not 2-byte aligned
    assert q(P, 1024, 64, P + 8, P, None) == _lib.EALIGN  # q not 16-byte aligned


def test_grouped_gemm_validation(lib):
    """Argument checks of the ragged-row grouped GEMM, all taken on the host
    before any device call."""
    f = lib.mxfp8_grouped_gemm
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_void_p, ctypes.c_void_p]
    ok = (P, P, P, P, P)
    assert f(*ok, 0, 1024, 256, 512, P, None) == _lib.EINVAL      # E < 1
    assert f(*ok, 2049, 1024, 256, 512, P, None) == _lib.EINVAL   # E above the maximum
    assert f(*ok, 4, 0, 256, 512, P, None) == _lib.EINVAL         # M < 1
    assert f(*ok, 4, 1 << 31, 256, 512, P, None) == _lib.EINVAL   # M above int32
    assert f(*ok, 4, 1024, 256, 500, P, None) == _lib.EINVAL      # K % 32 != 0
    assert f(*ok, 4, 1024, 0, 512, P, None) == _lib.EINVAL        # N < 1
    assert f(P, P, None, P, P, 4, 1024, 256, 512, P, None) == _lib.EINVAL  # null W
    assert f(P, P, P, P, P, 4, 1024, 256, 512, None, None) == _lib.EINVAL  # null out
    assert f(P + 8, P, P, P, P, 4, 1024, 256, 512, P, None) == _lib.EALIGN  # X not 16-byte aligned
    assert f(*ok, 4, 1024, 260, 512, P, None) == _lib.EALIGN      # N % 8 != 0 (output rows)
    assert f(*ok, 4, 1024, 256, 512, P + 2, None) == _lib.EALIGN  # out not 16-byte aligned


def test_grouped_gemm_tile_choice(lib):
    """Host-side tiling of the ragged-row grouped GEMM: the measured
    short-contraction cost (a per-tile hand-over plus a per-K-step part)
    decides the width; the row-tile bound is ceil(M/256) + E; a forced width
    is honoured; sizes the entry point rejects fail."""
    try:
        mx.set_tile_rows(0)
        # 16B forward (hidden 2048 -> 1408): 1408 = 4 x 352, no padding (two MMAs per chunk,
        # the drained row released before its stores)
        assert mx.grouped_gemm_tile_config(8, 1408, 2048, 32768) == {"tn": 352, "tiles_m_max": 136, "tiles_n": 4}
        # 16B data gradient (1408 -> 2048, 11 K-steps): 6 tiles of 352 (8 of 256 modelled 2% and
        # measured 0-3% apart)
        assert mx.grouped_gemm_tile_config(8, 2048, 1408, 32768) == {"tn": 352, "tiles_m_max": 136, "tiles_n": 6}
        # 671B up/gate forward (7168 -> 4096) and data gradient (4096 -> 7168)
        assert mx.grouped_gemm_tile_config(32, 4096, 7168, 262144)["tn"] == 256
        assert mx.grouped_gemm_tile_config(32, 7168, 4096, 262144)["tn"] == 448
        # 671B down forward (2048 -> 7168) and data gradient (7168 -> 2048)
        assert mx.grouped_gemm_tile_config(32, 7168, 2048, 524288) == {"tn": 448, "tiles_m_max": 2080, "tiles_n": 16}
        assert mx.grouped_gemm_tile_config(32, 2048, 7168, 524288)["tn"] == 256
        # narrow outputs: one column tile
        assert mx.grouped_gemm_tile_config(16, 64, 128, 900) == {"tn": 64, "tiles_m_max": 20, "tiles_n": 1}
        mx.set_tile_rows(224)
        assert mx.grouped_gemm_tile_config(8, 1408, 2048, 32768) == {"tn": 224, "tiles_m_max": 136, "tiles_n": 7}
        mx.set_tile_rows(0)
        for bad in ((0, 256, 512, 1024), (4, 260, 512, 1024), (4, 256, 500, 1024), (4, 256, 512, 0)):
            with pytest.raises(mx.Mxfp8Error):
                mx.grouped_gemm_tile_config(*bad)
    finally:
        mx.set_tile_rows(0)


def test_epilogue_store_setting(lib):
    """The epilogue store mode is a validated process-wide setting (host only)."""
    try:
        mx.set_epilogue_store(1)
        mx.set_epilogue_store(0)
        for bad in (-1, 2):
            with pytest.raises(mx.Mxfp8Error):
                mx.set_epilogue_store(bad)
    finally:
        mx.set_epilogue_store(0)


def test_sf_blocks_bytes(lib):
    """Size of the scale-factor blocks: tiles x 128-token grid steps x
    128-row blocks per tile x 512 bytes; 0 for sizes the layout rejects."""
    f = lib.mxfp8_sf_blocks_bytes
    f.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int]
    f.restype = ctypes.c_size_t
    assert f(2048, 32768, 256) == 8 * 256 * 2 * 512
    assert f(1408, 32768, 352) == 4 * 256 * 3 * 512
    assert f(7168, 524288, 416) == 18 * 4096 * 4 * 512
    assert f(100, 96, 16) == 7 * 1 * 1 * 512          # partial tile, partial step
    assert f(0, 1024, 256) == 0 and f(64, 1000, 256) == 0 and f(64, 1024, 17) == 0 and f(64, 1024, 0) == 0


def test_sf_entry_points_validation(lib):
    """Argument checks of the scale-factor-block path, taken on the host before
    any device call."""
    w = lib.mxfp8_wgrad_grouped_sf
    w.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    ok = (P, P, P, P, P)
    assert w(*ok, 4, 128, 256, 1024, 2, 256, P, None) == _lib.EINVAL      # kn not 0 or 1
    assert w(*ok, 4, 128, 256, 1024, 0, 17, P, None) == _lib.EINVAL       # tn not a multiple of 16
    assert w(*ok, 4, 128, 256, 1024, 0, 464, P, None) == _lib.EINVAL      # tn above 448
    assert w(P, P + 4, P, P, P, 4, 128, 256, 1024, 0, 256, P, None) == _lib.EALIGN  # sfA not 16-byte aligned
    assert w(P, None, P, P, P, 4, 128, 256, 1024, 0, 256, P, None) == _lib.EINVAL   # null sfA
    assert w(*ok, 4, 128, 256, 1000, 0, 256, P, None) == _lib.EINVAL     # M % 32 != 0
    assert w(None, None, None, None, None, 0, 128, 256, 1024, 0, 256, None, None) == _lib.OK  # E = 0: no-op
    q = lib.mxfp8_quantize_transpose_bf16_sf
    q.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 4
    assert q(P, 1024, 64, 0, P, None, P, None) == _lib.EINVAL     # tile_rows < 16
    assert q(P, 1024, 64, 24, P, None, P, None) == _lib.EINVAL    # tile_rows % 16 != 0
    assert q(P, 1024, 64, 256, P, None, None, None) == _lib.EINVAL  # null sf
    assert q(P, 1000, 64, 256, P, None, P, None) == _lib.EINVAL   # M % 32 != 0
    assert q(P, 1024, 64, 256, P + 8, None, P, None) == _lib.EALIGN  # q not 16-byte aligned
