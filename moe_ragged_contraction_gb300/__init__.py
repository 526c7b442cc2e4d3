"""GB300-native ragged MXFP8 MoE weight-gradient grouped GEMM.

dW[g] = dY[g]^T X[g] for every expert g, where per-expert token offsets cut
the contraction axis ("Ragged MXFP8 Weight Gradients: A FlyDSL Grouped GEMM on
MI355X", section 1), computed by hand-written sm_103a CUDA kernels (TMA,
tcgen05 block-scaled MMA, TMEM) behind the C ABI in ``include/mxfp8_wgrad.h``.

The Python API below is a thin ctypes binding: argument marshalling only.
"""
from ._lib import (  # noqa: F401
    Mxfp8Error,
    device_status,
    grouped_gemm,
    grouped_gemm_tile_config,
    lib_path,
    load,
    quantize_tokenwise,
    quantize_transpose_bf16,
    quantize_transpose_bf16_sf,
    set_epilogue_store,
    set_tile_orientation,
    set_tile_rows,
    set_timing_events,
    sf_blocks_bytes,
    tile_config,
    wgrad_grouped,
    wgrad_grouped_sf,
    workspace_bytes,
)
from .build import build  # noqa: F401
