"""GB300 (sm_103a) 4-bit quantized Mixture-of-Experts layer forward.

The compute path is the CUDA library libmoe_gb300.so (C ABI in include/moe_gb300.h); this
package is its thin Python binding. Build the library with
``quantized_grouped_gemm_router_gb300.build.build()``.
"""
from .binding import (  # noqa: F401
    ROUTE_FIELDS,
    Layer,
    MoeDims,
    MoeError,
    decode,
    decode_batch,
    decode_noalloc,
    decode_diag,
    DECODE_DIAG_NO_MATH,
    DECODE_DIAG_READ_ONLY,
    dims_of,
    lib,
    pack_weights,
    packed_bytes,
    prefill,
    prefill_ablation,
    prefill_diag,
    PREFILL_DIAG_READ_ONLY,
    PREFILL_ARM_HOST_ROUTING,
    PREFILL_ARM_TILE32,
    PREFILL_ARM_DENSE,
    PREFILL_ARM_WIDE_TILES,
    PREFILL_ARM_NARROW_TILES,
    ablation_aux_bytes,
    prefill_chunked,
    read_device_status,
    route,
    route_out_tensors,
    selftest_wait_timeout,
    status_string,
    tile_rows,
    prefill_tile_rows,
    upload_layer,
    workspace,
    workspace_bytes,
)
