"""Host-side checks of the C ABI (CPU only): the library loads, exports every symbol the header
declares, answers the host-only queries, and rejects bad arguments before launching anything.
Every call below fails argument validation, so no CUDA work is attempted."""
import ctypes
import os
import re

import pytest

from quantized_grouped_gemm_router_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe_gb300.h")


@pytest.fixture(scope="module")
def m():
    B.build()
    import quantized_grouped_gemm_router_gb300 as mod
    return mod


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)


def test_exports_every_declared_symbol(m):
    names = declared_functions()
    assert len(names) >= 10
    lib = m.lib()
    for n in names:
        assert hasattr(lib, n), n


def test_host_queries(m):
    from synthetic import FULL, TINY
    full = m.dims_of(FULL)
    R = m.tile_rows()
    assert R == 192
    # block-map tile height by token count: 32-row tiles while T * k <= 24 * E
    assert m.prefill_tile_rows(full, 1) == 32 and m.prefill_tile_rows(full, 768) == 32
    assert m.prefill_tile_rows(full, 769) == R and m.prefill_tile_rows(full, 4096) == R
    tiny = m.dims_of(TINY)
    lim = 24 * tiny.n_experts // tiny.top_k
    assert m.prefill_tile_rows(tiny, lim) == 32 and m.prefill_tile_rows(tiny, lim + 1) == R
    assert m.prefill_tile_rows(full, 0) == 0
    assert m.packed_bytes(full) == 257 * 1769472          # (E + 1) experts x 3*I*d*(1/2 + 4/64) bytes
    assert m.packed_bytes(m.dims_of(TINY)) == 17 * 3 * 128 * 256 * 9 // 16
    assert m.workspace_bytes(full, 1) > 0
    assert m.workspace_bytes(full, 4096) > m.workspace_bytes(full, 2048)
    assert m.workspace_bytes(full, 0) == 0 and m.workspace_bytes(full, 65537) == 0
    for bad in (dict(group=32), dict(d=2000), dict(inter=500), dict(shared_inter=256), dict(top_k=0),
                dict(top_k=17), dict(n_experts=4, top_k=8), dict(n_experts=2048)):
        dims = m.dims_of(FULL)
        for k, v in bad.items():
            setattr(dims, k, v)
        assert m.packed_bytes(dims) == 0 and m.workspace_bytes(dims, 16) == 0, bad
        assert m.prefill_tile_rows(dims, 16) == 0, bad
    for code in range(8):
        assert m.status_string(code) and m.status_string(code) != "unknown status"


def test_argument_errors_before_launch(m):
    from quantized_grouped_gemm_router_gb300.binding import MoeLayer, RouteOut
    from synthetic import FULL
    lib = m.lib()
    dims = m.dims_of(FULL)
    A = 1 << 20  # fake, never dereferenced: every call below fails validation first
    layer = MoeLayer(dims, A, None, A)
    ws_need = m.workspace_bytes(dims, 16)
    call = lambda L, x, T, y, ws, n: lib.moe_prefill(ctypes.byref(L), x, T, y, None, ws, n, None)  # noqa: E731
    assert call(layer, None, 16, A, A, ws_need) == 1                      # null x
    assert call(layer, A, 0, A, A, ws_need) == 1                          # T < 1
    assert call(layer, A, 70000, A, A, ws_need) == 2                      # T too large
    assert call(layer, A + 8, 16, A, A, ws_need) == 3                     # misaligned x
    assert call(layer, A, 16, A, A + 64, ws_need) == 3                    # ws not 128-aligned
    assert call(layer, A, 16, A, A, ws_need - 1) == 4                     # workspace too small
    bad = MoeLayer(m.dims_of(FULL), A, None, A + 16)
    assert call(bad, A, 16, A, A, ws_need) == 3                           # packed not 128-aligned
    bad.dims.group = 128
    assert call(bad, A, 16, A, A, ws_need) == 2
    out = RouteOut(*([A + 4] + [None] * 9))
    assert lib.moe_route(ctypes.byref(layer), A, None, 16, ctypes.byref(out), A, ws_need, None) == 3
    assert lib.moe_route(ctypes.byref(layer), None, None, 16, None, A, ws_need, None) == 1
    assert lib.moe_decode(ctypes.byref(layer), A, None, None, A, ws_need, None) == 1
    assert lib.moe_decode(ctypes.byref(layer), A, A, None, A, 16, None) == 4
    assert lib.moe_decode_diag(ctypes.byref(layer), A, A, A, ws_need, 3, None) == 1  # unknown mode
    assert lib.moe_decode_diag(ctypes.byref(layer), A, A, A, 16, 1, None) == 4      # workspace too small
    chunked = lambda x, T, y, chunk, n: lib.moe_prefill_chunked(ctypes.byref(layer), x, T, y, chunk, A, n, None)  # noqa: E731
    assert chunked(A, 0, A, 16, ws_need) == 1                             # T < 1
    assert chunked(A, 100000, A, 0, ws_need) == 1                         # chunk < 1
    assert chunked(None, 100000, A, 16, ws_need) == 1                     # null x
    assert chunked(A, 100000, A, 70000, ws_need) == 2                     # chunk above the single-call limit
    assert chunked(A, 100000, A + 2, 16, ws_need) == 3                    # misaligned y
    assert chunked(A, 100000, A, 32, ws_need) == 4                        # workspace smaller than one chunk
    assert chunked(A, 100000, A, 16, ws_need - 1) == 4
    assert lib.moe_selftest_wait_timeout(None, 256, None) == 1
    assert lib.moe_selftest_wait_timeout(A, 16, None) == 1                # smaller than the status header
    assert lib.moe_selftest_wait_timeout(A + 64, 256, None) == 3
    assert lib.moe_workspace_init(None, 256, None) == 1
    assert lib.moe_read_device_status(None, None) == 1
    abl = lambda x, T, arm, n, aux=None, na=0: lib.moe_prefill_ablation(  # noqa: E731
        ctypes.byref(layer), x, T, A, arm, A, n, aux, na, None)
    assert abl(A, 16, 0, ws_need) == 1                                    # unknown arm
    assert abl(A, 16, 6, ws_need) == 1
    diag = lambda T, mode, n: lib.moe_prefill_diag(ctypes.byref(layer), A, T, A, mode, A, n, None, None)  # noqa: E731
    assert diag(16, 2, ws_need) == 1                                      # unknown mode
    assert diag(16, 1, ws_need - 1) == 4                                  # workspace too small
    assert diag(0, 1, ws_need) == 1
    assert abl(A, 16, 3, ws_need) == 1                                    # dense arm without its buffer
    aux_need = lib.moe_prefill_ablation_aux_bytes(ctypes.byref(dims), 3)
    assert aux_need == 257 * 3 * 512 * 2048 * 2                           # every expert's weights in fp16
    assert lib.moe_prefill_ablation_aux_bytes(ctypes.byref(dims), 1) == 0
    assert abl(A, 16, 3, ws_need, A + 64, aux_need) == 3                  # aux not 128-aligned
    assert abl(A, 16, 3, ws_need, A, aux_need - 1) == 4
    assert abl(None, 16, 1, ws_need) == 1                                 # null x
    assert abl(A, 16, 2, ws_need - 1) == 4                                # workspace too small
    assert abl(A, 70000, 1, ws_need) == 2


def test_workspace_grows_with_tokens(m):
    """moe_prefill_chunked checks the workspace against its first (largest) chunk only: that is
    sound because a workspace for T tokens also serves every smaller T. Pinned over every T up to
    4096 and a spread of larger T, for the full and tiny shapes."""
    from synthetic import FULL, TINY
    for shape in (FULL, TINY):
        dims = m.dims_of(shape)
        ts = list(range(1, 4097)) + [5000, 8191, 8192, 16384, 32768, 65535, 65536]
        sizes = [m.workspace_bytes(dims, t) for t in ts]
        assert all(b > 0 for b in sizes)
        assert all(a <= b for a, b in zip(sizes, sizes[1:])), shape
