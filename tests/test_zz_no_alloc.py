"""The allocation-free decode entry point (moe_decode_noalloc) against the regular one.

moe_decode_noalloc serves callers that cannot allocate device memory (a host application that
owns all device memory and lends only input/output buffers, or code that must not allocate
after start-up). Called through the C ABI, it runs the same deterministic kernels as moe_decode
(fixed summation order), so on the same inputs it must return the same bits, on two calls in a
row (the second call reuses the library's fixed scratch array left over from the first); each
result is also checked against the oracle within the output tolerance the other tests use. This
file is collected last and passes both alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O  # noqa: E402
from synthetic import FULL, TINY, make_layer, make_tokens  # noqa: E402
from tests import moe_check as C  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    from quantized_grouped_gemm_router_gb300 import build as B
    B.build()
    import quantized_grouped_gemm_router_gb300 as mod
    assert torch.cuda.is_available()
    return mod


@pytest.mark.parametrize("shape,seed", [(FULL, 7), (TINY, 8)], ids=["full", "tiny"])
def test_decode_noalloc_matches_decode(m, shape, seed):
    npl = make_layer(shape, seed=seed)
    layer = m.upload_layer(npl)
    ws = m.workspace(layer.dims, 1)
    lib = m.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):                       # two calls in a row share the static scratch
        xn = make_tokens(1, shape.d, seed=seed, stream=call + 1)
        x = torch.from_numpy(xn.view(np.int16)).cuda()
        y_ref = m.decode(layer, x, ws)
        y = torch.full_like(x, 0x7FC0)            # NaN fill: every element must be written
        rc = lib.moe_decode_noalloc(ctypes.byref(layer.c), ctypes.c_void_p(x.data_ptr()),
                                    ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(stream))
        assert rc == 0, m.status_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref), f"call {call}: output bits differ from moe_decode"
        C.check_y(C.bf16_bits_f64(y), O.moe_forward(xn, npl, tile_rows=m.tile_rows())["y"], f"call {call}")
    assert m.read_device_status(ws) == 0


def test_decode_noalloc_rejects_oversized_shape(m):
    from quantized_grouped_gemm_router_gb300.binding import MoeLayer
    dims = m.dims_of(FULL)
    dims.inter = 16384         # 144 (k+1) I / 32 bytes of SwiGLU records exceed the fixed scratch
    dims.shared_inter = 16384
    A = 1 << 20                # never dereferenced: the shape check fails first
    layer = MoeLayer(dims, A, None, A)
    assert m.lib().moe_decode_noalloc(ctypes.byref(layer), A, A, None) == 2
