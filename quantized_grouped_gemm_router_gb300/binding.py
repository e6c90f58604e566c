"""ctypes binding of libmoe_gb300.so (argument marshalling only; every step runs in the CUDA
library). PyTorch supplies device memory and the current stream.

The names follow the C ABI in include/moe_gb300.h: pack_weights, route, prefill, decode,
read_device_status, status_string, workspace_bytes, tile_rows.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

c_void_p, c_int32, c_size_t = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t


class MoeDims(ctypes.Structure):
    _fields_ = [(n, c_int32) for n in ("d", "n_experts", "top_k", "inter", "shared_inter", "group")]


class Q4View(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("scale", c_void_p), ("bias", c_void_p)]


class MoeLayer(ctypes.Structure):
    _fields_ = [("dims", MoeDims), ("router_w", c_void_p), ("router_bias", c_void_p), ("packed", c_void_p)]


ROUTE_FIELDS = ("logits", "topk_idx", "topk_w", "counts", "offsets", "perm", "inv_perm", "tile_map",
                "n_tiles", "hidden")


class RouteOut(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ROUTE_FIELDS]


STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE", 3: "MOE_ERR_MISALIGNED",
          4: "MOE_ERR_WORKSPACE_TOO_SMALL", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_NONFINITE",
          7: "MOE_ERR_DEVICE_TIMEOUT", 8: "MOE_ERR_OUT_OF_RANGE"}


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)} ({status_string(code)})")
        self.code = code


_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built (there is no fallback path)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libmoe_gb300.so is not built ({LIB_PATH}); run "
                              "quantized_grouped_gemm_router_gb300.build.build() first")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER
        L.moe_packed_bytes.argtypes = [P(MoeDims)]
        L.moe_packed_bytes.restype = c_size_t
        L.moe_pack_weights.argtypes = [P(MoeDims)] + [Q4View] * 6 + [c_void_p, c_void_p]
        L.moe_pack_weights.restype = ctypes.c_int
        L.moe_workspace_bytes.argtypes = [P(MoeDims), c_int32]
        L.moe_workspace_bytes.restype = c_size_t
        L.moe_workspace_init.argtypes = [c_void_p, c_size_t, c_void_p]
        L.moe_workspace_init.restype = ctypes.c_int
        L.moe_tile_rows.argtypes = []
        L.moe_tile_rows.restype = c_int32
        L.moe_prefill_tile_rows.argtypes = [P(MoeDims), c_int32]
        L.moe_prefill_tile_rows.restype = c_int32
        L.moe_route.argtypes = [P(MoeLayer), c_void_p, c_void_p, c_int32, P(RouteOut), c_void_p, c_size_t, c_void_p]
        L.moe_route.restype = ctypes.c_int
        L.moe_prefill.argtypes = [P(MoeLayer), c_void_p, c_int32, c_void_p, P(RouteOut), c_void_p, c_size_t,
                                  c_void_p]
        L.moe_prefill.restype = ctypes.c_int
        L.moe_prefill_chunked.argtypes = [P(MoeLayer), c_void_p, ctypes.c_int64, c_void_p, c_int32, c_void_p,
                                          c_size_t, c_void_p]
        L.moe_prefill_chunked.restype = ctypes.c_int
        L.moe_decode.argtypes = [P(MoeLayer), c_void_p, c_void_p, P(RouteOut), c_void_p, c_size_t, c_void_p]
        L.moe_decode.restype = ctypes.c_int
        L.moe_prefill_timed.argtypes = L.moe_prefill.argtypes + [ctypes.POINTER(c_void_p)]
        L.moe_prefill_timed.restype = ctypes.c_int
        L.moe_decode_timed.argtypes = L.moe_decode.argtypes + [ctypes.POINTER(c_void_p)]
        L.moe_decode_timed.restype = ctypes.c_int
        L.moe_decode_diag.argtypes = [P(MoeLayer), c_void_p, c_void_p, c_void_p, c_size_t, ctypes.c_int, c_void_p]
        L.moe_decode_diag.restype = ctypes.c_int
        L.moe_decode_batch.argtypes = [P(MoeLayer), c_void_p, c_int32, c_void_p, P(RouteOut), c_void_p, c_size_t,
                                       c_void_p]
        L.moe_decode_batch.restype = ctypes.c_int
        L.moe_prefill_ablation.argtypes = [P(MoeLayer), c_void_p, c_int32, c_void_p, ctypes.c_int, c_void_p, c_size_t,
                                           c_void_p, c_size_t, c_void_p]
        L.moe_prefill_ablation.restype = ctypes.c_int
        L.moe_prefill_diag.argtypes = [P(MoeLayer), c_void_p, c_int32, c_void_p, ctypes.c_int, c_void_p, c_size_t,
                                       c_void_p, ctypes.POINTER(c_void_p)]
        L.moe_prefill_diag.restype = ctypes.c_int
        L.moe_prefill_ablation_aux_bytes.argtypes = [P(MoeDims), ctypes.c_int]
        L.moe_prefill_ablation_aux_bytes.restype = c_size_t
        L.moe_decode_noalloc.argtypes = [P(MoeLayer), c_void_p, c_void_p, c_void_p]
        L.moe_decode_noalloc.restype = ctypes.c_int
        L.moe_read_device_status.argtypes = [c_void_p, c_void_p]
        L.moe_selftest_wait_timeout.argtypes = [c_void_p, c_size_t, c_void_p]
        L.moe_selftest_wait_timeout.restype = ctypes.c_int
        L.moe_read_device_status.restype = ctypes.c_int
        L.moe_status_string.argtypes = [ctypes.c_int]
        L.moe_status_string.restype = ctypes.c_char_p
        _LIB = L
    return _LIB


def status_string(code: int) -> str:
    return lib().moe_status_string(code).decode()


def _check(code: int, what: str) -> None:
    if code != 0:
        raise MoeError(code, what)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def dims_of(shape) -> MoeDims:
    return MoeDims(shape.d, shape.n_experts, shape.top_k, shape.inter, shape.shared_inter, shape.group)


def tile_rows() -> int:
    """The largest block-map tile height."""
    return int(lib().moe_tile_rows())


def prefill_tile_rows(dims: MoeDims, T: int) -> int:
    """Block-map tile height of a T-token route / prefill call (32 or tile_rows())."""
    return int(lib().moe_prefill_tile_rows(ctypes.byref(dims), int(T)))


def packed_bytes(dims: MoeDims) -> int:
    return int(lib().moe_packed_bytes(ctypes.byref(dims)))


def workspace_bytes(dims: MoeDims, max_tokens: int) -> int:
    return int(lib().moe_workspace_bytes(ctypes.byref(dims), max_tokens))


def workspace(dims: MoeDims, max_tokens: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace (zeroed counters and status, as the library requires)."""
    n = workspace_bytes(dims, max_tokens)
    if n == 0:
        raise MoeError(2, "workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _check_dev(t: torch.Tensor, dtype, name: str) -> None:
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor of {dtype}")


def pack_weights(dims: MoeDims, mats: dict) -> torch.Tensor:
    """mats: name -> (q int32, scale int16, bias int16) CUDA tensors in the canonical layout for
    gate, up, down, sh_gate, sh_up, sh_down. Returns the packed uint8 buffer."""
    views = []
    for name in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        q, s, b = mats[name]
        _check_dev(q, torch.int32, name + ".q")
        _check_dev(s, torch.int16, name + ".scale")
        _check_dev(b, torch.int16, name + ".bias")
        views.append(Q4View(q.data_ptr(), s.data_ptr(), b.data_ptr()))
    n = packed_bytes(dims)
    if n == 0:
        raise MoeError(2, "packed_bytes")
    packed = torch.empty(n, dtype=torch.uint8, device=mats["gate"][0].device)
    _check(lib().moe_pack_weights(ctypes.byref(dims), *views, packed.data_ptr(), _stream()), "moe_pack_weights")
    return packed


class Layer:
    """Device-resident layer: bf16 router weight (int16 bits), optional fp32 router bias, packed experts."""

    def __init__(self, dims: MoeDims, router_w: torch.Tensor, router_bias, packed: torch.Tensor):
        _check_dev(router_w, torch.int16, "router_w")
        if router_bias is not None:
            _check_dev(router_bias, torch.float32, "router_bias")
        self.dims, self.router_w, self.router_bias, self.packed = dims, router_w, router_bias, packed
        self._c = MoeLayer(dims, router_w.data_ptr(), _ptr(router_bias), packed.data_ptr())

    @property
    def c(self) -> MoeLayer:
        return self._c


def route_out_tensors(dims: MoeDims, T: int, device, want=ROUTE_FIELDS, hidden: bool = False) -> dict:
    """Allocates the requested routing outputs (see moe_route_out in include/moe_gb300.h)."""
    E, k, A = dims.n_experts, dims.top_k, T * dims.top_k
    max_tiles = min(E, A) + A // prefill_tile_rows(dims, T)
    shapes = {"logits": ((T, E), torch.float32), "topk_idx": ((T, k), torch.int32),
              "topk_w": ((T, k), torch.float32), "counts": ((E,), torch.int32),
              "offsets": ((E + 1,), torch.int32), "perm": ((A,), torch.int32), "inv_perm": ((A,), torch.int32),
              "tile_map": ((max_tiles, 3), torch.int32), "n_tiles": ((1,), torch.int32),
              "hidden": ((2, A + T, dims.inter), torch.int16)}
    out = {}
    for name in want:
        if name == "hidden" and not hidden:
            continue
        shape, dt = shapes[name]
        out[name] = torch.empty(shape, dtype=dt, device=device)
    return out


def _route_struct(out: dict | None):
    if out is None:
        return None
    return RouteOut(*[_ptr(out.get(n)) for n in ROUTE_FIELDS])


def route(layer: Layer, x, T: int, ws: torch.Tensor, logits_in=None, out: dict | None = None) -> dict:
    if x is not None:
        _check_dev(x, torch.int16, "x")
    if logits_in is not None:
        _check_dev(logits_in, torch.float32, "logits_in")
    out = out if out is not None else route_out_tensors(layer.dims, T, ws.device)
    ro = _route_struct(out)
    _check(lib().moe_route(ctypes.byref(layer.c), _ptr(x), _ptr(logits_in), T, ctypes.byref(ro), ws.data_ptr(),
                           ws.numel(), _stream()), "moe_route")
    return out


def _events(events, n: int):
    """Raw cudaEvent_t handles of torch.cuda.Event objects (None entries allowed)."""
    if events is None:
        return None
    assert len(events) == n
    return (c_void_p * n)(*[None if e is None else e.cuda_event for e in events])


def prefill(layer: Layer, x: torch.Tensor, ws: torch.Tensor, y: torch.Tensor | None = None,
            out: dict | None = None, events=None) -> torch.Tensor:
    """events: optional 6 torch.cuda.Event objects (already recorded once, so they exist) that
    the library records at its kernel boundaries (see moe_prefill_timed)."""
    _check_dev(x, torch.int16, "x")
    T = x.shape[0]
    y = y if y is not None else torch.empty_like(x)
    ro = _route_struct(out)
    args = (ctypes.byref(layer.c), x.data_ptr(), T, y.data_ptr(), ctypes.byref(ro) if ro is not None else None,
            ws.data_ptr(), ws.numel(), _stream())
    if events is None:
        _check(lib().moe_prefill(*args), "moe_prefill")
    else:
        _check(lib().moe_prefill_timed(*args, _events(events, 6)), "moe_prefill_timed")
    return y


PREFILL_ARM_HOST_ROUTING, PREFILL_ARM_TILE32, PREFILL_ARM_DENSE = 1, 2, 3
PREFILL_ARM_WIDE_TILES, PREFILL_ARM_NARROW_TILES = 4, 5
PREFILL_DIAG_READ_ONLY = 1


def prefill_diag(layer: Layer, x: torch.Tensor, ws: torch.Tensor, mode: int, y: torch.Tensor | None = None,
                 events=None) -> torch.Tensor:
    """moe_prefill_diag: moe_prefill with the two grouped GEMMs replaced by their read-only probes
    (mode 1; y becomes zeros). events: optional 6 events at the kernel boundaries, as for prefill."""
    _check_dev(x, torch.int16, "x")
    y = y if y is not None else torch.empty_like(x)
    _check_dev(y, torch.int16, "y")
    _check(lib().moe_prefill_diag(ctypes.byref(layer.c), x.data_ptr(), x.shape[0], y.data_ptr(), int(mode),
                                  ws.data_ptr(), ws.numel(), _stream(), _events(events, 6)), "moe_prefill_diag")
    return y


def ablation_aux_bytes(dims: MoeDims, arm: int) -> int:
    return int(lib().moe_prefill_ablation_aux_bytes(ctypes.byref(dims), int(arm)))


def prefill_ablation(layer: Layer, x: torch.Tensor, ws: torch.Tensor, arm: int,
                     y: torch.Tensor | None = None, aux: torch.Tensor | None = None) -> torch.Tensor:
    """moe_prefill_ablation: moe_prefill with the block map built on the host after a stream
    synchronisation (arm 1), with 32-row block-map tiles in the wide GEMM configuration (arm 2), on
    weights expanded to fp16 into `aux` first (arm 3; aux of ablation_aux_bytes(dims, 3) bytes), or
    with the wide (arm 4) or narrow (arm 5) GEMM configuration forced."""
    _check_dev(x, torch.int16, "x")
    y = y if y is not None else torch.empty_like(x)
    _check(lib().moe_prefill_ablation(ctypes.byref(layer.c), x.data_ptr(), x.shape[0], y.data_ptr(), int(arm),
                                      ws.data_ptr(), ws.numel(), _ptr(aux), 0 if aux is None else aux.numel(),
                                      _stream()), "moe_prefill_ablation")
    return y


def prefill_chunked(layer: Layer, x: torch.Tensor, ws: torch.Tensor, chunk_tokens: int,
                    y: torch.Tensor | None = None) -> torch.Tensor:
    """moe_prefill_chunked: prefill of all rows of x in chunks of at most chunk_tokens rows, with
    a workspace sized for one chunk."""
    _check_dev(x, torch.int16, "x")
    y = y if y is not None else torch.empty_like(x)
    _check(lib().moe_prefill_chunked(ctypes.byref(layer.c), x.data_ptr(), x.shape[0], y.data_ptr(), int(chunk_tokens),
                                     ws.data_ptr(), ws.numel(), _stream()), "moe_prefill_chunked")
    return y


def decode(layer: Layer, x: torch.Tensor, ws: torch.Tensor, y: torch.Tensor | None = None,
           out: dict | None = None, events=None) -> torch.Tensor:
    """events: optional 4 torch.cuda.Event objects (see moe_decode_timed)."""
    _check_dev(x, torch.int16, "x")
    y = y if y is not None else torch.empty_like(x)
    ro = _route_struct(out)
    args = (ctypes.byref(layer.c), x.data_ptr(), y.data_ptr(), ctypes.byref(ro) if ro is not None else None,
            ws.data_ptr(), ws.numel(), _stream())
    if events is None:
        _check(lib().moe_decode(*args), "moe_decode")
    else:
        _check(lib().moe_decode_timed(*args, _events(events, 4)), "moe_decode_timed")
    return y


def decode_batch(layer: Layer, x: torch.Tensor, ws: torch.Tensor, y: torch.Tensor | None = None,
                 out: dict | None = None) -> torch.Tensor:
    """moe_decode_batch: decode of the T = x.shape[0] <= 8 token rows of x at once."""
    _check_dev(x, torch.int16, "x")
    y = y if y is not None else torch.empty_like(x)
    ro = _route_struct(out)
    _check(lib().moe_decode_batch(ctypes.byref(layer.c), x.data_ptr(), x.shape[0], y.data_ptr(),
                                  ctypes.byref(ro) if ro is not None else None, ws.data_ptr(), ws.numel(),
                                  _stream()), "moe_decode_batch")
    return y


DECODE_DIAG_NO_MATH, DECODE_DIAG_READ_ONLY = 1, 2


def decode_diag(layer: Layer, x: torch.Tensor, ws: torch.Tensor, mode: int, y: torch.Tensor | None = None) -> torch.Tensor:
    """moe_decode_diag: the decode chain with the GEMV arithmetic deleted (mode 1) or the expert
    kernel's weight copies alone (mode 2)."""
    _check_dev(x, torch.int16, "x")
    y = y if y is not None else torch.empty_like(x)
    _check(lib().moe_decode_diag(ctypes.byref(layer.c), x.data_ptr(), y.data_ptr(), ws.data_ptr(), ws.numel(),
                                 int(mode), _stream()), "moe_decode_diag")
    return y


def decode_noalloc(layer: Layer, x: torch.Tensor, y: torch.Tensor) -> torch.Tensor:
    """Batch-1 decode through moe_decode_noalloc: no workspace, the library allocates nothing."""
    _check_dev(x, torch.int16, "x")
    _check_dev(y, torch.int16, "y")
    _check(lib().moe_decode_noalloc(ctypes.byref(layer.c), x.data_ptr(), y.data_ptr(), _stream()),
           "moe_decode_noalloc")
    return y


def selftest_wait_timeout(ws: torch.Tensor) -> None:
    """moe_selftest_wait_timeout: a bounded device wait that is never satisfied gives up (about a
    second) and records MOE_ERR_DEVICE_TIMEOUT in ws; read it with read_device_status."""
    _check(lib().moe_selftest_wait_timeout(ws.data_ptr(), ws.numel(), _stream()), "moe_selftest_wait_timeout")


def read_device_status(ws: torch.Tensor) -> int:
    return int(lib().moe_read_device_status(ws.data_ptr(), _stream()))


def upload_layer(np_layer: dict, device="cuda") -> Layer:
    """Copies a canonical numpy layer (see synthetic.moe_inputs) to the device and packs it."""
    import numpy as np

    def dev(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a).view(dt)).to(device)

    dims = dims_of(np_layer["shape"])
    mats = {n: (dev(np_layer[n]["q"], np.int32), dev(np_layer[n]["scale"], np.int16),
                dev(np_layer[n]["bias"], np.int16)) for n in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down")}
    packed = pack_weights(dims, mats)
    rb = np_layer.get("router_bias")
    layer = Layer(dims, dev(np_layer["router_w"], np.int16), None if rb is None else dev(rb, np.float32), packed)
    torch.cuda.current_stream().synchronize()  # canonical copies are released on return
    return layer
