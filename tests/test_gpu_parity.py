"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on a GB300.

Routing integers are compared bit for bit on identical logits; logits, weights, hidden rows
and outputs within the tolerances stated in tests/moe_check.py.
"""
import functools

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O  # noqa: E402
from synthetic import CONFIGS, FULL, TINY, LayerShape, make_layer, make_tokens  # noqa: E402
from tests import moe_check as C  # noqa: E402

pytestmark = pytest.mark.gpu

# Shapes that take the general top-k paths (more than 8 experts per token, more than 256 experts).
MID = LayerShape(d=256, n_experts=300, top_k=9, inter=128, shared_inter=128)
WIDE = LayerShape(d=256, n_experts=1024, top_k=16, inter=128, shared_inter=128)
# Shapes that take the decode down kernel's other work splits: 32 parts of 32 intermediate rows
# (two chunks of 16 parts), 12 parts (six 64-column groups per chunk), and the widest decode
# (d = 3072, 192 down blocks) with 20 parts (a last chunk of 4 parts whose copies run past the
# end of the weights and read zeros there).
LONGI = LayerShape(d=256, n_experts=16, top_k=2, inter=1024, shared_inter=1024)
ODDI = LayerShape(d=384, n_experts=16, top_k=4, inter=384, shared_inter=384)
BIGD = LayerShape(d=3072, n_experts=32, top_k=8, inter=640, shared_inter=640)


@pytest.fixture(scope="module")
def m():
    from quantized_grouped_gemm_router_gb300 import build as B
    B.build()
    import quantized_grouped_gemm_router_gb300 as mod
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return mod


@functools.lru_cache(maxsize=8)
def _np_layer(shape, seed, bias):
    return make_layer(shape, seed, bias)


_DEV_LAYERS = {}


def dev_layer(m, shape, seed=0, bias=None):
    key = (shape, seed, bias)
    if key not in _DEV_LAYERS:
        _DEV_LAYERS[key] = m.upload_layer(_np_layer(shape, seed, bias))
    return _DEV_LAYERS[key]


def to_dev(a):
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_route(m, layer, T, logits=None, x=None):
    ws = m.workspace(layer.dims, T)
    out = m.route(layer, None if x is None else to_dev(x), T, ws,
                  logits_in=None if logits is None else to_dev(logits))
    torch.cuda.synchronize()
    assert m.read_device_status(ws) == 0
    return C.to_np(out)


# ------------------------------------------------------------------------------ routing
def crafted_logits(T, E, kind, seed=0):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return rng.standard_normal((T, E)).astype(np.float32)
    if kind == "ties":
        l = (np.round(rng.standard_normal((T, E)) * 2) / 2).astype(np.float32)
        l[0::7] = 0.25                       # all-equal rows -> experts 0..k-1
        l[3::7] = -0.0
        l[3::7, 5::9] = 0.0                  # -0.0 and +0.0 tie
        return l
    if kind == "skew":
        l = rng.standard_normal((T, E)).astype(np.float32)
        l[:, :8] += 50.0                     # every token picks experts 0..7
        return l
    raise ValueError(kind)


@pytest.mark.parametrize("shape", [TINY, FULL], ids=["tiny", "full"])
@pytest.mark.parametrize("T,kind", [(1, "normal"), (64, "ties"), (65, "normal"), (300, "ties"),
                                    (300, "skew"), (2048, "normal"), (2048, "skew"), (517, "ties")])
def test_route_given_logits_bit_exact(m, shape, T, kind):
    layer = dev_layer(m, shape)
    logits = crafted_logits(T, shape.n_experts, kind, seed=T)
    gpu = run_route(m, layer, T, logits=logits)
    np.testing.assert_array_equal(gpu["logits"], logits)
    C.check_routing_exact(gpu, logits, shape.n_experts, shape.top_k, m.prefill_tile_rows(layer.dims, T))


@pytest.mark.parametrize("shape", [MID, WIDE], ids=["E300k9", "E1024k16"])
@pytest.mark.parametrize("T,kind", [(1, "normal"), (65, "ties"), (300, "normal"), (300, "skew")])
def test_route_wide_shapes_bit_exact(m, shape, T, kind):
    """top_k up to 16 and up to 1024 experts (the general warp top-k paths)."""
    test_route_given_logits_bit_exact(m, shape, T, kind)


@pytest.mark.parametrize("name", ["tiny", "prefill512", "skew2048"])
def test_route_router_gemm(m, name):
    shape, T, bias = CONFIGS[name]
    npl = _np_layer(shape, 0, bias)
    layer = dev_layer(m, shape, 0, bias)
    x = make_tokens(T, shape.d, seed=1)
    gpu = run_route(m, layer, T, x=x)
    ref_logits = O.router_logits(x, npl["router_w"], npl["router_bias"])
    tol = C.logit_tolerance(x, npl["router_w"]) + 1e-6 * np.abs(ref_logits)
    assert np.all(np.abs(gpu["logits"].astype(np.float64) - ref_logits) <= tol)
    C.check_routing_exact(gpu, gpu["logits"], shape.n_experts, shape.top_k, m.prefill_tile_rows(layer.dims, T))
    diff, ok = C.selection_with_near_ties(gpu["logits"], ref_logits, tol, shape.top_k)
    assert ok, f"tokens {diff} select different experts without a near tie"


def test_route_nonfinite_sets_status(m):
    layer = dev_layer(m, TINY)
    logits = crafted_logits(8, TINY.n_experts, "normal")
    logits[3, 2] = np.nan
    ws = m.workspace(layer.dims, 8)
    m.route(layer, None, 8, ws, logits_in=to_dev(logits))
    assert m.read_device_status(ws) == 6
    assert m.read_device_status(ws) == 0      # sticky until read, then cleared
    m.route(layer, None, 8, ws, logits_in=to_dev(crafted_logits(8, TINY.n_experts, "normal")))
    assert m.read_device_status(ws) == 0


# ------------------------------------------------------------------------------ packing
def _unpermute_nibbles(w):
    """Packed word -> canonical word: canonical column j sits in nibble slot j // 2 + 4 (j % 2)."""
    w = w.astype(np.uint32)
    out = np.zeros_like(w)
    for j in range(8):
        slot = j // 2 + 4 * (j % 2)
        out |= ((w >> np.uint32(4 * slot)) & np.uint32(15)) << np.uint32(4 * j)
    return out


def _unpack_expert(pe, d, inter):
    """One expert's packed bytes -> canonical (q, scale, bias) of gate, up and down, read back by
    the layout moe_pack_weights documents: gate|up as 128-row x 64-column blocks (block m, quarter
    q of 32 rows, K block kb at ((4 m + q) KB + kb) x 2304 bytes: gate then up, each [column half]
    [32 rows][16 bytes of codes], then 32 (scale, bias) words); down as [K block][column half]
    [128-row block][128 rows][16 bytes] of codes, then [K block][128-row block][128 rows] words."""
    KB, KBI, M, DM = d // 64, inter // 64, inter // 128, d // 128
    gu_bytes = M * KB * 2 * 4608
    gu = pe[:gu_bytes].reshape(M, 4, KB, 2, 1152)
    mats = {}
    for mi, name in enumerate(("gate", "up")):
        blk = gu[:, :, :, mi, :]
        codes = np.ascontiguousarray(blk[..., :1024]).view("<u4").reshape(M, 4, KB, 2, 32, 4)
        words = codes.transpose(0, 1, 4, 2, 3, 5).reshape(inter, KB * 8)      # row, (kb, half, word)
        sb = np.ascontiguousarray(blk[..., 1024:]).view("<u4").reshape(M, 4, KB, 32)
        sb = sb.transpose(0, 1, 3, 2).reshape(inter, KB)
        mats[name] = (_unpermute_nibbles(words), (sb & 0xFFFF).astype(np.uint16), (sb >> 16).astype(np.uint16))
    dn = pe[gu_bytes:]
    n_codes = KBI * 2 * DM * 2048
    codes = np.ascontiguousarray(dn[:n_codes]).view("<u4").reshape(KBI, 2, DM, 128, 4)
    words = codes.transpose(2, 3, 0, 1, 4).reshape(d, KBI * 8)
    sb = np.ascontiguousarray(dn[n_codes:]).view("<u4").reshape(KBI, DM, 128).transpose(1, 2, 0).reshape(d, KBI)
    mats["down"] = (_unpermute_nibbles(words), (sb & 0xFFFF).astype(np.uint16), (sb >> 16).astype(np.uint16))
    return mats


@pytest.mark.parametrize("shape", [TINY, FULL], ids=["tiny", "full"])
def test_pack_layout_exact(m, shape):
    """moe_pack_weights writes exactly the documented layout: reading every expert's codes,
    scales and biases back from the packed bytes (a numpy reading of the layout, independent of
    the kernels that consume it) gives the canonical inputs bit for bit; packing twice gives the
    same bytes."""
    npl = _np_layer(shape, 0, None)
    names = ("gate", "up", "down", "sh_gate", "sh_up", "sh_down")
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a).view(dt)).cuda()  # noqa: E731
    mats = {n: (dev(npl[n]["q"], np.int32), dev(npl[n]["scale"], np.int16), dev(npl[n]["bias"], np.int16))
            for n in names}
    dims = m.dims_of(shape)
    a = m.pack_weights(dims, mats)
    b = m.pack_weights(dims, mats)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    pa = a.cpu().numpy()
    assert pa.size == m.packed_bytes(dims)
    E, d, inter = shape.n_experts, shape.d, shape.inter
    stride = pa.size // (E + 1)
    for e in range(E + 1):
        got = _unpack_expert(pa[e * stride:(e + 1) * stride], d, inter)
        for name in ("gate", "up", "down"):
            src = npl[name if e < E else "sh_" + name]
            q = np.asarray(src["q"]).view(np.uint32)
            sc, bi = np.asarray(src["scale"]).view(np.uint16), np.asarray(src["bias"]).view(np.uint16)
            if e < E:
                q, sc, bi = q[e], sc[e], bi[e]
            np.testing.assert_array_equal(got[name][0], q.reshape(got[name][0].shape), f"expert {e} {name} codes")
            np.testing.assert_array_equal(got[name][1], sc.reshape(got[name][1].shape), f"expert {e} {name} scales")
            np.testing.assert_array_equal(got[name][2], bi.reshape(got[name][2].shape), f"expert {e} {name} biases")


# ------------------------------------------------------------------------------ prefill
def prefill_and_check(m, shape, T, seed=0, bias=None, npl=None, layer=None, hidden=False):
    npl = npl if npl is not None else _np_layer(shape, seed, bias)
    layer = layer if layer is not None else dev_layer(m, shape, seed, bias)
    x = make_tokens(T, shape.d, seed=seed + 100)
    ws = m.workspace(layer.dims, T)
    out = m.route_out_tensors(layer.dims, T, "cuda", hidden=hidden)
    y = m.prefill(layer, to_dev(x), ws, out=out)
    torch.cuda.synchronize()
    assert m.read_device_status(ws) == 0
    g = C.to_np(out)
    R = m.prefill_tile_rows(layer.dims, T)
    C.check_routing_exact(g, g["logits"], shape.n_experts, shape.top_k, R)
    ref_logits = O.router_logits(x, npl["router_w"], npl["router_bias"])
    tol = C.logit_tolerance(x, npl["router_w"]) + 1e-6 * np.abs(ref_logits)
    diff, ok = C.selection_with_near_ties(g["logits"], ref_logits, tol, shape.top_k)
    assert ok, f"tokens {diff} select different experts without a near tie"
    routing = None
    if diff:  # follow the GPU's selection, weights from the oracle's own logits
        idx = g["topk_idx"]
        sel = np.take_along_axis(ref_logits.astype(np.float64), idx.astype(np.int64), axis=1)
        w = np.exp(sel - sel.max(1, keepdims=True))
        routing = (idx, w / w.sum(1, keepdims=True))
    ref = O.moe_forward(x, npl, tile_rows=R, routing=routing)
    stats = C.check_y(y, ref["y"])
    print(f"prefill T={T}: {stats}")
    if hidden:
        H = O.hidden_sorted(x, npl, ref["grouping"])
        planes = out["hidden"].cpu().numpy().view(np.float16).astype(np.float64)
        C.check_y(planes[0] + planes[1], H, "hidden")
    return stats, g


@pytest.mark.parametrize("T", [1, 4, 37, 300])
def test_prefill_tiny_shape(m, T):
    prefill_and_check(m, TINY, T, hidden=True)


@pytest.mark.parametrize("shape,T", [(LONGI, 37), (ODDI, 37)], ids=["I1024", "d384I384"])
def test_prefill_other_widths(m, shape, T):
    prefill_and_check(m, shape, T, hidden=True)


def test_prefill_config_tiny(m):
    shape, T, _ = CONFIGS["tiny"]
    prefill_and_check(m, shape, T)


def test_prefill_full_512(m):
    shape, T, bias = CONFIGS["prefill512"]
    prefill_and_check(m, shape, T, bias=bias)


def test_prefill_full_skew_2048(m):
    shape, T, bias = CONFIGS["skew2048"]
    _, g = prefill_and_check(m, shape, T, bias=bias, hidden=True)
    assert g["counts"].max() > 256   # several tiles for the heaviest experts


def test_prefill_forced_tile_edges(m):
    """Every token picks experts 0..k-1: each gets T rows (whole tiles, then a ragged tail), in
    the narrow configuration (384 and 385 tokens: 12 tiles of 32 rows, then one of 1) and in the
    wide one (960 and 961 tokens: 5 tiles of 192 rows, then one of 1)."""
    shape = FULL
    npl = dict(_np_layer(shape, 3, None))
    rb = np.zeros(shape.n_experts, dtype=np.float32)
    rb[: shape.top_k] = 100.0
    npl["router_bias"] = rb
    layer = m.upload_layer(npl)
    for T, R in ((384, 32), (385, 32), (960, m.tile_rows()), (961, m.tile_rows())):
        assert m.prefill_tile_rows(layer.dims, T) == R
        _, g = prefill_and_check(m, shape, T, seed=3, npl=npl, layer=layer)
        assert np.all(g["counts"][: shape.top_k] == T)
        assert int(g["n_tiles"][0]) == shape.top_k * -(-T // R)


def integer_layer(shape, seed, force_top=False):
    """Every weight of every expert is scale 1, bias -8, so w = q - 8 is an integer in -8..7
    (the packed codes stay random); optionally a router bias that sends every token to experts
    0..k-1."""
    npl = dict(_np_layer(shape, seed, None))
    for mat in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        q = dict(npl[mat])
        q["scale"] = np.full_like(q["scale"], 0x3F80)  # bf16 1.0
        q["bias"] = np.full_like(q["bias"], 0xC100)    # bf16 -8.0
        npl[mat] = q
    if force_top:
        rb = np.zeros(shape.n_experts, dtype=np.float32)
        rb[: shape.top_k] = 100.0
        npl["router_bias"] = rb
    return npl


def sparse_sign_tokens(T, d, nnz, seed):
    """x = +-1 on nnz random features of each row, 0 elsewhere (bf16 bits): with w in -8..7,
    |g|, |u| <= 8 nnz, far below 2^24, so every partial sum is an exact integer in fp32."""
    rng = np.random.default_rng(seed)
    x = np.zeros((T, d), dtype=np.float32)
    for t in range(T):
        cols = rng.choice(d, nnz, replace=False)
        x[t, cols] = rng.choice(np.array([-1.0, 1.0], dtype=np.float32), nnz)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("T,force_top", [(800, False), (784, True), (300, False), (400, True)],
                         ids=["wide_cfg_short_tiles", "wide_cfg_192", "narrow_cfg", "narrow_cfg_forced"])
def test_prefill_integer_weights_exact_hidden(m, T, force_top):
    """Integer-valued case of the expert GEMMs: g and u are exact integers on both sides whatever
    the order of the K sums (tiles of at most half an accumulator buffer split K over the two MMA
    issuers, taller tiles split rows). Wide configuration: 800 tokens give ~25 rows per expert;
    784 tokens forced onto experts 0..k-1 give tiles of 192 rows and a ragged 16. Narrow
    configuration (32-row tiles): 300 tokens (~9 rows per expert), and 400 tokens forced onto
    experts 0..k-1 (12 tiles of 32 and a ragged 16). The SwiGLU rows must then equal the oracle's
    up to the rounding of silu and of the fp16 pair: 1e-5 relative + 1e-7 absolute, where one unit
    of error in g or u moves h by at least ~1/|g| > 1e-3 relative."""
    shape = FULL
    npl = integer_layer(shape, 21, force_top)
    layer = m.upload_layer(npl)
    x = sparse_sign_tokens(T, shape.d, 32, seed=T)
    ws = m.workspace(layer.dims, T)
    out = m.route_out_tensors(layer.dims, T, "cuda", hidden=True)
    m.prefill(layer, to_dev(x), ws, out=out)
    torch.cuda.synchronize()
    assert m.read_device_status(ws) == 0
    g = C.to_np({k: v for k, v in out.items() if k != "hidden"})
    R = m.prefill_tile_rows(layer.dims, T)
    assert R == (32 if T * shape.top_k <= 24 * shape.n_experts else m.tile_rows())
    C.check_routing_exact(g, g["logits"], shape.n_experts, shape.top_k, R)
    if force_top:
        assert np.all(g["counts"][: shape.top_k] == T)
    grouping = O.group_assignments(g["topk_idx"], shape.n_experts, R)
    H = O.hidden_sorted(x, npl, grouping)
    planes = out["hidden"].cpu().numpy().view(np.float16).astype(np.float64)
    err = np.abs(planes[0] + planes[1] - H)
    worst = float(np.max(err / (1e-5 * np.abs(H) + 1e-7)))
    assert worst <= 1.0, f"hidden rows off by {worst:.2f} x tolerance"


def mixed_scale_layer(shape, seed):
    """The synthetic layer with a quarter of the (row, group) scales of every matrix raised to
    0.0625..0.25 (bias -8 * scale, exact in bf16): scales the narrow configuration's subnormal
    dequantization (|scale| < 2^-4) cannot take, mixed with ones it can inside the same warps."""
    npl = dict(_np_layer(shape, seed, None))
    rng = np.random.default_rng(seed + 1)
    for mat in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        q = dict(npl[mat])
        sc = np.asarray(q["scale"]).view(np.uint16).copy()
        pick = rng.random(sc.shape) < 0.25
        big = (np.float32(2.0) ** rng.uniform(-4.0, -2.0, size=sc.shape)).astype(np.float32)
        big_bits = (big.view(np.uint32) >> 16).astype(np.uint16)  # truncated to bf16: still >= 2^-4
        sc[pick] = big_bits[pick]
        f = (sc.astype(np.uint32) << 16).view(np.float32)
        q["scale"] = sc.view(np.asarray(q["scale"]).dtype)
        q["bias"] = ((np.float32(-8.0) * f).view(np.uint32) >> 16).astype(np.uint16).view(np.asarray(q["bias"]).dtype)
        npl[mat] = q
    return npl


@pytest.mark.parametrize("T", [300, 2000], ids=["narrow_cfg", "wide_cfg"])
def test_prefill_mixed_scales(m, T):
    """Warps whose rows mix scales below and above 2^-4 take the base-subtracting dequantization,
    the others the subnormal one (narrow configuration); both must match the oracle."""
    npl = mixed_scale_layer(FULL, 31)
    layer = m.upload_layer(npl)
    assert m.prefill_tile_rows(layer.dims, T) == (32 if T * FULL.top_k <= 24 * FULL.n_experts else m.tile_rows())
    prefill_and_check(m, FULL, T, seed=31, npl=npl, layer=layer, hidden=True)


def test_prefill_out_of_range_sets_status(m):
    """x beyond the fp16 operand range is reported on the device instead of silently saturating."""
    layer = dev_layer(m, TINY)
    x = make_tokens(8, TINY.d, seed=4)
    x[2, 17] = 0x7F00                          # bf16 1.7e38
    ws = m.workspace(layer.dims, 8)
    m.prefill(layer, to_dev(x), ws)
    assert m.read_device_status(ws) == 8
    m.prefill(layer, to_dev(make_tokens(8, TINY.d, seed=4)), ws)
    assert m.read_device_status(ws) == 0


@pytest.mark.parametrize("shape", [MID, WIDE], ids=["E300k9", "E1024k16"])
def test_prefill_wide_shapes(m, shape):
    prefill_and_check(m, shape, 200, hidden=True)


def test_prefill_scale_outside_fp16_range_sets_status(m):
    """A shared-expert scale the fp16 dequantization cannot hold exactly (2^-24, below the normal
    fp16 range) or that could overflow it (32768: 15 * scale > 65504) is reported as
    MOE_ERR_OUT_OF_RANGE; the unmodified layer reports nothing."""
    x = to_dev(make_tokens(64, TINY.d, seed=6))
    for bits in (0x3380, 0x4700):
        npl = dict(_np_layer(TINY, 0, None))
        q = dict(npl["sh_gate"])
        q["scale"] = q["scale"].copy()
        q["scale"][5, 2] = bits
        npl["sh_gate"] = q
        layer = m.upload_layer(npl)
        ws = m.workspace(layer.dims, 64)
        m.prefill(layer, x, ws)
        assert m.read_device_status(ws) == 8, hex(bits)
    layer = dev_layer(m, TINY)
    ws = m.workspace(layer.dims, 64)
    m.prefill(layer, x, ws)
    assert m.read_device_status(ws) == 0


def test_prefill_repeatable(m):
    shape = TINY
    layer = dev_layer(m, shape)
    x = to_dev(make_tokens(200, shape.d, seed=9))
    ws = m.workspace(layer.dims, 200)
    y1 = C.bf16_bits_f64(m.prefill(layer, x, ws))
    y2 = C.bf16_bits_f64(m.prefill(layer, x, ws))
    assert m.read_device_status(ws) == 0
    # the fp32 combine adds in any order: the two runs may differ by one bf16 unit of the output
    np.testing.assert_allclose(y1, y2, rtol=2.0 ** -7, atol=1e-6)



def test_prefill_full_replays_identical(m):
    """Two full-size layers prefilled alternately, 12 times each: the hidden rows (no atomics on
    their path) must be bit-identical every time and y equal up to the rounding order of the
    fp32 combine (one bf16 unit). Catches pipeline races that corrupt an occasional work item."""
    T = 4096
    layers = [dev_layer(m, FULL, seed) for seed in (0, 1)]
    xs = [to_dev(make_tokens(T, FULL.d, seed=50 + seed)) for seed in (0, 1)]
    ws = m.workspace(layers[0].dims, T)

    def run(i):
        out = m.route_out_tensors(layers[i].dims, T, "cuda", want=("n_tiles", "hidden"), hidden=True)
        y = m.prefill(layers[i], xs[i], ws, out=out)
        return out["hidden"].clone(), y.view(torch.bfloat16).float()

    first = [run(0), run(1)]
    for rep in range(12):
        for i in (0, 1):
            h, y = run(i)
            h0, y0 = first[i]
            assert torch.equal(h, h0), f"replay {rep} layer {i}: hidden rows differ"
            bad = (y - y0).abs() > 2.0 ** -7 * torch.clamp(y0.abs(), min=1e-3) + 1e-6
            assert not bool(bad.any()), f"replay {rep} layer {i}: {int(bad.sum())} outputs differ"
    torch.cuda.synchronize()
    assert m.read_device_status(ws) == 0

# ------------------------------------------------------------------------------ prefill ablation arms
@pytest.mark.parametrize("arm", [1, 2, 3, 4, 5], ids=["host_routing", "tile32", "dense", "wide_cfg", "narrow_cfg"])
@pytest.mark.parametrize("shape,T,bias", [(TINY, 300, None), (FULL, 512, None), (FULL, 2048, "zipf")],
                         ids=["tiny300", "full512", "skew2048"])
def test_prefill_ablation_arms(m, arm, shape, T, bias):
    """Both ablation arms compute the same layer: against the oracle (sampled rows at full size)
    and against moe_prefill up to the fp32 summation order of the combine and of K sums over
    tiles of another width."""
    npl, layer = _np_layer(shape, 0, bias), dev_layer(m, shape, 0, bias)
    x = make_tokens(T, shape.d, seed=400 + T)
    xd = to_dev(x)
    ws = m.workspace(layer.dims, T)
    n_aux = m.ablation_aux_bytes(layer.dims, arm)
    aux = torch.empty(n_aux, dtype=torch.uint8, device="cuda") if n_aux else None
    y = m.prefill_ablation(layer, xd, ws, arm, aux=aux)
    torch.cuda.synchronize()
    assert m.read_device_status(ws) == 0
    y1 = m.prefill(layer, xd, ws)
    torch.cuda.synchronize()
    assert _same_up_to_summation_order(y, y1) == 0
    rows = np.arange(T) if T <= 300 else np.unique(np.concatenate([[0, T - 1], np.random.default_rng(T).choice(T, 30)]))
    C.check_y(y[torch.as_tensor(rows, device=y.device)], _oracle_rows(m, layer, npl, shape, x[rows]))


# ------------------------------------------------------------------------------ bounded-chunk prefill
def _oracle_rows(m, layer, npl, shape, x):
    """Oracle y for the token rows x; where the oracle's k-th and (k+1)-th logits lie within the
    logit tolerance, the selection follows the GPU's own logits (from moe_route on the same rows)."""
    g = run_route(m, layer, x.shape[0], x=x)
    ref_logits = O.router_logits(x, npl["router_w"], npl["router_bias"])
    tol = C.logit_tolerance(x, npl["router_w"]) + 1e-6 * np.abs(ref_logits)
    diff, ok = C.selection_with_near_ties(g["logits"], ref_logits, tol, shape.top_k)
    assert ok, f"tokens {diff} select different experts without a near tie"
    routing = None
    if diff:
        idx = g["topk_idx"]
        sel = np.take_along_axis(ref_logits.astype(np.float64), idx.astype(np.int64), axis=1)
        w = np.exp(sel - sel.max(1, keepdims=True))
        routing = (idx, w / w.sum(1, keepdims=True))
    return O.moe_forward(x, npl, tile_rows=m.tile_rows(), routing=routing)["y"]


def _same_up_to_summation_order(y, y0):
    """bf16 outputs of the same rows prefilled in different chunks. A row's expert tiles differ in
    size between chunkings, and a tile of at most 96 rows sums its K blocks in another order, so
    the hidden rows and the combine may round differently in fp32: one bf16 unit plus an absolute
    2^-12 of the output's rms (fp32 reordering of sums whose terms reach the output's size)."""
    a = torch.as_tensor(y).view(torch.bfloat16).float()
    b = torch.as_tensor(y0).view(torch.bfloat16).float()
    rms = float(b.pow(2).mean().sqrt())
    bad = (a - b).abs() > 2.0 ** -7 * b.abs() + 2.0 ** -12 * rms
    return int(bad.sum())


@pytest.mark.parametrize("T,chunk", [(300, 64), (5, 1), (37, 100), (192 * 3 + 1, 192)])
def test_prefill_chunked_tiny(m, T, chunk):
    """Chunks of 64 rows (4 whole + a ragged 44), one row per chunk, a chunk larger than the
    prompt, and chunks of exactly one block-map tile: y against the oracle on every row and
    against a single moe_prefill call."""
    npl, layer = _np_layer(TINY, 0, None), dev_layer(m, TINY)
    x = make_tokens(T, TINY.d, seed=200 + T)
    ws = m.workspace(layer.dims, min(chunk, T))
    y = m.prefill_chunked(layer, to_dev(x), ws, chunk)
    torch.cuda.synchronize()
    assert m.read_device_status(ws) == 0
    C.check_y(y, _oracle_rows(m, layer, npl, TINY, x))
    y1 = m.prefill(layer, to_dev(x), m.workspace(layer.dims, T))
    assert _same_up_to_summation_order(y, y1) == 0


def test_prefill_chunked_full(m):
    """Full-size layer, 5000 tokens in chunks of 2048 (two whole chunks + a ragged 904): equal to one
    moe_prefill call up to fp32 summation order, and sampled rows (every chunk's first and last
    row among them) against the oracle."""
    T, chunk = 5000, 2048
    npl, layer = _np_layer(FULL, 0, None), dev_layer(m, FULL)
    x = make_tokens(T, FULL.d, seed=301)
    xd = to_dev(x)
    ws = m.workspace(layer.dims, chunk)
    y = m.prefill_chunked(layer, xd, ws, chunk)
    torch.cuda.synchronize()
    assert m.read_device_status(ws) == 0
    y1 = m.prefill(layer, xd, m.workspace(layer.dims, T))
    assert _same_up_to_summation_order(y, y1) == 0
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, chunk - 1, chunk, 2 * chunk - 1, 2 * chunk, T - 1],
                                     rng.choice(T, 26, replace=False)]))
    C.check_y(y[torch.as_tensor(rows, device=y.device)], _oracle_rows(m, layer, npl, FULL, x[rows]))


def test_prefill_chunked_beyond_single_call_limit(m):
    """70001 tokens (over the 65536 of one moe_prefill call) with a workspace for 32768: every row
    finite, sampled rows (the chunk edges among them) against the oracle."""
    T, chunk = 70001, 32768
    npl, layer = _np_layer(TINY, 0, None), dev_layer(m, TINY)
    x = make_tokens(T, TINY.d, seed=302)
    ws = m.workspace(layer.dims, chunk)
    y = m.prefill_chunked(layer, to_dev(x), ws, chunk)
    torch.cuda.synchronize()
    assert m.read_device_status(ws) == 0
    yf = C.bf16_bits_f64(y)
    assert np.all(np.isfinite(yf))
    rng = np.random.default_rng(8)
    rows = np.unique(np.concatenate([[0, chunk - 1, chunk, 2 * chunk - 1, 2 * chunk, T - 1],
                                     rng.choice(T, 58, replace=False)]))
    C.check_y(yf[rows], _oracle_rows(m, layer, npl, TINY, x[rows]))


# ------------------------------------------------------------------------------ decode
@pytest.mark.parametrize("shape,bias,seed", [(TINY, None, 0), (FULL, None, 0), (FULL, None, 1),
                                             (FULL, "zipf", 2), (MID, None, 3), (WIDE, None, 4),
                                             (LONGI, None, 5), (ODDI, None, 6), (BIGD, None, 7)],
                         ids=["tiny", "full0", "full1", "zipf", "E300k9", "E1024k16", "I1024", "d384I384",
                              "d3072I640"])
def test_decode(m, shape, bias, seed):
    npl = _np_layer(shape, seed, bias)
    layer = dev_layer(m, shape, seed, bias)
    for step in range(3):
        x = make_tokens(1, shape.d, seed=seed, stream=step + 1)
        ws = m.workspace(layer.dims, 1)
        out = m.route_out_tensors(layer.dims, 1, "cuda", want=("logits", "topk_idx", "topk_w"))
        y = m.decode(layer, to_dev(x), ws, out=out)
        torch.cuda.synchronize()
        assert m.read_device_status(ws) == 0
        g = C.to_np(out)
        idx_ref, w_ref = O.select_experts(g["logits"], shape.top_k)
        np.testing.assert_array_equal(g["topk_idx"], idx_ref)
        assert np.max(np.abs(g["topk_w"] - w_ref)) <= C.W_TOL
        ref_logits = O.router_logits(x, npl["router_w"], npl["router_bias"])
        tol = C.logit_tolerance(x, npl["router_w"]) + 1e-6 * np.abs(ref_logits)
        assert np.all(np.abs(g["logits"] - ref_logits) <= tol)
        diff, ok = C.selection_with_near_ties(g["logits"], ref_logits, tol, shape.top_k)
        assert ok and not diff
        ref = O.moe_forward(x, npl, tile_rows=m.tile_rows())
        C.check_y(y, ref["y"])



@pytest.mark.parametrize("shape,T,force", [(FULL, 2, False), (FULL, 3, False), (FULL, 5, False), (FULL, 8, False),
                                           (FULL, 8, True), (FULL, 1, False), (TINY, 4, False), (WIDE, 6, False),
                                           (LONGI, 3, False), (ODDI, 5, False)],
                         ids=["full2", "full3", "full5", "full8", "full8_shared_experts", "full1", "tiny4",
                              "E1024k16_6", "I1024_3", "d384I384_5"])
def test_decode_batch(m, shape, T, force):
    """moe_decode_batch on T tokens: the routing of every token bit-exact against the oracle's
    selection on the GPU's logits, every token's y within the output tolerance of the oracle and
    equal to its own batch-1 moe_decode up to fp32 summation order; `force` sends every token to
    experts 0..k-1 (one distinct expert set shared by all tokens)."""
    npl = dict(_np_layer(shape, 5, None))
    if force:
        rb = np.zeros(shape.n_experts, dtype=np.float32)
        rb[: shape.top_k] = 100.0
        npl["router_bias"] = rb
        layer = m.upload_layer(npl)
    else:
        layer = dev_layer(m, shape, 5, None)
    x = make_tokens(T, shape.d, seed=600 + T)
    ws = m.workspace(layer.dims, T)
    out = m.route_out_tensors(layer.dims, T, "cuda", want=("logits", "topk_idx", "topk_w"))
    y = m.decode_batch(layer, to_dev(x), ws, out=out)
    torch.cuda.synchronize()
    assert m.read_device_status(ws) == 0
    g = C.to_np(out)
    idx_ref, w_ref = O.select_experts(g["logits"], shape.top_k)
    np.testing.assert_array_equal(g["topk_idx"], idx_ref)
    assert np.max(np.abs(g["topk_w"] - w_ref)) <= C.W_TOL
    if force:
        assert np.all(np.sort(g["topk_idx"], axis=1) == np.arange(shape.top_k))
    ref_logits = O.router_logits(x, npl["router_w"], npl["router_bias"])
    tol = C.logit_tolerance(x, npl["router_w"]) + 1e-6 * np.abs(ref_logits)
    assert np.all(np.abs(g["logits"] - ref_logits) <= tol)
    diff, ok = C.selection_with_near_ties(g["logits"], ref_logits, tol, shape.top_k)
    assert ok and not diff
    C.check_y(y, O.moe_forward(x, npl, tile_rows=m.tile_rows())["y"])
    ws1 = m.workspace(layer.dims, 1)
    for t in range(T):
        y1 = m.decode(layer, to_dev(x[t:t + 1]), ws1)
        assert _same_up_to_summation_order(y[t:t + 1], y1) == 0, f"token {t}"


def test_decode_batch_rejects_shapes(m):
    layer = dev_layer(m, FULL)
    ws = m.workspace(layer.dims, 16)
    with pytest.raises(m.MoeError):
        m.decode_batch(layer, to_dev(make_tokens(9, FULL.d, seed=1)), ws)   # more than 8 tokens


def test_decode_out_of_range_sets_status(m):
    """x beyond the fp16 operand range of the decode GEMVs (65536) is reported on the device."""
    layer = dev_layer(m, TINY)
    x = make_tokens(1, TINY.d, seed=4)
    x[0, 17] = 0x4780                          # bf16 65536
    ws = m.workspace(layer.dims, 1)
    m.decode(layer, to_dev(x), ws)
    assert m.read_device_status(ws) == 8
    m.decode(layer, to_dev(make_tokens(1, TINY.d, seed=4)), ws)
    assert m.read_device_status(ws) == 0


def test_bounded_wait_gives_up_and_reports(m):
    """Failure detection without a GPU fault: a bounded mbarrier wait that nothing satisfies (the
    wait routine of the GEMM and decode kernels) gives up after about a second and records
    MOE_ERR_DEVICE_TIMEOUT, which the host reads once and which is then cleared; the context stays
    usable (a decode right after matches the oracle)."""
    import time
    layer = dev_layer(m, TINY)
    ws = m.workspace(layer.dims, 1)
    t0 = time.perf_counter()
    m.selftest_wait_timeout(ws)
    assert m.read_device_status(ws) == 7
    assert 0.2 < time.perf_counter() - t0 < 60
    assert m.read_device_status(ws) == 0
    x = make_tokens(1, TINY.d, seed=0, stream=1)
    y = m.decode(layer, to_dev(x), ws)
    torch.cuda.synchronize()
    assert m.read_device_status(ws) == 0
    C.check_y(y, O.moe_forward(x, _np_layer(TINY, 0, None), tile_rows=m.tile_rows())["y"])


def test_decode_diagnostics(m):
    """moe_decode_diag: the arithmetic-deleted chain gives zeros, the read-only probe only reads;
    neither disturbs the workspace for the next regular decode."""
    layer = dev_layer(m, FULL)
    ws = m.workspace(layer.dims, 1)
    x = make_tokens(1, FULL.d, seed=21)
    xd = to_dev(x)
    y = m.decode_diag(layer, xd, ws, m.DECODE_DIAG_NO_MATH)
    torch.cuda.synchronize()
    assert m.read_device_status(ws) == 0
    assert not bool((y.view(torch.int16) & 0x7FFF).any()), "no-math decode must give zeros"
    m.decode_diag(layer, xd, ws, m.DECODE_DIAG_READ_ONLY)
    torch.cuda.synchronize()
    assert m.read_device_status(ws) == 0
    with pytest.raises(m.MoeError):
        m.decode_diag(layer, xd, ws, 3)
    y = m.decode(layer, xd, ws)
    torch.cuda.synchronize()
    C.check_y(C.bf16_bits_f64(y), O.moe_forward(x, _np_layer(FULL, 0, None), tile_rows=m.tile_rows())["y"], "decode after diagnostics")

@pytest.mark.parametrize("shape,T,bias", [(FULL, 512, None), (FULL, 2048, "zipf"), (ODDI, 300, None),
                                          (BIGD, 100, None)])
def test_prefill_read_probe(m, shape, T, bias):
    """moe_prefill_diag's read-only probes: no device error (every bounded wait was satisfied, so
    every copy landed), y zeros (nothing accumulated), the events in kernel order; regular prefills
    before and after give the same y up to the combine's summation order; an unknown mode is
    refused."""
    layer = dev_layer(m, shape, 0, bias)
    xd = to_dev(make_tokens(T, shape.d, seed=610 + T))
    ws = m.workspace(layer.dims, T)
    y0 = m.prefill(layer, xd, ws)
    y = torch.full_like(xd, 0x3C00)
    m.prefill_diag(layer, xd, ws, m.PREFILL_DIAG_READ_ONLY, y=y)
    torch.cuda.synchronize()
    assert m.read_device_status(ws) == 0
    assert not bool((y & 0x7FFF).any()), "the read-only probes accumulate nothing"
    # events at the kernel boundaries, recorded eagerly and as nodes of a captured graph
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in evs:
        e.record()
    m.prefill_diag(layer, xd, ws, m.PREFILL_DIAG_READ_ONLY, y=y, events=evs)
    torch.cuda.synchronize()
    assert all(evs[i].elapsed_time(evs[i + 1]) >= 0 for i in range(5))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        m.prefill_diag(layer, xd, ws, m.PREFILL_DIAG_READ_ONLY, y=y, events=evs)
    g.replay()
    torch.cuda.synchronize()
    assert all(evs[i].elapsed_time(evs[i + 1]) >= 0 for i in range(5))
    assert m.read_device_status(ws) == 0
    with pytest.raises(m.MoeError):
        m.prefill_diag(layer, xd, ws, 2)
    y1 = m.prefill(layer, xd, ws)
    torch.cuda.synchronize()
    assert m.read_device_status(ws) == 0
    assert _same_up_to_summation_order(y0, y1) == 0


def test_decode_matches_prefill_T1(m):
    shape = FULL
    layer = dev_layer(m, shape)
    x = to_dev(make_tokens(1, shape.d, seed=5))
    y_dec = C.bf16_bits_f64(m.decode(layer, x, m.workspace(layer.dims, 1)))
    y_pre = C.bf16_bits_f64(m.prefill(layer, x, m.workspace(layer.dims, 1)))
    C.check_y(y_dec, y_pre, "decode vs prefill")
