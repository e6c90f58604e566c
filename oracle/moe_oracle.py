"""Plain, slow, obviously correct CPU oracle of the 4-bit quantized MoE layer forward pass.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and bench.py's CPU
baseline / reference arm, never by the product path. It shares no code with the CUDA library.

Sources (page: "Perplexity's Lily beats MLX-LM on MacBook M5 because it only runs one model",
agentnative.dev):
  * "Why Qwen3.6-35B-A3B is a weird workload": a router scores 256 experts, picks 8, and one
    shared expert sees every token.
  * "Prefill: keep routing on the GPU, dequantize in flight": groupwise affine 4-bit weights,
    one bf16 scale and bias per 64 weights; routing = histogram, prefix scan, scatter and block
    map after the top-8 selection.
  * "Decode: minimize bytes per token" (fusion list): expert input projections with the gate
    activation; expert output projection with the routing scores and the shared expert.

Readings where the pages are silent (each is also listed in the design notes):
  * w = scale*q + bias with q in 0..15 unsigned, code c%8 of a row in bits 4*(c%8) of word c//8.
  * Selection on the fp32 logits, largest first, ties to the lower expert index, -0.0 == +0.0;
    weights = softmax restricted to the selected k (= softmax, top-k, renormalise).
  * Gate activation = SwiGLU: h = silu(W_gate x) * (W_up x), silu(z) = z / (1 + exp(-z)).
  * The shared expert is added unscaled (weight 1).
  * Scatter is stable in assignment order a = t*k + j; block map tiles are
    (expert, first row, rows) in expert order with a fixed tile height.

Precision: dequantized weights are exact in fp64; every dot product and the SwiGLU run in fp64;
router logits are rounded to fp32 (the precision the selection is taken in) before the optional
fp32 router bias is added. The layer output y is returned in fp64, unrounded.
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------------------------------------
# Number formats
# ----------------------------------------------------------------------------------------------
def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    u32 = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def unpack_codes(q, cols: int) -> np.ndarray:
    """4-bit codes of a canonical packed matrix: code of column c = (q[c//8] >> 4*(c%8)) & 0xF.

    MLX affine layout (page "Setup": "MLX affine 4-bit checkpoint with group size 64"),
    eight codes per uint32, low nibble first along the input dimension.
    """
    q = np.asarray(q, dtype=np.uint32)
    shifts = (np.arange(8, dtype=np.uint32) * np.uint32(4))
    codes = (q[..., :, None] >> shifts) & np.uint32(0xF)
    codes = codes.reshape(q.shape[:-1] + (q.shape[-1] * 8,))
    assert codes.shape[-1] == cols
    return codes.astype(np.int64)


def dequant(mat: dict, group: int = 64) -> np.ndarray:
    """Groupwise affine dequantization, exact in fp64: w[r, c] = scale[r, c//g] * q[r, c] + bias[r, c//g].

    Section "Prefill: keep routing on the GPU, dequantize in flight": every group of 64 weights
    shares a bf16 scale and a bf16 bias.
    """
    scale = bf16_to_f64(mat["scale"])
    bias = bf16_to_f64(mat["bias"])
    cols = scale.shape[-1] * group
    q = unpack_codes(mat["q"], cols).astype(np.float64)
    return q * np.repeat(scale, group, axis=-1) + np.repeat(bias, group, axis=-1)


def silu(z):
    """silu(z) = z / (1 + exp(-z)), the gate activation of SwiGLU (section "Decode: minimize bytes
    per token" names the experts' gate activation; SwiGLU is the reading taken)."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


# ----------------------------------------------------------------------------------------------
# Router and selection ("a router scores 256 expert sub-networks, picks 8")
# ----------------------------------------------------------------------------------------------
def router_logits(x_bits, router_w_bits, router_bias=None) -> np.ndarray:
    """l[t, e] = fp32( sum_i x[t, i] * W_r[e, i] ) (+ b_e in fp32).

    bf16 x bf16 products are exact in fp64 and the fp64 sum is rounded once to fp32, the
    precision the top-k decision is taken in.
    """
    l64 = bf16_to_f64(x_bits) @ bf16_to_f64(router_w_bits).T
    l32 = l64.astype(np.float32)
    if router_bias is not None:
        l32 = (l32 + np.asarray(router_bias, dtype=np.float32)).astype(np.float32)
    return l32


def select_experts(logits, k: int):
    """Top-k per token and its routing weights.

    Order: largest fp32 logit first, equal logits -> lower expert index first (-0.0 equals
    +0.0). Weights: w_j = exp(l_j - l_max) / sum over the k selected of exp(l - l_max), i.e.
    softmax over all experts, keep the top k, renormalise (the ratio is the same).
    Returns (topk_idx int32 [T, k], topk_w float64 [T, k]).
    """
    l = np.asarray(logits, dtype=np.float32)
    if not np.all(np.isfinite(l)):
        raise ValueError("non-finite router logits are outside the method's domain")
    # A stable sort of the negated logits keeps equal values in ascending expert order.
    order = np.argsort(-l, axis=1, kind="stable")[:, :k]
    top = np.take_along_axis(l, order, axis=1).astype(np.float64)
    ex = np.exp(top - top[:, :1])
    w = ex / ex.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w


# ----------------------------------------------------------------------------------------------
# Grouping: histogram -> exclusive prefix scan -> stable scatter -> block map
# (section "Prefill: keep routing on the GPU, dequantize in flight")
# ----------------------------------------------------------------------------------------------
def group_assignments(topk_idx, n_experts: int, tile_rows: int) -> dict:
    """Expert-contiguous order of the T*k token-expert assignments.

    Assignment a = t*k + j (token t, slot j) of expert e goes to sorted position
    p = offsets[e] + #{a' < a : expert(a') = e}; perm[p] = a, inv_perm[a] = p.
    Tiles: for each expert with rows, (e, r0, min(tile_rows, counts[e] - r0)) for
    r0 = 0, tile_rows, ...; experts in ascending order.
    """
    flat = np.asarray(topk_idx, dtype=np.int64).reshape(-1)
    n_assign = flat.shape[0]
    counts = np.zeros(n_experts, dtype=np.int64)
    for e in flat:                                   # histogram
        counts[e] += 1
    offsets = np.zeros(n_experts + 1, dtype=np.int64)
    for e in range(n_experts):                       # exclusive prefix scan
        offsets[e + 1] = offsets[e] + counts[e]
    cursor = offsets[:-1].copy()
    perm = np.empty(n_assign, dtype=np.int64)
    inv_perm = np.empty(n_assign, dtype=np.int64)
    for a in range(n_assign):                        # stable scatter, assignment order
        e = flat[a]
        perm[cursor[e]] = a
        inv_perm[a] = cursor[e]
        cursor[e] += 1
    tiles = []
    for e in range(n_experts):                       # block map
        for r0 in range(0, int(counts[e]), tile_rows):
            tiles.append((e, r0, min(tile_rows, int(counts[e]) - r0)))
    tile_map = np.array(tiles, dtype=np.int32).reshape(-1, 3)
    return {
        "counts": counts.astype(np.int32),
        "offsets": offsets.astype(np.int32),
        "perm": perm.astype(np.int32),
        "inv_perm": inv_perm.astype(np.int32),
        "tile_map": tile_map,
        "n_tiles": int(tile_map.shape[0]),
    }


# ----------------------------------------------------------------------------------------------
# Experts (SwiGLU) and the weighted combine with the shared expert
# ----------------------------------------------------------------------------------------------
def _expert_mats(layer: dict, e):
    if e == "shared":
        return layer["sh_gate"], layer["sh_up"], layer["sh_down"]
    pick = lambda m: {key: m[key][e] for key in ("q", "scale", "bias")}  # noqa: E731
    return pick(layer["gate"]), pick(layer["up"]), pick(layer["down"])


def expert_ffn(x64, gate: dict, up: dict, down: dict, group: int = 64, return_hidden: bool = False):
    """One expert on rows x64 [n, d]: h = silu(W_g x) * (W_u x); out = W_d h (all fp64).

    Section "Decode: minimize bytes per token" (fusion list): the input projections feed the gate
    activation, whose output goes through the output projection.
    """
    g = x64 @ dequant(gate, group).T
    u = x64 @ dequant(up, group).T
    h = silu(g) * u
    out = h @ dequant(down, group).T
    if return_hidden:
        return out, {"g": g, "u": u, "h": h}
    return out


def hidden_sorted(x_bits, layer: dict, grouping: dict) -> np.ndarray:
    """SwiGLU outputs h in expert-sorted row order: rows p < T*k are assignments perm[p];
    rows T*k + t are the shared expert on token t. Shape [T*k + T, I], fp64."""
    shape = layer["shape"]
    x64 = bf16_to_f64(x_bits)
    T, k = x64.shape[0], shape.top_k
    H = np.zeros((T * k + T, shape.inter), dtype=np.float64)
    offs, perm = grouping["offsets"], grouping["perm"]
    for e in range(shape.n_experts):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi > lo:
            toks = perm[lo:hi] // k
            _, hid = expert_ffn(x64[toks], *_expert_mats(layer, e), group=shape.group, return_hidden=True)
            H[lo:hi] = hid["h"]
    _, hid = expert_ffn(x64, *_expert_mats(layer, "shared"), group=shape.group, return_hidden=True)
    H[T * k:] = hid["h"]
    return H


def moe_forward(x_bits, layer: dict, tile_rows: int = 128, routing=None) -> dict:
    """The whole layer: y[t] = sum_j w[t,j] * FFN_{e(t,j)}(x_t) + FFN_shared(x_t).

    Section "Why Qwen3.6-35B-A3B is a weird workload": the router picks 8 of 256 experts per
    token and one shared expert sees every token (added with weight 1, the reading taken);
    section "Decode: minimize bytes per token": the routing scores weight the output projection.

    ``routing`` = (topk_idx, topk_w) overrides the oracle's own selection (used when the
    comparison must follow a selection taken on another path's logits).
    Returns logits (fp32), topk_idx, topk_w (fp64), the grouping, and y (fp64).
    """
    shape = layer["shape"]
    x64 = bf16_to_f64(x_bits)
    T = x64.shape[0]
    logits = router_logits(x_bits, layer["router_w"], layer.get("router_bias"))
    if routing is None:
        topk_idx, topk_w = select_experts(logits, shape.top_k)
    else:
        topk_idx, topk_w = (np.asarray(r) for r in routing)
    grouping = group_assignments(topk_idx, shape.n_experts, tile_rows)
    y = np.zeros((T, shape.d), dtype=np.float64)
    offs, perm, k = grouping["offsets"], grouping["perm"], shape.top_k
    w_flat = topk_w.reshape(-1).astype(np.float64)
    for e in range(shape.n_experts):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            continue
        assign = perm[lo:hi]
        toks = assign // k
        out = expert_ffn(x64[toks], *_expert_mats(layer, e), group=shape.group)
        y[toks] += w_flat[assign][:, None] * out     # each token appears once per expert
    y += expert_ffn(x64, *_expert_mats(layer, "shared"), group=shape.group)
    return {"logits": logits, "topk_idx": topk_idx, "topk_w": topk_w, "grouping": grouping, "y": y}
