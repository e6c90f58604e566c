"""Pins of the CPU oracle to facts outside itself (CPU only).

Each check compares the oracle with something it does not compute: hand-derived values from
the pages' format, pure-Python brute force on tiny inputs, closed forms, exact integer cases,
library routines for special cases, and invariants of the grouping. ``test_planted_mistakes``
shows that plausible slips in the oracle (dropped bias, nibble order, tie-break, transposed
operand, missing shared expert, unnormalised weights) each fail at least one pin.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import moe_oracle as O
from synthetic import LayerShape, make_layer, make_tokens, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(vals):
    return f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


# ------------------------------------------------------------------------------------------
# Number formats
# ------------------------------------------------------------------------------------------
def pin_bf16_values():
    # bit patterns worked by hand: sign | 8-bit exponent (bias 127) | 7-bit mantissa
    table = {0x3F80: 1.0, 0xC000: -2.0, 0x3F00: 0.5, 0xC080: -4.0, 0x3C00: 2.0 ** -7,
             0x4049: 3.140625, 0x0000: 0.0, 0x8000: -0.0, 0x3FC0: 1.5}
    got = O.bf16_to_f64(np.array(list(table), dtype=np.uint16))
    assert np.array_equal(got, np.array(list(table.values())))


def pin_golden_group():
    with open(os.path.join(GOLDEN, "q4_group_example.json")) as f:
        g = json.load(f)
    words = np.array([[int(w, 16) for w in g["words"]]], dtype=np.uint32)
    codes = O.unpack_codes(words, 64)
    assert codes[0].tolist() == g["codes"]
    mat = {"q": words, "scale": np.array([[int(g["scale_bits"], 16)]], dtype=np.uint16),
           "bias": np.array([[int(g["bias_bits"], 16)]], dtype=np.uint16)}
    assert O.dequant(mat)[0].tolist() == g["weights"]


def pin_dequant_special_cases():
    rng = np.random.default_rng(5)
    scale = _bf16(rng.uniform(0.01, 0.03, size=(3, 2)))
    bias = _bf16(-8.0 * O.bf16_to_f64(scale))
    # every code 8 with bias = -8*scale gives exactly zero weights
    mat = {"q": np.full((3, 16), 0x88888888, dtype=np.uint32), "scale": scale, "bias": bias}
    assert np.all(O.dequant(mat) == 0.0)
    # scale 1, bias -8: w = q - 8, an integer per code, independent of column grouping
    words = rng.integers(0, 2**32, size=(3, 16), dtype=np.uint32)
    mat = {"q": words, "scale": _bf16(np.ones((3, 2))), "bias": _bf16(np.full((3, 2), -8.0))}
    w = O.dequant(mat)
    for r in range(3):
        for c in range(128):
            assert w[r, c] == ((int(words[r, c // 8]) >> (4 * (c % 8))) & 15) - 8
    # the group of column c is c // 64: a distinct scale per group shows up in the right columns
    mat = {"q": np.full((1, 16), 0x99999999, dtype=np.uint32),
           "scale": _bf16([[1.0, 2.0]]), "bias": _bf16([[0.0, 0.5]])}
    w = O.dequant(mat)[0]
    assert np.all(w[:64] == 9.0) and np.all(w[64:] == 18.5)


def pin_silu_closed_forms():
    # sigmoid(ln 3) = 3/4 and sigmoid(-ln 3) = 1/4, so silu(+-ln 3) = +-ln3 * {3/4, 1/4}
    z = np.array([0.0, math.log(3.0), -math.log(3.0), 40.0, -800.0])
    s = O.silu(z)
    assert s[0] == 0.0
    assert abs(s[1] - 0.75 * math.log(3.0)) < 1e-15
    assert abs(s[2] + 0.25 * math.log(3.0)) < 1e-15
    assert abs(s[3] - 40.0) < 1e-12 and s[4] == 0.0


# ------------------------------------------------------------------------------------------
# Router and selection
# ------------------------------------------------------------------------------------------
def pin_router_integer_exact():
    rng = np.random.default_rng(1)
    x = rng.integers(-3, 4, size=(5, 128))
    wr = rng.integers(-2, 3, size=(6, 128))
    got = O.router_logits(_bf16(x), _bf16(wr))
    for t in range(5):
        for e in range(6):
            assert got[t, e] == float(sum(int(a) * int(b) for a, b in zip(x[t], wr[e])))
    bias = np.array([0.5, -1.0, 0, 0, 0, 2.25], dtype=np.float32)
    got_b = O.router_logits(_bf16(x), _bf16(wr), bias)
    assert np.array_equal(got_b, got + bias)


def _brute_topk(row, k):
    key = lambda e: (-(row[e] + 0.0), e)  # noqa: E731  (+0.0 folds -0.0 onto +0.0)
    return sorted(range(len(row)), key=key)[:k]


def pin_topk_bruteforce():
    rng = np.random.default_rng(2)
    cases = [rng.standard_normal((64, 16)).astype(np.float32)]
    tied = np.round(rng.standard_normal((64, 16)) * 2) / 2          # many exact ties
    cases.append(tied.astype(np.float32))
    hand = np.zeros((4, 16), dtype=np.float32)
    hand[1, [3, 7, 9]] = 1.0                                        # tie straddling k
    hand[2, :] = -0.0
    hand[2, [5, 11]] = 0.0                                          # -0.0 == +0.0
    hand[3, ::-1] = np.arange(16, dtype=np.float32)
    cases.append(hand)
    for logits in cases:
        for k in (1, 2, 5, 16):
            idx, w = O.select_experts(logits, k)
            for t in range(logits.shape[0]):
                row = [float(v) for v in logits[t]]
                want = _brute_topk(row, k)
                assert idx[t].tolist() == want
                ex = [math.exp(row[e] - row[want[0]]) for e in want]
                tot = sum(ex)
                for j in range(k):
                    assert abs(w[t, j] - ex[j] / tot) <= 1e-15
    assert O.select_experts(hand, 2)[0][0].tolist() == [0, 1]       # all-equal row: lowest first
    assert O.select_experts(hand, 2)[0][1].tolist() == [3, 7]


def pin_topk_special_weights():
    rng = np.random.default_rng(3)
    l = rng.standard_normal((32, 24)).astype(np.float32)
    _, w1 = O.select_experts(l, 1)
    assert np.all(w1 == 1.0)
    _, w_eq = O.select_experts(np.full((2, 24), 0.7, dtype=np.float32), 6)
    assert np.allclose(w_eq, 1.0 / 6, rtol=1e-15, atol=0)
    idx, w_all = O.select_experts(l, 24)                            # k = E: full softmax
    soft = scipy.special.softmax(l.astype(np.float64), axis=1)
    assert np.allclose(np.take_along_axis(soft, idx, axis=1), w_all, rtol=1e-13, atol=0)
    _, w8 = O.select_experts(l, 8)
    assert np.allclose(w8.sum(axis=1), 1.0, rtol=0, atol=1e-14) and np.all(np.diff(w8, axis=1) <= 0)


# ------------------------------------------------------------------------------------------
# Grouping
# ------------------------------------------------------------------------------------------
def pin_grouping(tile_rows=4):
    rng = np.random.default_rng(4)
    T, k, E = 37, 3, 8
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    idx[:10] = [0, 1, 2]                                            # one heavy expert
    G = O.group_assignments(idx, E, tile_rows)
    flat = idx.reshape(-1)
    assert G["counts"].sum() == T * k
    assert np.all(np.diff(G["offsets"]) >= 0) and G["offsets"][0] == 0 and G["offsets"][-1] == T * k
    assert sorted(G["perm"].tolist()) == list(range(T * k))          # bijection
    assert np.all(G["inv_perm"][G["perm"]] == np.arange(T * k))
    brute = sorted(range(T * k), key=lambda a: (flat[a], a))        # stable sort by expert
    assert G["perm"].tolist() == brute
    for e in range(E):
        seg = G["perm"][G["offsets"][e]:G["offsets"][e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg // k) > 0)
        assert G["counts"][e] == int(np.sum(flat == e))
    tiles = []
    for e in range(E):
        c, r = int(G["counts"][e]), 0
        while r < c:
            tiles.append([e, r, min(tile_rows, c - r)])
            r += tile_rows
    assert G["tile_map"].tolist() == tiles and G["n_tiles"] == len(tiles)


def pin_page_facts():
    with open(os.path.join(GOLDEN, "page_facts.json")) as f:
        facts = json.load(f)["facts"]
    f0 = facts[0]
    rng = np.random.default_rng(6)
    idx = np.stack([rng.permutation(f0["n_experts"])[:f0["top_k"]] for _ in range(f0["tokens"])])
    G = O.group_assignments(idx, f0["n_experts"], 128)
    assert int(G["counts"].sum()) == f0["assignments"]
    assert G["counts"].mean() == f0["mean_rows_per_expert"]
    f2 = facts[2]
    assert 4 + 2 * 16 / f2["group"] == f2["bits_per_weight"]
    assert abs(f2["bf16_gb"] * f2["bits_per_weight"] / 16 - f2["q4_gb_reported"]) < 0.5


# ------------------------------------------------------------------------------------------
# Experts and combine
# ------------------------------------------------------------------------------------------
TINY_PIN = LayerShape(d=64, n_experts=4, top_k=2, inter=64, shared_inter=64)


def _py_dense_forward(x_bits, layer):
    """All-experts dense loop in pure Python floats; unselected experts get weight 0."""
    sh = layer["shape"]
    x = O.bf16_to_f64(x_bits).tolist()
    logits = O.router_logits(x_bits, layer["router_w"], layer.get("router_bias"))

    def mat(m, e=None):
        pick = (lambda a: a[e]) if e is not None else (lambda a: a)
        q, s, b = pick(m["q"]), O.bf16_to_f64(pick(m["scale"])), O.bf16_to_f64(pick(m["bias"]))
        rows, cols = s.shape[0], s.shape[1] * 64
        return [[s[r][c // 64] * ((int(q[r][c // 8]) >> (4 * (c % 8))) & 15) + b[r][c // 64]
                 for c in range(cols)] for r in range(rows)]

    def ffn(xt, g, u, dn):
        gv = [sum(a * b for a, b in zip(row, xt)) for row in g]
        uv = [sum(a * b for a, b in zip(row, xt)) for row in u]
        h = [gz / (1.0 + math.exp(-gz)) * uz for gz, uz in zip(gv, uv)]
        return [sum(a * b for a, b in zip(row, h)) for row in dn]

    experts = [(mat(layer["gate"], e), mat(layer["up"], e), mat(layer["down"], e)) for e in range(sh.n_experts)]
    shared = (mat(layer["sh_gate"]), mat(layer["sh_up"]), mat(layer["sh_down"]))
    ys = []
    for t in range(len(x)):
        row = [float(v) for v in logits[t]]
        sel = _brute_topk(row, sh.top_k)
        ex = {e: math.exp(row[e] - row[sel[0]]) for e in sel}
        tot = sum(ex.values())
        y = ffn(x[t], *shared)
        for e in range(sh.n_experts):
            w = ex[e] / tot if e in ex else 0.0
            contrib = ffn(x[t], *experts[e])
            y = [a + w * b for a, b in zip(y, contrib)]
        ys.append(y)
    return np.array(ys)


def pin_dense_bruteforce():
    layer = make_layer(TINY_PIN, seed=11)
    x = make_tokens(3, TINY_PIN.d, seed=11)
    got = O.moe_forward(x, layer, tile_rows=2)["y"]
    want = _py_dense_forward(x, layer)
    assert np.allclose(got, want, rtol=1e-10, atol=1e-10)


def pin_integer_expert():
    rng = np.random.default_rng(7)
    n, d, I = 3, 64, 64
    words = lambda rows, cols: rng.integers(0, 2**32, size=(rows, cols // 8), dtype=np.uint32)  # noqa: E731
    one = lambda rows, cols: _bf16(np.ones((rows, cols // 64)))  # noqa: E731
    m8 = lambda rows, cols: _bf16(np.full((rows, cols // 64), -8.0))  # noqa: E731
    gate = {"q": words(I, d), "scale": one(I, d), "bias": m8(I, d)}
    up = {"q": words(I, d), "scale": one(I, d), "bias": m8(I, d)}
    down = {"q": words(d, I), "scale": one(d, I), "bias": m8(d, I)}
    xi = rng.integers(-2, 3, size=(n, d))
    _, hid = O.expert_ffn(xi.astype(np.float64), gate, up, down, return_hidden=True)
    code = lambda m, r, c: ((int(m["q"][r, c // 8]) >> (4 * (c % 8))) & 15) - 8  # noqa: E731
    for t in range(n):
        for f in range(I):
            assert hid["g"][t, f] == sum(code(gate, f, c) * int(xi[t, c]) for c in range(d))
            assert hid["u"][t, f] == sum(code(up, f, c) * int(xi[t, c]) for c in range(d))


def pin_zero_routed_is_shared_only():
    layer = make_layer(TINY_PIN, seed=12)
    for m in ("gate", "up", "down"):
        layer[m]["scale"][:] = 0
        layer[m]["bias"][:] = 0
    x = make_tokens(5, TINY_PIN.d, seed=12)
    y = O.moe_forward(x, layer)["y"]
    sh = O.expert_ffn(O.bf16_to_f64(x), layer["sh_gate"], layer["sh_up"], layer["sh_down"])
    assert np.array_equal(y, sh)


def pin_token_permutation():
    layer = make_layer(TINY_PIN, seed=13)
    x = make_tokens(6, TINY_PIN.d, seed=13)
    pi = np.array([4, 0, 5, 2, 1, 3])
    a, b = O.moe_forward(x, layer), O.moe_forward(x[pi], layer)
    assert np.array_equal(a["topk_idx"][pi], b["topk_idx"])
    assert np.allclose(a["y"][pi], b["y"], rtol=1e-12, atol=1e-12)


def pin_hidden_sorted_matches_forward():
    layer = make_layer(TINY_PIN, seed=14)
    x = make_tokens(5, TINY_PIN.d, seed=14)
    out = O.moe_forward(x, layer, tile_rows=2)
    H = O.hidden_sorted(x, layer, out["grouping"])
    # the combine rebuilt from the sorted hidden rows equals the layer output
    G, k = out["grouping"], TINY_PIN.top_k
    y = np.zeros_like(out["y"])
    for e in range(TINY_PIN.n_experts):
        for p in range(G["offsets"][e], G["offsets"][e + 1]):
            a = G["perm"][p]
            y[a // k] += out["topk_w"].reshape(-1)[a] * (H[p] @ O.dequant({kk: layer["down"][kk][e] for kk in ("q", "scale", "bias")}).T)
    y += H[5 * k:] @ O.dequant(layer["sh_down"]).T
    assert np.allclose(y, out["y"], rtol=1e-12, atol=1e-12)


PINS = [pin_bf16_values, pin_golden_group, pin_dequant_special_cases, pin_silu_closed_forms,
        pin_router_integer_exact, pin_topk_bruteforce, pin_topk_special_weights, pin_grouping,
        pin_page_facts, pin_dense_bruteforce, pin_integer_expert, pin_zero_routed_is_shared_only,
        pin_token_permutation, pin_hidden_sorted_matches_forward]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ------------------------------------------------------------------------------------------
# Plausible mistakes planted in the oracle must each break a pin
# ------------------------------------------------------------------------------------------
def _fails_some_pin():
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            return True
    return False


def _mut_no_bias(mat, group=64):
    s = O.bf16_to_f64(mat["scale"])
    q = O.unpack_codes(mat["q"], s.shape[-1] * group).astype(np.float64)
    return q * np.repeat(s, group, axis=-1)


def _mut_high_nibble_first(q, cols):
    q = np.asarray(q, dtype=np.uint32)
    shifts = (np.uint32(28) - np.arange(8, dtype=np.uint32) * np.uint32(4))
    return ((q[..., :, None] >> shifts) & np.uint32(0xF)).reshape(q.shape[:-1] + (cols,)).astype(np.int64)


def _mut_ties_to_higher(logits, k):
    l = np.asarray(logits, dtype=np.float32)
    E = l.shape[1]
    order = (E - 1 - np.argsort(-l[:, ::-1], axis=1, kind="stable"))[:, :k]
    top = np.take_along_axis(l, order, axis=1).astype(np.float64)
    w = np.exp(top - top[:, :1])
    return order.astype(np.int32), w / w.sum(1, keepdims=True)


def _mut_unnormalised(logits, k):
    idx, _ = _orig_select(logits, k)
    l = np.asarray(logits, dtype=np.float64)
    soft = np.exp(l - l.max(1, keepdims=True))
    soft /= soft.sum(1, keepdims=True)
    return idx, np.take_along_axis(soft, idx, axis=1)


_orig_select = O.select_experts


def _mut_transposed_router(x_bits, w_bits, bias=None):
    x, w = O.bf16_to_f64(x_bits), O.bf16_to_f64(w_bits)
    l = (x @ w[:, ::-1].T).astype(np.float32)       # input dimension reversed
    return l if bias is None else (l + bias).astype(np.float32)


def _mut_gelu_gate(z):
    z = np.asarray(z, dtype=np.float64)
    return 0.5 * z * (1 + np.tanh(0.79788456 * (z + 0.044715 * z ** 3)))


def _mut_unstable_scatter(topk_idx, n_experts, tile_rows):
    G = _orig_group(topk_idx, n_experts, tile_rows)
    perm = G["perm"].copy()
    for e in range(n_experts):
        lo, hi = G["offsets"][e], G["offsets"][e + 1]
        perm[lo:hi] = perm[lo:hi][::-1]
    G["perm"] = perm
    G["inv_perm"][perm] = np.arange(perm.size)
    return G


_orig_group = O.group_assignments

MUTATIONS = {
    "dequant_without_bias": ("dequant", _mut_no_bias),
    "high_nibble_first": ("unpack_codes", _mut_high_nibble_first),
    "ties_to_higher_index": ("select_experts", _mut_ties_to_higher),
    "weights_not_renormalised": ("select_experts", _mut_unnormalised),
    "router_operand_transposed": ("router_logits", _mut_transposed_router),
    "gelu_instead_of_silu": ("silu", _mut_gelu_gate),
    "unstable_scatter": ("group_assignments", _mut_unstable_scatter),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(O, attr, fn)
    monkeypatch.setattr(oracle, attr, fn, raising=False)
    assert _fails_some_pin(), f"planted mistake {name} passed every pin"


def test_planted_missing_shared(monkeypatch):
    def forward_without_shared(x_bits, layer, tile_rows=128, routing=None):
        lay = dict(layer)
        lay["sh_down"] = {k: (np.zeros_like(v) if k != "q" else v) for k, v in layer["sh_down"].items()}
        return _orig_forward(x_bits, lay, tile_rows, routing)

    monkeypatch.setattr(O, "moe_forward", forward_without_shared)
    assert _fails_some_pin()


_orig_forward = O.moe_forward
