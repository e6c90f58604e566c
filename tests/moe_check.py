"""Comparison rules between the CUDA path and the oracle (shared by the GPU tests, smoke and bench).

Routing (integers) must match bit for bit when both sides route the same fp32 logits. Logits,
routing weights and outputs are floating point and are compared within the tolerances below:
  * logits: |l_gpu - l_ref| <= 2^-16 * sum_i |x_i * W_r[e, i]| (+ one fp32 ulp of the bias add)
  * routing weights: |w_gpu - w_ref| <= 1e-6
  * outputs: max |y_gpu - y_ref| <= 2e-2 * max(1, |y_ref|) elementwise and
    ||y_gpu - y_ref||_F / ||y_ref||_F <= 5e-3.
When the GPU's own logits select a different expert set than the oracle's for some token, the
token is accepted only if the oracle's gap between the k-th and (k+1)-th logit is within twice
the logit tolerance (a near tie); the output comparison then follows the GPU's selection.
"""
from __future__ import annotations

import numpy as np

import oracle as O

Y_ELEM_TOL = 2e-2
Y_FROB_TOL = 5e-3
W_TOL = 1e-6


def bf16_bits_f64(t) -> np.ndarray:
    a = t.cpu().numpy() if hasattr(t, "cpu") else np.asarray(t)
    return O.bf16_to_f64(a.view(np.uint16))


def check_y(y_gpu, y_ref: np.ndarray, what: str = "y") -> dict:
    y = y_gpu if isinstance(y_gpu, np.ndarray) else bf16_bits_f64(y_gpu)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite GPU output"
    err = np.abs(y - y_ref)
    bound = Y_ELEM_TOL * np.maximum(1.0, np.abs(y_ref))
    worst = float(np.max(err / bound)) if err.size else 0.0
    frob = float(np.linalg.norm(err) / max(np.linalg.norm(y_ref), 1e-300))
    assert worst <= 1.0, f"{what}: elementwise error {worst:.3f} x tolerance"
    assert frob <= Y_FROB_TOL, f"{what}: relative Frobenius error {frob:.2e}"
    return {"max_err_over_tol": worst, "rel_frob": frob}


def logit_tolerance(x_bits, wr_bits) -> np.ndarray:
    return 2.0 ** -16 * (np.abs(O.bf16_to_f64(x_bits)) @ np.abs(O.bf16_to_f64(wr_bits)).T)


def check_routing_exact(gpu: dict, logits_used: np.ndarray, E: int, k: int, tile_rows: int) -> None:
    """Routes the GPU's own fp32 logits with the oracle and demands identical integer results."""
    idx_ref, w_ref = O.select_experts(logits_used, k)
    G = O.group_assignments(idx_ref, E, tile_rows)
    T = logits_used.shape[0]
    np.testing.assert_array_equal(gpu["topk_idx"], idx_ref)
    assert np.max(np.abs(gpu["topk_w"].astype(np.float64) - w_ref)) <= W_TOL
    for name in ("counts", "offsets", "perm", "inv_perm"):
        np.testing.assert_array_equal(gpu[name], G[name], err_msg=name)
    n = int(gpu["n_tiles"][0])
    assert n == G["n_tiles"]
    np.testing.assert_array_equal(gpu["tile_map"][:n], G["tile_map"])
    assert gpu["counts"].sum() == T * k


def selection_with_near_ties(gpu_logits, ref_logits, tol, k):
    """Returns (tokens whose expert sets differ, all such tokens are near ties)."""
    idx_g, _ = O.select_experts(gpu_logits, k)
    idx_r, _ = O.select_experts(ref_logits, k)
    diff = [t for t in range(idx_g.shape[0]) if set(idx_g[t]) != set(idx_r[t])]
    ok = True
    for t in diff:
        srt = np.sort(ref_logits[t].astype(np.float64))[::-1]
        if srt[k - 1] - srt[k] > 2 * tol[t].max():
            ok = False
    return diff, ok


def to_np(d: dict) -> dict:
    return {k: v.cpu().numpy() for k, v in d.items()}
