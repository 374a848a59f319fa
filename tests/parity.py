"""Parity rules between the CUDA library and the CPU oracle (shared by the GPU tests).

The rules (a reading of the layer's definition, stated once):
  * routing: on every token whose renormalised 8th/9th probability gap exceeds 1e-4,
    the chosen expert set must equal the oracle's exactly, in rank order wherever the
    adjacent probabilities differ by more than 1e-4 of the chosen mass; on a near-tie
    token the GPU's set must be one of the sets the oracle itself lists as valid;
  * weights: within 1e-5 of the oracle's (fp32 exp and division against double);
  * counts / offsets / permutation: exactly the histogram, exclusive scan and stable
    grouping of the GPU's own (validated) choices;
  * output: max |gpu - oracle| <= 1e-2 * max |oracle| over the compared tokens, where a
    near-tie token is compared with the oracle's output for the valid choice the GPU
    made (computed by the oracle, never taken from the GPU).
Expected values always come from ``oracle``; the GPU's choice only selects among them.
"""
from __future__ import annotations

import numpy as np

import synth
from oracle import Oracle, valid_choices

GAP_TOL = 1e-4
W_TOL = 1e-5
# A layer with an input RMSNorm routes on xn = bf16(x * r * w): the GPU's fp32 r and the
# oracle's double r differ by about 1e-7 (relative), so now and then an element of xn lands
# on the neighbouring bf16 value.  One such element i moves every logit e by
# delta = ulp(xn_i) * W_r[e, i], at most 2^-7 * |xn_i * W_r[e, i]|, and a renormalised
# weight by at most delta / 4 (the softmax derivative w_k (1 - w_k) <= 1/4), i.e. at most
# 2^-9 * |xn_i * W_r[e, i]|.  The bound below covers one such element with
# |xn_i * W_r[e, i]| up to 0.25 (|xn_i| = 4 against a router weight of 3 standard
# deviations); the largest difference seen over 40 stacked layers is 7.9e-5 (decode, T=8).
W_TOL_NORM = 5e-4
OUT_REL_TOL = 1e-2


def bf16_to_f64(bits) -> np.ndarray:
    return synth.f32_from_bf16_bits(np.asarray(bits, np.uint16)).astype(np.float64)


def check_routing(o: Oracle, L, x: np.ndarray, idx_gpu: np.ndarray, w_gpu: np.ndarray, ref=None):
    """Returns (report dict, alt dict token -> oracle-valid expert list the GPU chose)."""
    T, K = idx_gpu.shape
    ref = ref if ref is not None else o.route(L, x)
    w_tol = W_TOL_NORM if getattr(L, "norm_w", None) is not None else W_TOL
    near = ref["gap"] <= GAP_TOL
    alt = {}
    near_sets = {}
    flips = 0
    w_err = 0.0
    for t in range(T):
        g_set = sorted(idx_gpu[t].tolist())
        if not near[t]:
            assert g_set == sorted(ref["idx"][t].tolist()), f"token {t}: {idx_gpu[t]} vs {ref['idx'][t]}"
            # rank order where the oracle's probabilities are well separated
            logits = o.router_logits(L, x[t])
            _, _, _, ps, order = o.route_logits(L.dims, logits)
            S = ps[:K].sum()
            for k in range(K):
                sep_lo = k == 0 or ps[k - 1] - ps[k] > GAP_TOL * S
                sep_hi = ps[k] - ps[k + 1] > GAP_TOL * S
                if sep_lo and sep_hi:
                    assert idx_gpu[t, k] == order[k], f"token {t} rank {k}"
            wmap = dict(zip(ref["idx"][t].tolist(), ref["w"][t].tolist()))
            for k in range(K):
                d = abs(w_gpu[t, k] - wmap[int(idx_gpu[t, k])])
                w_err = max(w_err, d)
                assert d <= w_tol, f"token {t} weight {k}: |diff| {d} > {w_tol}"
        else:
            logits = o.router_logits(L, x[t])
            choices = valid_choices(o, L.dims, logits, GAP_TOL)
            near_sets[t] = choices
            match = [c for c in choices if sorted(c) == g_set]
            assert match, f"near-tie token {t}: GPU set {g_set} not among the valid sets {choices}"
            if g_set != sorted(ref["idx"][t].tolist()):
                flips += 1
                alt[t] = match[0]
            else:
                wmap = dict(zip(ref["idx"][t].tolist(), ref["w"][t].tolist()))
                for k in range(K):
                    d = abs(w_gpu[t, k] - wmap[int(idx_gpu[t, k])])
                    w_err = max(w_err, d)
                    assert d <= w_tol, f"token {t} weight {k}: |diff| {d} > {w_tol}"
    return dict(tokens=T, near_ties=int(near.sum()), flips=flips, w_err=w_err, near_sets=near_sets), alt


def check_tables(idx_gpu: np.ndarray, counts, offsets, perm, n_experts=256):
    flat = idx_gpu.reshape(-1)
    exp_counts = np.bincount(flat, minlength=n_experts)
    assert np.array_equal(np.asarray(counts)[:n_experts], exp_counts)
    exp_off = np.concatenate([[0], np.cumsum(exp_counts)])
    assert np.array_equal(np.asarray(offsets)[:n_experts + 1], exp_off)
    assert np.array_equal(np.asarray(perm)[:flat.size], np.argsort(flat, kind="stable"))


def check_output(o: Oracle, L, x: np.ndarray, out_gpu: np.ndarray, tokens=None, residual=False, alt=None,
                 ref_out=None, any_of=None):
    """Compares out_gpu (bf16 bits [T, H]) on `tokens` with the oracle.  Returns
    (max abs error, max abs oracle).

    ``alt``: token -> the valid expert set the GPU chose (from the routing check).
    ``any_of``: token -> every valid expert set of a near-tie token, for outputs whose
    routing was computed by a different kernel than the one the routing check read (the
    decode forward and the decode router sum the logits in different orders, so on a
    near tie they may pick different valid sets): such a token matches the closest of
    the oracle's outputs for those sets."""
    alt = alt or {}
    any_of = any_of or {}
    T = x.shape[0]
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    if ref_out is None:
        ref_out = o.forward(L, x[tokens], residual=residual)["out"]
    ref = bf16_to_f64(ref_out).copy()
    for i, t in enumerate(tokens):
        if int(t) in alt:
            ob, _ = o.token_forward_choice(L, x[t], alt[int(t)], residual=residual)
            ref[i] = bf16_to_f64(ob)
    got = bf16_to_f64(out_gpu[tokens])
    for i, t in enumerate(tokens):
        if int(t) in any_of:
            best = None
            for c in any_of[int(t)]:
                ob, _ = o.token_forward_choice(L, x[t], c, residual=residual)
                cand = bf16_to_f64(ob)
                if best is None or np.max(np.abs(got[i] - cand)) < np.max(np.abs(got[i] - best)):
                    best = cand
            ref[i] = best
    err = float(np.max(np.abs(got - ref)))
    scale = float(np.max(np.abs(ref)))
    assert np.all(np.isfinite(got)), "non-finite GPU output"
    assert err <= OUT_REL_TOL * scale, f"max err {err} > {OUT_REL_TOL} * {scale}"
    return err, scale
