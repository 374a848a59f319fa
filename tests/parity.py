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
# A layer with an input RMSNorm routes on bf16(x * r): the GPU's fp32 r and the oracle's
# double r differ by ~1e-7, so about one element in 2e4 rounds to the neighbouring bf16
# value, which moves a logit by up to 2^-8 * |x_i| * |W_r| (~1e-4) and a weight by a few
# 1e-5; the bound keeps a decade of headroom.
W_TOL_NORM = 1e-3
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
    flips = 0
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
                assert abs(w_gpu[t, k] - wmap[int(idx_gpu[t, k])]) <= w_tol, f"token {t} weight {k}"
        else:
            logits = o.router_logits(L, x[t])
            choices = valid_choices(o, L.dims, logits, GAP_TOL)
            match = [c for c in choices if sorted(c) == g_set]
            assert match, f"near-tie token {t}: GPU set {g_set} not among the valid sets {choices}"
            if g_set != sorted(ref["idx"][t].tolist()):
                flips += 1
                alt[t] = match[0]
            else:
                wmap = dict(zip(ref["idx"][t].tolist(), ref["w"][t].tolist()))
                for k in range(K):
                    assert abs(w_gpu[t, k] - wmap[int(idx_gpu[t, k])]) <= w_tol
    return dict(tokens=T, near_ties=int(near.sum()), flips=flips), alt


def check_tables(idx_gpu: np.ndarray, counts, offsets, perm, n_experts=256):
    flat = idx_gpu.reshape(-1)
    exp_counts = np.bincount(flat, minlength=n_experts)
    assert np.array_equal(np.asarray(counts)[:n_experts], exp_counts)
    exp_off = np.concatenate([[0], np.cumsum(exp_counts)])
    assert np.array_equal(np.asarray(offsets)[:n_experts + 1], exp_off)
    assert np.array_equal(np.asarray(perm)[:flat.size], np.argsort(flat, kind="stable"))


def check_output(o: Oracle, L, x: np.ndarray, out_gpu: np.ndarray, tokens=None, residual=False, alt=None,
                 ref_out=None):
    """Compares out_gpu (bf16 bits [T, H]) on `tokens` with the oracle.  Returns
    (max abs error, max abs oracle)."""
    alt = alt or {}
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
    err = float(np.max(np.abs(got - ref)))
    scale = float(np.max(np.abs(ref)))
    assert np.all(np.isfinite(got)), "non-finite GPU output"
    assert err <= OUT_REL_TOL * scale, f"max err {err} > {OUT_REL_TOL} * {scale}"
    return err, scale
