"""Pins of the grouped-query decode-attention oracle (oracle/gqa_oracle.c) against facts
fixed outside it: closed forms (one cached key; identical keys, where attention is the
plain mean of the values; two keys along one axis, where the weights are a logistic
function of the score difference), the grouping itself (grouped-query attention is
multi-head attention over key/value heads repeated Hq/Hkv times), invariance under a
permutation of the cached positions, and the sequence length (rows at or past it never
matter).  Four planted mistakes (scale 1/D, heads interleaved across groups, the last key
dropped, values read from the keys) must each fail a pin.

Sources: 16 query heads share 2 key/value heads (aimanavo.com, "Why is Perplexity's local
AI Lily faster than MLX", section "Qwen3.6's 256 experts and two layer kinds make the
MLX/Lily gap"); decode reads every KV row once per step for all the query heads of a group
(same page, section "Prefill and decode are not treated as the same job").
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import synth
from oracle import Oracle

D = 128


def bf(x):
    return synth.bf16_bits_from_f32(np.asarray(x, np.float32))


def f(bits):
    return synth.f32_from_bf16_bits(np.asarray(bits, np.uint16)).astype(np.float64)


def check_single_key(o):
    q, k, v, _ = synth.make_gqa(1, 2, 5, needles=0)
    lens = np.array([1, 1], np.int32)
    out, aout = o.gqa_decode(q, k, v, lens)
    for b in range(2):
        for h in range(16):
            assert np.array_equal(out[b, h], f(v[b, h // 8, 0])), (b, h)
            assert np.array_equal(aout[b, h], np.abs(f(v[b, h // 8, 0])))


def check_identical_keys_give_the_mean(o):
    q, k, v, _ = synth.make_gqa(2, 1, 37, needles=0)
    k[:] = k[:, :, :1, :]                       # every cached key the same
    out, _ = o.gqa_decode(q, k, v, np.array([37], np.int32))
    for h in range(16):
        want = np.mean(f(v[0, h // 8]), axis=0)
        assert np.allclose(out[0, h], want, rtol=0, atol=1e-12), h


def check_two_keys_logistic(o):
    # q = a e_0, k_0 = b0 e_0, k_1 = b1 e_0: scores a b_i / sqrt(D); weight of key 0 is
    # 1 / (1 + exp(s_1 - s_0))
    a, b0, b1 = 3.0, 2.5, -1.5
    q = np.zeros((1, 16, D), np.float32)
    q[0, :, 0] = a
    k = np.zeros((1, 2, 2, D), np.float32)
    k[0, :, 0, 0], k[0, :, 1, 0] = b0, b1
    rng = np.random.default_rng(5)
    v = rng.normal(size=(1, 2, 2, D)).astype(np.float32)
    out, _ = o.gqa_decode(bf(q), bf(k), bf(v), np.array([2], np.int32))
    s0, s1 = a * b0 / math.sqrt(D), a * b1 / math.sqrt(D)
    p0 = 1.0 / (1.0 + math.exp(s1 - s0))
    vv = f(bf(v))
    for h in range(16):
        want = p0 * vv[0, h // 8, 0] + (1 - p0) * vv[0, h // 8, 1]
        assert np.allclose(out[0, h], want, rtol=1e-14, atol=1e-14), h


def check_gqa_is_repeated_kv_mha(o):
    q, k, v, lens = synth.make_gqa(3, 2, 50, lens=[50, 17])
    out, _ = o.gqa_decode(q, k, v, lens)
    k16 = np.repeat(k, 8, axis=1)               # KV head j serves query heads 8j .. 8j+7
    v16 = np.repeat(v, 8, axis=1)
    mha, _ = o.gqa_decode(q, k16, v16, lens)
    assert np.array_equal(out, mha)


def check_permutation_of_positions(o):
    q, k, v, _ = synth.make_gqa(4, 1, 64)
    out, _ = o.gqa_decode(q, k, v, np.array([64], np.int32))
    perm = np.random.default_rng(6).permutation(64)
    out2, _ = o.gqa_decode(q, k[:, :, perm], v[:, :, perm], np.array([64], np.int32))
    assert np.allclose(out, out2, rtol=0, atol=1e-12)


def check_rows_past_the_length_ignored(o):
    q, k, v, _ = synth.make_gqa(5, 2, 40, lens=[29, 40])
    lens = np.array([29, 40], np.int32)
    out, _ = o.gqa_decode(q, k, v, lens)
    k2, v2 = k.copy(), v.copy()
    k2[0, :, 29:] = bf(np.full((2, 11, D), 30.0))   # keys that would dominate if read
    v2[0, :, 29:] = bf(np.full((2, 11, D), 1e4))
    out2, _ = o.gqa_decode(q, k2, v2, lens)
    assert np.array_equal(out, out2)
    out3, _ = o.gqa_decode(q[:1], k[:1, :, :29], v[:1, :, :29], np.array([29], np.int32))
    assert np.allclose(out[:1], out3, rtol=0, atol=1e-13)


ALL_CHECKS = [check_single_key, check_identical_keys_give_the_mean, check_two_keys_logistic,
              check_gqa_is_repeated_kv_mha, check_permutation_of_positions, check_rows_past_the_length_ignored]

MUTANTS = {11: "scale 1/D", 12: "heads interleaved across groups", 13: "last key dropped",
           14: "values read from the keys"}


@pytest.mark.parametrize("check", ALL_CHECKS, ids=[c.__name__ for c in ALL_CHECKS])
def test_gqa_oracle_pin(check):
    check(Oracle())


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=[MUTANTS[m] for m in sorted(MUTANTS)])
def test_gqa_mutant_is_caught(mutant):
    o = Oracle(mutant)
    caught = []
    for check in ALL_CHECKS:
        try:
            check(o)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(check.__name__)
    assert caught, f"no pin catches GQA mutant {mutant} ({MUTANTS[mutant]})"
