"""Grouped-query decode attention on the GPU (gqa_decode_attention, through the C ABI)
against the CPU oracle: 16 query heads over 2 KV heads, head size 128, at 4K and 32K
cached positions, ragged lengths, the largest batch, one cached position, and
determinism.

Tolerance, derived from the kernel's arithmetic: scores are fp32 sums of exact bf16
products, the probabilities are rounded to bf16 (relative error at most 2^-9) and the
normaliser sums the rounded values, so each output element is a convex combination
whose weights are within 2^-8 (relative) of the exact ones; its error is then at most
2^-8 * sum_i p_i |v_i| (the oracle's ``abs_out``), plus the final bf16 rounding (2^-9 of
the value) and fp32 accumulation (far below either).  The bound asserted per element:
|gpu - oracle| <= 2^-8 * abs_out + 2^-8 * |oracle| + 1e-6.  The synthetic keys include
planted "needles" (a head's own query copied into its KV head), so every head attends
sharply to its own positions and a head or position mix-up moves outputs by O(1).
"""
from __future__ import annotations

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    from bit_expert_layer_gb300.build import build
    build()
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    from bit_expert_layer_gb300 import _abi
    return _abi


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def run_gpu(abi, q, k, v, lens):
    B, S_max = k.shape[0], k.shape[2]
    qd, kd, vd = _dev(q), _dev(k), _dev(v)
    out = torch.empty_like(qd)
    n = abi.gqa_decode_workspace_bytes(B)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    abi.gqa_decode_attention(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), lens, B, S_max, out.data_ptr(),
                             ws.data_ptr(), n)
    torch.cuda.synchronize()
    assert abi.gqa_decode_get_error(ws.data_ptr()) == abi.MOE_OK
    return out.cpu().numpy().view(np.uint16), (qd, kd, vd, out, ws, n)


def check(oracle, got_bits, q, k, v, lens):
    want, aw = oracle.gqa_decode(q, k, v, lens)
    got = synth.f32_from_bf16_bits(got_bits).astype(np.float64)
    assert np.all(np.isfinite(got))
    bound = 2.0 ** -8 * aw + 2.0 ** -8 * np.abs(want) + 1e-6
    err = np.abs(got - want)
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert np.all(err <= bound), (worst, err[worst], bound[worst])
    return float(np.max(err)), float(np.max(err / bound))


@pytest.mark.parametrize("B,S", [(8, 4096), (2, 32768)], ids=["ctx4K-B8", "ctx32K-B2"])
def test_gqa_contexts(oracle, lib, B, S):
    q, k, v, lens = synth.make_gqa(10 + B, B, S)
    got, _ = run_gpu(lib, q, k, v, lens)
    err, frac = check(oracle, got, q, k, v, lens)
    print(f"gqa B={B} S={S}: max err {err:.3e}, worst err/bound {frac:.3f}")


def test_gqa_ragged_lengths(oracle, lib):
    lens = [1, 2, 63, 64, 65, 127, 1000, 4097]
    q, k, v, _ = synth.make_gqa(21, len(lens), 4160, lens=lens)
    got, _ = run_gpu(lib, q, k, v, lens)
    check(oracle, got, q, k, v, np.asarray(lens, np.int32))


def test_gqa_largest_batch_and_single_position(oracle, lib):
    B = 64
    lens = [1 + (b * 37) % 300 for b in range(B)]
    q, k, v, _ = synth.make_gqa(22, B, 300, lens=lens)
    got, _ = run_gpu(lib, q, k, v, lens)
    check(oracle, got, q, k, v, np.asarray(lens, np.int32))
    # one cached position: the output is that position's value row, rounded to bf16
    q1, k1, v1, _ = synth.make_gqa(23, 3, 9, lens=[1, 1, 1], needles=0)
    got1, _ = run_gpu(lib, q1, k1, v1, [1, 1, 1])
    for b in range(3):
        for h in range(16):
            assert np.array_equal(got1[b, h], v1[b, h // 8, 0])


def test_gqa_rows_past_length_not_read_into_result(oracle, lib):
    lens = [100, 3000]
    q, k, v, _ = synth.make_gqa(24, 2, 3072, lens=lens)
    got, _ = run_gpu(lib, q, k, v, lens)
    k2, v2 = k.copy(), v.copy()
    k2[0, :, 100:] = synth.bf16_bits_from_f32(np.full((2, 2972, 128), 40.0, np.float32))
    v2[0, :, 100:] = synth.bf16_bits_from_f32(np.full((2, 2972, 128), 1e4, np.float32))
    got2, _ = run_gpu(lib, q, k2, v2, lens)
    assert np.array_equal(got, got2)


def test_gqa_deterministic_and_workspace_reusable(lib):
    lens = [5000, 777, 64]
    q, k, v, _ = synth.make_gqa(25, 3, 5000, lens=lens)
    a, (qd, kd, vd, out, ws, n) = run_gpu(lib, q, k, v, lens)
    for _ in range(3):      # the same workspace again: its tickets were left at zero
        lib.gqa_decode_attention(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), lens, 3, 5000, out.data_ptr(),
                                 ws.data_ptr(), n)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy().view(np.uint16), a)
    assert lib.gqa_decode_get_error(ws.data_ptr()) == lib.MOE_OK
