"""The stacked form of the layer on the GPU against the oracle: a single layer with its
input RMSNorm, and the full 40-layer stack (18.2 GB of 4-bit weights) at T=16384
prefill and T=8 / T=1 decode, in the launch configuration the benchmark times (one
shared workspace, in-place residual through moe_stack_forward).

The stack is checked teacher-forced, layer by layer: the layers are also run one at a
time through the device entry (whose final result must equal the stack entry's bit for
bit), and at every one of the 40 layers the oracle receives the GPU's own input to that
layer for a sample of tokens.  Each layer is then held to the single-layer bounds
(routing exact or a valid near-tie choice, output within 1e-2 of the oracle's largest
magnitude), so a routing choice that an earlier layer's rounding moved across a narrow
gap never carries into a later comparison.  A chained comparison (the oracle following
its own outputs through all 40 layers) stays as a secondary check.
"""
from __future__ import annotations

import numpy as np
import pytest

import synth
from parity import bf16_to_f64, check_output, check_routing

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    from bit_expert_layer_gb300.build import build
    build()
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    from bit_expert_layer_gb300 import layer
    return layer


def to_dev(x_np):
    return torch.from_numpy(np.ascontiguousarray(x_np).view(np.int16)).cuda().view(torch.bfloat16)


def to_host(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("T", [3, 40])
def test_layer_with_input_norm(oracle, lib, T):
    L = synth.stack_layer(5)
    layer = lib.MoELayer(lib.DeviceWeights(L), max_tokens=64)
    x_np = synth.make_x(21, T)
    x = to_dev(x_np)
    out = layer.forward(x, residual=True)
    r = layer.route(x)
    torch.cuda.synchronize()
    assert layer.get_error() == 0
    rep, alt = check_routing(oracle, L, x_np, r["idx"].cpu().numpy(), r["w"].cpu().numpy())
    check_output(oracle, L, x_np, to_host(out), residual=True, alt=alt)
    print(f"norm layer T={T}: {rep}")


def stack_tolerance(scale: float, n_layers: int) -> float:
    """Bound of the secondary, chained comparison after n layers.  Each layer's output is
    the layer tolerance (1e-2 of the scale) away at most, and the residual stream is
    rounded to bf16 once per layer: where the two sides' unrounded sums straddle a
    rounding boundary they land one bf16 unit apart, and such one-unit steps add up like
    a random walk over the layers, about sqrt(n) units of the largest magnitude."""
    ulp = 2.0 ** (np.floor(np.log2(scale)) - 7)
    return 1e-2 * scale + np.sqrt(n_layers) * ulp


def _stack_chain(oracle, hosts, x_np):
    cur = x_np.copy()
    keep = np.ones(x_np.shape[0], bool)
    for h in hosts:
        r = oracle.forward(h, cur, residual=True)
        keep &= r["gap"] > 1e-4
        cur = r["out"]
    return cur, keep


def _teacher_forced(oracle, lib, hosts, layers, x_np, sample, label):
    """Runs the layers one by one through the device entry on the whole input, keeps each
    layer's input, output and routing on the sampled tokens, and checks every layer
    against the oracle on the GPU's own input.  Returns the final device output (all
    tokens) and the per-layer (max error, scale) list."""
    cur = to_dev(x_np)
    per_layer = []
    near_total = flips_total = 0
    w_err = 0.0
    for l, (h, layer) in enumerate(zip(hosts, layers)):
        inp = to_host(cur)[sample]
        r = layer.route(cur)
        nxt = layer.forward(cur, residual=True)
        torch.cuda.synchronize()
        assert layer.get_error() == 0, f"{label} layer {l}: device error"
        idx = r["idx"].cpu().numpy()[sample]
        w = r["w"].cpu().numpy()[sample]
        out = to_host(nxt)[sample]
        rep, alt = check_routing(oracle, h, inp, idx, w)
        # decode: the router entry and the fused forward are different kernels
        any_of = rep["near_sets"] if x_np.shape[0] <= 8 else None
        err, scale = check_output(oracle, h, inp, out, residual=True, alt=alt, any_of=any_of)
        per_layer.append((err, scale))
        near_total += rep["near_ties"]
        flips_total += rep["flips"]
        w_err = max(w_err, rep["w_err"])
        cur = nxt
    worst = max(e / s for e, s in per_layer)
    print(f"{label}: {len(sample)} tokens x {len(hosts)} layers teacher-forced; near-ties {near_total}, "
          f"flips {flips_total}, max weight diff {w_err:.2e}, worst layer err/scale {worst:.3e}")
    print(f"{label} per-layer max err / scale: " +
          " ".join(f"{l}:{e:.3g}/{s:.3g}" for l, (e, s) in enumerate(per_layer)))
    return cur, per_layer


def test_short_prefill_stack_T1000(oracle, lib):
    """Four stacked layers at T=1000, the size where the router runs as four-CTA clusters
    and the small token blocks take the swapped down GEMM: the stack entry (each layer's
    combine writing the next layer's normalised input, its interleaved copy and its shared
    gate) equals the layer-by-layer computation bit for bit, and every layer follows the
    oracle on its own input (teacher-forced) for a sample of tokens."""
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(4) as ex:
        hosts = list(ex.map(lambda l: synth.stack_layer(l, threads=2), range(4)))
    T = 1000
    ws = lib.new_workspace(T)
    layers = [lib.MoELayer(lib.DeviceWeights(h), T, workspace=ws) for h in hosts]
    stack = lib.MoEStack(layers)
    x_np = synth.make_x(3, T)
    x = to_dev(x_np)
    stack.forward_(x)
    torch.cuda.synchronize()
    assert layers[0].get_error() == 0
    rng = np.random.default_rng(1000)
    sample = np.unique(np.concatenate([rng.choice(T, 40, replace=False), [0, T - 2, T - 1]]))
    final, _ = _teacher_forced(oracle, lib, hosts, layers, x_np, sample, "stack prefill T=1000")
    assert torch.equal(final.view(torch.int16), x.view(torch.int16))


@pytest.fixture(scope="module")
def stack40(lib):
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(4) as ex:
        hosts = list(ex.map(lambda l: synth.stack_layer(l, threads=2), range(40)))
    T = 16384
    ws = lib.new_workspace(T)
    layers = [lib.MoELayer(lib.DeviceWeights(h), T, workspace=ws) for h in hosts]
    return hosts, layers, lib.MoEStack(layers)


def test_full_stack_40_layers_prefill(oracle, lib, stack40):
    hosts, layers, stack = stack40
    T = 16384
    x_np = synth.make_x(0, T)
    x = to_dev(x_np)
    stack.forward_(x)
    torch.cuda.synchronize()
    assert layers[0].get_error() == 0
    got = to_host(x)
    assert np.all(np.isfinite(bf16_to_f64(got)))

    # teacher-forced, every layer, on 72 tokens (64 random, the first and last 4)
    rng = np.random.default_rng(40)
    sample = np.unique(np.concatenate([rng.choice(T, 64, replace=False), [0, 1, 2, 3, T - 4, T - 3, T - 2, T - 1]]))
    final, per_layer = _teacher_forced(oracle, lib, hosts, layers, x_np, sample, "stack prefill T=16384")
    # the stack entry is the layer-by-layer computation, bit for bit
    assert torch.equal(final.view(torch.int16), x.view(torch.int16))

    # secondary: the oracle chained on its own outputs through all 40 layers
    sample2 = np.unique(np.concatenate([rng.choice(T, 110, replace=False), [0, T - 1]]))
    ref, keep = _stack_chain(oracle, hosts, x_np[sample2])
    # about 3% of tokens sit within 1e-4 of a routing tie at each layer, so roughly
    # 0.97^40 = 30% of tokens stay comparable through all 40 layers
    assert keep.sum() >= 12, keep.sum()
    ref_v = bf16_to_f64(ref[keep])
    err = np.max(np.abs(bf16_to_f64(got[sample2][keep]) - ref_v))
    scale = np.max(np.abs(ref_v))
    bound = stack_tolerance(scale, len(hosts))
    assert err <= bound, (err, scale)
    ulp = 2.0 ** (np.floor(np.log2(scale)) - 7)
    print(f"stack prefill chained: {int(keep.sum())}/{len(sample2)} tokens compared, max err {err:.3e} "
          f"= {err / ulp:.2f} bf16 units at scale {scale:.3e}; 1e-2 * scale = {1e-2 * scale:.3e}, "
          f"sqrt(40) units = {np.sqrt(40) * ulp:.3e}")

    # the first layer alone, routing tables exact on the full T
    r = layers[0].route(to_dev(x_np))
    sub = np.arange(0, T, 64)
    idx = r["idx"].cpu().numpy()
    check_routing(oracle, hosts[0], x_np[sub], idx[sub], r["w"].cpu().numpy()[sub])
    counts = r["counts"].cpu().numpy()
    assert counts.sum() == 8 * T and np.array_equal(counts, np.bincount(idx.reshape(-1), minlength=256))


@pytest.mark.parametrize("T", [8, 1])
def test_full_stack_40_layers_decode(oracle, lib, stack40, T):
    """The fused decode kernel (one launch runs all 40 layers) against the layers run one
    at a time (bit for bit), and every layer teacher-forced against the oracle; no token
    is left out."""
    hosts, layers, stack = stack40
    x_np = synth.make_x(1, T)
    x = to_dev(x_np)
    stack.forward_(x)
    torch.cuda.synchronize()
    assert layers[0].get_error() == 0
    final, _ = _teacher_forced(oracle, lib, hosts, layers, x_np, np.arange(T), f"stack decode T={T}")
    assert torch.equal(final.view(torch.int16), x.view(torch.int16))
