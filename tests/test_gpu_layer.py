"""Parity of the CUDA layer (through the C ABI) with the CPU oracle, on the GPU.

Workloads are the seeded synthetic layer at its real shapes: T=32 (the reference
configuration), T=1 and 8 (decode), T=512 uniform, T=4096 with the skewed log-Zipf
router bias, a sweep of ragged T, all tokens forced onto one expert set, exact routing
ties, in-place residual, determinism, a short stack, and argument errors.  The rules are in
tests/parity.py.
"""
from __future__ import annotations

import numpy as np
import pytest

import synth
from parity import bf16_to_f64, check_output, check_routing, check_tables

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


@pytest.fixture(scope="module")
def host0():
    return synth.make_layer(0)


@pytest.fixture(scope="module")
def dev0(lib, host0):
    w = lib.DeviceWeights(host0)
    return lib.MoELayer(w, max_tokens=4096)


def to_dev(x_np):
    return torch.from_numpy(np.ascontiguousarray(x_np).view(np.int16)).cuda().view(torch.bfloat16)


def to_host(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run(layer, x_np, residual=False):
    x = to_dev(x_np)
    out = layer.forward(x, residual=residual)
    r = layer.route(x)
    torch.cuda.synchronize()
    assert layer.get_error() == 0
    return to_host(out), {k: v.cpu().numpy() for k, v in r.items()}


def full_check(oracle, L, layer, x, residual=False, sample=None):
    out, r = run(layer, x, residual)
    rep, alt = check_routing(oracle, L, x, r["idx"], r["w"])
    check_tables(r["idx"], r["counts"], r["offsets"], r["perm"])
    # at T <= 8 the router entry and the fused decode forward are different kernels
    any_of = rep["near_sets"] if x.shape[0] <= 8 else None
    err, scale = check_output(oracle, L, x, out, tokens=sample, residual=residual, alt=alt, any_of=any_of)
    return rep, err, scale


def test_reference_T32(oracle, host0, dev0):
    x = synth.make_x(0, 32)
    rep, err, scale = full_check(oracle, host0, dev0, x)
    print(f"T=32 {rep} max_err={err:.3e} scale={scale:.3e}")


@pytest.mark.parametrize("T", [1, 8])
def test_decode(oracle, host0, dev0, T):
    x = synth.make_x(0, T)
    rep, err, scale = full_check(oracle, host0, dev0, x)
    print(f"T={T} {rep} max_err={err:.3e} scale={scale:.3e}")


@pytest.mark.parametrize("T", [2, 3, 7, 9, 31, 33, 63, 64, 65, 127, 128, 129, 191, 192, 193])
def test_ragged_sweep(oracle, host0, dev0, T):
    """Both sides of the token counts where the path changes: decode (T <= 8), the GEMV
    expert kernels (T <= 192) and the tcgen05 ones."""
    x = synth.make_x(100 + T, T)
    full_check(oracle, host0, dev0, x)


def test_prefill_T512(oracle, host0, dev0):
    x = synth.make_x(0, 512)
    rep, err, scale = full_check(oracle, host0, dev0, x)   # every token
    print(f"T=512 {rep} max_err={err:.3e} scale={scale:.3e}")


def test_skewed_T4096(oracle, lib):
    L = synth.make_layer(0, skew=True)
    layer = lib.MoELayer(lib.DeviceWeights(L), max_tokens=4096)
    x = synth.make_x(0, 4096)
    out, r = run(layer, x)
    rep, alt = check_routing(oracle, L, x, r["idx"], r["w"])
    check_tables(r["idx"], r["counts"], r["offsets"], r["perm"])
    counts = r["counts"]
    heavy = np.argsort(-counts)[:3]
    rng = np.random.default_rng(4096)
    sample = set(rng.choice(4096, 512, replace=False).tolist()) | set(range(4088, 4096))
    for e in heavy:   # tokens from the heaviest experts' last (ragged) tiles
        slots = r["perm"][r["offsets"][e]:r["offsets"][e + 1]]
        sample |= set((slots[-4:] // 8).tolist())
    light = [e for e in range(256) if 0 < counts[e] <= 2][:4]
    for e in light:
        slots = r["perm"][r["offsets"][e]:r["offsets"][e + 1]]
        sample |= set((slots // 8).tolist())
    sample = np.array(sorted(sample))
    err, scale = check_output(oracle, L, x, out, tokens=sample, alt=alt)
    print(f"T=4096 skew {rep} touched={int((counts > 0).sum())} top={sorted(counts)[-3:]} "
          f"max_err={err:.3e} scale={scale:.3e}")


@pytest.mark.parametrize("T", [33, 64, 129, 192, 193, 384, 385, 600, 1024, 1025])
def test_all_tokens_on_one_expert_set(oracle, lib, T):
    """Every token on the same 8 experts (and the shared one), so each of them holds T
    rows: in the GEMV kernels (T <= 192) blocks of more rows than one CTA's chunk of 32,
    up to six chunks; in the tcgen05 kernels a big block of 193 rows, a full block plus
    a partial block of 128 and 129 rows (the largest small block, run with the operands
    swapped up to T = 1024, and the smallest big one), and T on both sides of the token
    count above which the small blocks stay in the ordinary down GEMM."""
    L = synth.make_layer(7)
    chosen = [3, 17, 40, 77, 100, 150, 200, 255]
    bias = np.zeros(256, np.float32)
    bias[chosen] = 20.0
    L.router_bias = bias
    layer = lib.MoELayer(lib.DeviceWeights(L), max_tokens=1100)
    x = synth.make_x(7, T)
    out, r = run(layer, x)
    assert set(np.unique(r["idx"]).tolist()) == set(chosen)
    assert all(r["counts"][e] == T for e in chosen)
    rep, alt = check_routing(oracle, L, x, r["idx"], r["w"])
    check_output(oracle, L, x, out, alt=alt)   # every token


@pytest.mark.parametrize("T", [1, 8, 40])
def test_exact_ties_lowest_index(oracle, lib, T):
    """Every router logit equal (zero router matrix, no bias): each token takes experts
    0..7, each with weight exactly 1/8, on the decode path (T <= 8) and the prefill path;
    the output follows the oracle, which breaks the tie the same way."""
    L = synth.make_layer(11)
    L.router_w = np.zeros_like(L.router_w)
    layer = lib.MoELayer(lib.DeviceWeights(L), max_tokens=64)
    x = synth.make_x(11, T)
    out, r = run(layer, x)
    assert (r["idx"] == np.arange(8)[None, :]).all()
    assert (r["w"] == np.float32(0.125)).all()
    assert (r["counts"][:8] == T).all() and (r["counts"][8:256] == 0).all()
    check_output(oracle, L, x, out)


@pytest.mark.parametrize("T", [4095, 4096, 4097])
def test_router_kernel_switch(oracle, lib, T):
    """Up to 4096 tokens the router runs as four-CTA clusters that split K and exchange
    partial logits; above, as two-CTA clusters (up to 8192; beyond, one CTA per 128 tokens
    over the whole K, covered by test_prefill_T8192 at T = 8200).  Both sides of the first
    switch, with ragged last blocks: the routing of every token, the tables, and the
    output of a sample that includes the last block."""
    L = synth.make_layer(13)
    layer = lib.MoELayer(lib.DeviceWeights(L), max_tokens=4100)
    x = synth.make_x(13, T)
    out, r = run(layer, x)
    rep, alt = check_routing(oracle, L, x, r["idx"], r["w"])
    check_tables(r["idx"], r["counts"], r["offsets"], r["perm"])
    rng = np.random.default_rng(T)
    sample = np.array(sorted(set(rng.choice(T, 48, replace=False).tolist()) | set(range(T - 8, T))))
    err, scale = check_output(oracle, L, x, out, tokens=sample, alt=alt)
    print(f"T={T} {rep} max_err={err:.3e} scale={scale:.3e}")


@pytest.mark.parametrize("T", [8192, 8200])
def test_prefill_T8192(oracle, lib, T):
    """A larger prefill (about 256 rows per expert: full token blocks and a partial one for
    most experts) on both sides of the switch from the two-CTA cluster router (T = 8192)
    to the whole-K one (T = 8200): the routing of every token and the output of a sample
    that includes the partial blocks of the fullest experts and the last tokens."""
    L = synth.make_layer(17)
    layer = lib.MoELayer(lib.DeviceWeights(L), max_tokens=8200)
    x = synth.make_x(17, T)
    out, r = run(layer, x)
    rep, alt = check_routing(oracle, L, x, r["idx"], r["w"])
    check_tables(r["idx"], r["counts"], r["offsets"], r["perm"])
    counts = r["counts"]
    rng = np.random.default_rng(T)
    sample = set(rng.choice(T, 48, replace=False).tolist()) | set(range(T - 4, T))
    for e in np.argsort(counts)[-2:]:   # the last rows of the fullest experts (a partial block)
        slots = r["perm"][r["offsets"][e]:r["offsets"][e + 1]]
        sample |= set((slots[-3:] // 8).tolist())
    err, scale = check_output(oracle, L, x, out, tokens=np.array(sorted(sample)), alt=alt)
    print(f"T={T} near_ties={rep['near_ties']} flips={rep['flips']} max_err={err:.3e} scale={scale:.3e}")


def test_max_tokens(oracle, lib):
    """The largest token count a layer accepts (65536): router blocks in several waves,
    the scan's longest histogram walk, schedules near their capacity (about 68 gate/up and
    270 down tiles per CTA).  The tables over every slot, the routing of a sample and the
    output of a sample that includes the last tokens."""
    T = 65536
    L = synth.make_layer(19)
    layer = lib.MoELayer(lib.DeviceWeights(L), max_tokens=T)
    x = synth.make_x(19, T)
    out, r = run(layer, x)
    check_tables(r["idx"], r["counts"], r["offsets"], r["perm"])
    rng = np.random.default_rng(T)
    sub = np.unique(np.concatenate([rng.choice(T, 512, replace=False), np.arange(T - 8, T)]))
    rep, alt = check_routing(oracle, L, x[sub], r["idx"][sub], r["w"][sub])
    alt = {int(sub[i]): v for i, v in alt.items()}
    # output tokens from the routing sample, so that a near-tie choice is known for each
    tok = np.unique(np.concatenate([rng.choice(sub, 24, replace=False), np.arange(T - 4, T)]))
    err, scale = check_output(oracle, L, x, out, tokens=tok, alt=alt)
    print(f"T={T} near_ties={rep['near_ties']} flips={rep['flips']} max_err={err:.3e} scale={scale:.3e}")


@pytest.mark.parametrize("T", [4100, 8200])
def test_exact_ties_large_T(oracle, lib, T):
    """Exact ties (zero router matrix) with the two-CTA cluster router (T = 4100) and the
    whole-K router (T = 8200): experts 0..7 with weight 1/8 for every token."""
    L = synth.make_layer(11)
    L.router_w = np.zeros_like(L.router_w)
    layer = lib.MoELayer(lib.DeviceWeights(L), max_tokens=T)
    x = synth.make_x(11, T)
    out, r = run(layer, x)
    assert (r["idx"] == np.arange(8)[None, :]).all()
    assert (r["w"] == np.float32(0.125)).all()
    assert (r["counts"][:8] == T).all() and (r["counts"][8:256] == 0).all()
    check_output(oracle, L, x, out, tokens=np.array([0, 1, 2047, 4095, 4096, T - 1]))


@pytest.mark.parametrize("T", [5, 40])
def test_residual_in_place(oracle, host0, dev0, T):
    x_np = synth.make_x(9, T)
    x = to_dev(x_np)
    dev0.forward(x, out=x, residual=True)
    torch.cuda.synchronize()
    assert dev0.get_error() == 0
    out = to_host(x)
    r = dev0.route(to_dev(x_np))
    rep, alt = check_routing(oracle, host0, x_np, r["idx"].cpu().numpy(), r["w"].cpu().numpy())
    any_of = rep["near_sets"] if T <= 8 else None
    check_output(oracle, host0, x_np, out, residual=True, alt=alt, any_of=any_of)


def test_deterministic(host0, dev0):
    for T in (300, 6):
        x = to_dev(synth.make_x(11, T))
        a = dev0.forward(x)
        b = dev0.forward(x)
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_short_stack(oracle, lib):
    """The stack entry against the layers run one by one (bit-identical), and each layer
    teacher-forced against the oracle: the oracle gets the GPU's own input of that layer,
    so a routing choice that an earlier layer's rounding moved across a narrow gap does
    not carry into later layers."""
    hosts = [synth.stack_layer(l) for l in range(3)]
    ws = lib.new_workspace(64)
    layers = [lib.MoELayer(lib.DeviceWeights(h), max_tokens=64, workspace=ws) for h in hosts]
    stack = lib.MoEStack(layers)
    for T in (24, 5):
        x_np = synth.make_x(12, T)
        x = to_dev(x_np)
        stack.forward_(x)
        torch.cuda.synchronize()
        got = to_host(x)
        cur = x_np.copy()
        for h, layer in zip(hosts, layers):
            inp = cur
            cur = to_host(layer.forward(to_dev(inp), residual=True))
            torch.cuda.synchronize()
            assert layer.get_error() == 0
            r = oracle.forward(h, inp, residual=True)
            keep = r["gap"] > 1e-4
            # about 2% of tokens sit within 1e-4 of a tie at each layer of this router
            assert keep.sum() >= T // 2
            ref = bf16_to_f64(r["out"][keep])
            err = np.max(np.abs(bf16_to_f64(cur[keep]) - ref))
            assert err <= 1e-2 * np.max(np.abs(ref)), err
        assert np.array_equal(cur, got)
        # the host-memory entry gives the same bytes as the device entry
        xh = torch.from_numpy(x_np.view(np.int16)).pin_memory()
        oh = torch.empty_like(xh).pin_memory()
        stack.forward_host(xh, oh)
        torch.cuda.synchronize()
        assert np.array_equal(oh.numpy().view(np.uint16), got)


def test_argument_errors(lib, dev0):
    from bit_expert_layer_gb300 import _abi
    x = to_dev(synth.make_x(0, 16))
    out = torch.empty_like(x)
    with pytest.raises(_abi.MoEError) as ei:
        _abi.moe_forward(dev0.handle, x.data_ptr(), 0, out.data_ptr())
    assert ei.value.status == _abi.MOE_ERR_INVALID_ARG
    with pytest.raises(_abi.MoEError) as ei:
        _abi.moe_forward(dev0.handle, x.data_ptr(), 5000, out.data_ptr())
    assert ei.value.status == _abi.MOE_ERR_INVALID_ARG
    with pytest.raises(_abi.MoEError) as ei:
        _abi.moe_forward(dev0.handle, x.data_ptr() + 2, 8, out.data_ptr())
    assert ei.value.status == _abi.MOE_ERR_ALIGNMENT
    with pytest.raises(_abi.MoEError) as ei:
        _abi.moe_forward(dev0.handle, x.data_ptr(), 16, x.data_ptr() + 4096)
    assert ei.value.status == _abi.MOE_ERR_INVALID_ARG
    with pytest.raises(_abi.MoEError) as ei:
        _abi.moe_forward_residual(dev0.handle, x.data_ptr(), 16, x.data_ptr() + 4096)
    assert ei.value.status == _abi.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert dev0.get_error() == 0
