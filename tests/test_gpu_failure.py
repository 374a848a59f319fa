"""The failure path of the bounded device waits, exercised on purpose without faulting or
hanging the GPU.

Every wait of a launch on another thread's work gives up after a time limit, records
MOE_ERR_TIMEOUT in the layer's error word and ends the launch early; copies and MMAs
already in flight still land and tensor memory is freed before each CTA exits.  Here the
limit is set to 1 ns (moe_set_wait_limit_ns), so the first wait that is not already
satisfied gives up.  The test asserts that the error is reported, and that the next call
on the same layer object, with the default limit restored, matches the oracle: the
aborted launch left no tensor memory allocated, no copy in flight and no hand-off state
that the next launch could misread.
"""
from __future__ import annotations

import numpy as np
import pytest

import synth
from parity import check_output, check_routing

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


@pytest.fixture(scope="module")
def layer0(lib):
    L = synth.make_layer(0)
    return L, lib.MoELayer(lib.DeviceWeights(L), max_tokens=320)


# A prefill of 300 tokens runs the kernels that wait (the cluster router's and the tcgen05
# GEMMs' mbarriers); up to 192 tokens the expert GEMMs are GEMVs on mma.sync that wait on
# nothing but their own CTA's barriers, and only the router would time out.
@pytest.mark.parametrize("T", [300, 1], ids=["prefill-T300", "decode-T1"])
def test_timeout_reported_then_next_call_correct(oracle, lib, layer0, T):
    from bit_expert_layer_gb300 import _abi
    L, layer = layer0
    x_np = synth.make_x(60 + T, T)
    x = to_dev(x_np)
    layer.forward(x)
    torch.cuda.synchronize()
    assert layer.get_error() == _abi.MOE_OK
    _abi.moe_set_wait_limit_ns(1)
    try:
        for _ in range(2):
            layer.forward(x)
        torch.cuda.synchronize()
    finally:
        _abi.moe_set_wait_limit_ns(0)
    assert layer.get_error() == _abi.MOE_ERR_TIMEOUT
    assert layer.get_error() == _abi.MOE_OK          # reading cleared it
    out = layer.forward(x)
    r = layer.route(x)
    torch.cuda.synchronize()
    assert layer.get_error() == _abi.MOE_OK
    rep, alt = check_routing(oracle, L, x_np, r["idx"].cpu().numpy(), r["w"].cpu().numpy())
    any_of = rep["near_sets"] if T <= 8 else None
    check_output(oracle, L, x_np, to_host(out), alt=alt, any_of=any_of)


def test_static_decode_timeout_reported_then_next_call_correct(oracle, lib, layer0):
    """The same for moe_decode_forward_static, whose error word lives in its own array."""
    from bit_expert_layer_gb300 import _abi
    L, layer = layer0
    cw = layer.weights.c()
    T = 4
    x_np = synth.make_x(77, T)
    x = to_dev(x_np)
    out = torch.empty_like(x)
    _abi.moe_decode_forward_static(cw, x.data_ptr(), T, out.data_ptr())
    torch.cuda.synchronize()
    assert _abi.moe_decode_static_get_error() == _abi.MOE_OK
    _abi.moe_set_wait_limit_ns(1)
    try:
        _abi.moe_decode_forward_static(cw, x.data_ptr(), T, out.data_ptr())
        torch.cuda.synchronize()
    finally:
        _abi.moe_set_wait_limit_ns(0)
    assert _abi.moe_decode_static_get_error() == _abi.MOE_ERR_TIMEOUT
    assert _abi.moe_decode_static_get_error() == _abi.MOE_OK
    out = torch.empty_like(x)
    _abi.moe_decode_forward_static(cw, x.data_ptr(), T, out.data_ptr())
    r = layer.route(x)
    torch.cuda.synchronize()
    assert _abi.moe_decode_static_get_error() == _abi.MOE_OK
    rep, alt = check_routing(oracle, L, x_np, r["idx"].cpu().numpy(), r["w"].cpu().numpy())
    check_output(oracle, L, x_np, to_host(out), alt=alt, any_of=rep["near_sets"])
