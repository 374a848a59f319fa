"""moe_decode_forward_static: the decode forward for callers that cannot allocate
device memory (a plug-in whose host owns all device memory and gives out none, or a
decode loop that must never reach cudaMalloc).  Its scratch is a fixed array inside
the library instead of a caller workspace.  Checked through the C ABI against the
regular entry point (moe_forward / moe_forward_residual on a layer with a workspace),
with the output tolerance of the other parity tests, and against the CPU oracle, on two
calls in a row so the second call starts from the array the first one left behind; the
array's own error word (moe_decode_static_get_error) must stay clear.

This file is named to be collected last.
"""
from __future__ import annotations

import numpy as np
import pytest

import synth
from parity import check_output, check_routing

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

TOL = 1e-2   # max |new - regular| <= TOL * max |regular|, as in the oracle parity tests


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _host(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _close(a, b):
    af, bf = a.float(), b.float()
    assert torch.isfinite(af).all()
    err = (af - bf).abs().max().item()
    assert err <= TOL * bf.abs().max().item(), err


@pytest.mark.parametrize("stacked", [False, True])
def test_static_decode_matches_regular_entry(oracle, stacked):
    from bit_expert_layer_gb300 import _abi
    from bit_expert_layer_gb300 import layer as ml
    from bit_expert_layer_gb300.build import build
    build()
    host = synth.stack_layer(3) if stacked else synth.make_layer(0)
    w = ml.DeviceWeights(host)
    regular = ml.MoELayer(w, max_tokens=16)
    cw = w.c()
    for T in (1, 8, 5):
        x_np = synth.make_x(30 + T, T)
        x = _dev(x_np)
        ref = regular.forward(x, residual=stacked)
        outs = []
        for _ in range(2):                      # two calls in a row
            out = torch.empty_like(x)
            _abi.moe_decode_forward_static(cw, x.data_ptr(), T, out.data_ptr(), stacked)
            outs.append(out)
        r = regular.route(x)
        torch.cuda.synchronize()
        assert regular.get_error() == 0
        assert _abi.moe_decode_static_get_error() == _abi.MOE_OK
        rep, alt = check_routing(oracle, host, x_np, r["idx"].cpu().numpy(), r["w"].cpu().numpy())
        for out in outs:
            _close(out, ref)
            check_output(oracle, host, x_np, _host(out), residual=stacked, alt=alt, any_of=rep["near_sets"])


def test_static_decode_in_place_residual(oracle):
    """out == x with the residual: the kernel's last phase writes rows that other CTAs
    read as the layer input earlier in the same launch."""
    from bit_expert_layer_gb300 import _abi
    from bit_expert_layer_gb300 import layer as ml
    host = synth.stack_layer(4)
    w = ml.DeviceWeights(host)
    regular = ml.MoELayer(w, max_tokens=16)
    T = 8
    x_np = synth.make_x(48, T)
    ref = regular.forward(_dev(x_np), residual=True)
    x = _dev(x_np)
    _abi.moe_decode_forward_static(w.c(), x.data_ptr(), T, x.data_ptr(), True)
    r = regular.route(_dev(x_np))
    torch.cuda.synchronize()
    assert _abi.moe_decode_static_get_error() == _abi.MOE_OK
    _close(x, ref)
    rep, alt = check_routing(oracle, host, x_np, r["idx"].cpu().numpy(), r["w"].cpu().numpy())
    check_output(oracle, host, x_np, _host(x), residual=True, alt=alt, any_of=rep["near_sets"])


def test_static_decode_rejects_sizes_beyond_its_scratch():
    from bit_expert_layer_gb300 import _abi
    from bit_expert_layer_gb300 import layer as ml
    w = ml.DeviceWeights(synth.make_layer(0))
    x = _dev(synth.make_x(0, 9))
    out = torch.empty_like(x)
    for T in (0, 9):
        with pytest.raises(_abi.MoEError) as ei:
            _abi.moe_decode_forward_static(w.c(), x.data_ptr(), T, out.data_ptr())
        assert ei.value.status == _abi.MOE_ERR_INVALID_ARG
        assert "static scratch" in str(ei.value)
