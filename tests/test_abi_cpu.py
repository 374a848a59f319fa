"""The C-ABI library loads on a machine without a GPU and exports every entry point
that include/moe_layer.h and include/gqa_decode.h declare; host-side validation runs
before any CUDA call."""
import ctypes as C

import pytest

from bit_expert_layer_gb300 import _abi
from bit_expert_layer_gb300.build import build


@pytest.fixture(scope="module")
def lib():
    build()
    return _abi.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _abi.declared_functions()
    assert "moe_forward" in names and "moe_route" in names and "moe_layer_create" in names
    assert "gqa_decode_attention" in names and "moe_set_wait_limit_ns" in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def _cfg(**kw):
    base = dict(hidden=2048, n_experts=256, top_k=8, inter=512, shared_inter=512, group_size=64, bits=4,
                max_tokens=1024)
    base.update(kw)
    return _abi.MoeConfig(*base.values())


def test_workspace_bytes(lib):
    a = _abi.moe_workspace_bytes(_cfg(max_tokens=1024))
    b = _abi.moe_workspace_bytes(_cfg(max_tokens=2048))
    assert a > 0 and b > a and a % 256 == 0
    # the big buffers per token: h and y in 9 rows (9 * (1024 + 4096) bytes), the
    # interleaved copy of x, the I/O and norm buffers (3 * 4096 bytes)
    assert b - a >= 1024 * (9 * (1024 + 4096) + 3 * 4096)
    assert _abi.moe_workspace_bytes(_cfg(bits=8)) == 0


@pytest.mark.parametrize("bad", [dict(hidden=4096), dict(n_experts=128), dict(top_k=4), dict(inter=768),
                                 dict(shared_inter=1024), dict(group_size=32), dict(bits=8), dict(max_tokens=0),
                                 dict(max_tokens=1 << 20)])
def test_create_refuses_other_layouts(lib, bad):
    """Like Lily's load-time refusal of any other checkpoint layout."""
    h = C.c_void_p()
    w = _abi.MoeWeights()
    st = lib.moe_layer_create(C.byref(_cfg(**bad)), C.byref(w), None, 0, C.byref(h))
    assert st == _abi.MOE_ERR_UNSUPPORTED and not h.value


def test_create_argument_checks(lib):
    h = C.c_void_p()
    w = _abi.MoeWeights()
    assert lib.moe_layer_create(C.byref(_cfg()), C.byref(w), None, 0, C.byref(h)) == _abi.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_create(None, C.byref(w), None, 0, C.byref(h)) == _abi.MOE_ERR_INVALID_ARG
    fake = 1 << 40
    q = _abi.MoeQMat(fake, fake, fake)
    w = _abi.MoeWeights(q, q, q, q, q, q, fake, None, fake, None)
    assert lib.moe_layer_create(C.byref(_cfg()), C.byref(w), fake, 16, C.byref(h)) == _abi.MOE_ERR_WORKSPACE
    assert lib.moe_layer_create(C.byref(_cfg()), C.byref(w), fake + 16, 1 << 40,
                                C.byref(h)) == _abi.MOE_ERR_ALIGNMENT
    qm = _abi.MoeQMat(fake + 4, fake, fake)
    w2 = _abi.MoeWeights(qm, q, q, q, q, q, fake, None, fake, None)
    assert lib.moe_layer_create(C.byref(_cfg()), C.byref(w2), fake, 1 << 40, C.byref(h)) == _abi.MOE_ERR_ALIGNMENT
    w2 = _abi.MoeWeights(q, q, q, q, q, q, fake, None, fake, fake + 2)
    assert lib.moe_layer_create(C.byref(_cfg()), C.byref(w2), fake, 1 << 40, C.byref(h)) == _abi.MOE_ERR_ALIGNMENT


def test_call_argument_checks_need_no_gpu(lib):
    assert lib.moe_forward(None, None, 1, None, None) == _abi.MOE_ERR_INVALID_ARG
    assert lib.moe_route(None, None, 1, None, None, None, None, None, None) == _abi.MOE_ERR_INVALID_ARG
    assert lib.moe_stack_forward(None, 0, None, 1, None) == _abi.MOE_ERR_INVALID_ARG
    assert lib.moe_forward_launches(None, 1) == 0
    assert lib.moe_stack_forward_launches(None, 1, 1) == 0
    null_layers = (C.c_void_p * 2)(None, None)
    assert lib.moe_stack_forward_launches(null_layers, 2, 1) == 0


def test_status_strings(lib):
    for code in _abi.STATUS:
        assert _abi.moe_status_string(code)
    assert _abi.moe_status_string(99) == "unknown status"


def test_gqa_host_checks(lib):
    """Sizes and pointers are checked on the host before anything reaches the device."""
    assert _abi.gqa_decode_workspace_bytes(0) == 0 and _abi.gqa_decode_workspace_bytes(65) == 0
    a, b = _abi.gqa_decode_workspace_bytes(1), _abi.gqa_decode_workspace_bytes(8)
    assert a > 0 and b > a
    fake = 1 << 20   # never dereferenced: every call below fails its host check first
    for args, st in [((fake, fake, fake, [4], 0, 8, fake, fake, b), _abi.MOE_ERR_INVALID_ARG),
                     ((fake, fake, fake, [9], 1, 8, fake, fake, b), _abi.MOE_ERR_INVALID_ARG),
                     ((fake, fake, fake, [0], 1, 8, fake, fake, b), _abi.MOE_ERR_INVALID_ARG),
                     ((fake + 2, fake, fake, [4], 1, 8, fake, fake, b), _abi.MOE_ERR_ALIGNMENT),
                     ((fake, fake, fake, [4], 1, 8, fake, fake + 16, b), _abi.MOE_ERR_ALIGNMENT),
                     ((fake, fake, fake, [4], 1, 8, fake, fake, a - 1), _abi.MOE_ERR_WORKSPACE)]:
        with pytest.raises(_abi.MoEError) as ei:
            _abi.gqa_decode_attention(*args)
        assert ei.value.status == st, (args, ei.value.status)
