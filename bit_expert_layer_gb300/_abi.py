"""ctypes binding of the C ABI declared in ``include/moe_layer.h``.

Argument marshalling only: every step of the layer runs in the CUDA library.  The
functions keep the C names and take raw integers for device pointers and streams.
Loading fails loudly if the library has not been built; nothing here falls back to
any other implementation.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_layer.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "moe_layer.h")
HEADERS = [HEADER, os.path.join(os.path.dirname(_PKG), "include", "gqa_decode.h")]

STATUS = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_ALIGNMENT",
    4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_DEVICE_BOUNDS", 7: "MOE_ERR_WORKSPACE",
}
MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_ALIGNMENT = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_BOUNDS, MOE_ERR_WORKSPACE = 4, 5, 6, 7


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        detail = ""
        try:
            d = lib().moe_last_error_detail()
            detail = d.decode() if d else ""
        except Exception:  # pragma: no cover - the library itself failed to load
            pass
        super().__init__(f"{where}: {STATUS.get(status, status)}" + (f" ({detail})" if detail else ""))


class MoeConfig(C.Structure):
    _fields_ = [(n, C.c_int) for n in
                ("hidden", "n_experts", "top_k", "inter", "shared_inter", "group_size", "bits", "max_tokens")]


class MoeQMat(C.Structure):
    _fields_ = [("q", C.c_void_p), ("scales", C.c_void_p), ("biases", C.c_void_p)]


class MoeWeights(C.Structure):
    _fields_ = [("gate", MoeQMat), ("up", MoeQMat), ("down", MoeQMat),
                ("sh_gate", MoeQMat), ("sh_up", MoeQMat), ("sh_down", MoeQMat),
                ("router_w", C.c_void_p), ("router_bias", C.c_void_p), ("shared_gate_w", C.c_void_p),
                ("norm_w", C.c_void_p)]


_lib = None


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run bit_expert_layer_gb300.build.build()")
        L = C.CDLL(LIB_PATH)
        P, I, S = C.c_void_p, C.c_int, C.c_int
        L.moe_workspace_bytes.argtypes = [C.POINTER(MoeConfig)]
        L.moe_workspace_bytes.restype = C.c_size_t
        L.moe_layer_create.argtypes = [C.POINTER(MoeConfig), C.POINTER(MoeWeights), P, C.c_size_t, C.POINTER(P)]
        L.moe_layer_create.restype = S
        L.moe_route.argtypes = [P, P, I, P, P, P, P, P, P]
        L.moe_route.restype = S
        L.moe_forward.argtypes = [P, P, I, P, P]
        L.moe_forward.restype = S
        L.moe_forward_residual.argtypes = [P, P, I, P, P]
        L.moe_forward_residual.restype = S
        L.moe_stack_forward.argtypes = [P, I, P, I, P]
        L.moe_stack_forward.restype = S
        L.moe_stack_forward_host.argtypes = [P, I, P, I, P, P]
        L.moe_stack_forward_host.restype = S
        L.moe_forward_launches.argtypes = [P, I]
        L.moe_forward_launches.restype = I
        L.moe_stack_forward_launches.argtypes = [P, I, I]
        L.moe_stack_forward_launches.restype = I
        L.moe_layer_get_error.argtypes = [P]
        L.moe_layer_get_error.restype = S
        L.moe_layer_destroy.argtypes = [P]
        L.moe_layer_destroy.restype = None
        L.moe_status_string.argtypes = [S]
        L.moe_status_string.restype = C.c_char_p
        L.moe_last_error_detail.argtypes = []
        L.moe_last_error_detail.restype = C.c_char_p
        L.moe_decode_forward_static.argtypes = [C.POINTER(MoeWeights), P, I, P, I, P]
        L.moe_decode_forward_static.restype = S
        L.moe_decode_static_get_error.argtypes = []
        L.moe_decode_static_get_error.restype = S
        L.gqa_decode_workspace_bytes.argtypes = [I]
        L.gqa_decode_workspace_bytes.restype = C.c_size_t
        L.gqa_decode_attention.argtypes = [P, P, P, P, I, I, P, P, C.c_size_t, P]
        L.gqa_decode_attention.restype = S
        L.gqa_decode_get_error.argtypes = [P]
        L.gqa_decode_get_error.restype = S
        L.moe_decode_trace.argtypes = [P, P, C.c_size_t]
        L.moe_decode_trace.restype = S
        L.moe_set_wait_limit_ns.argtypes = [C.c_ulonglong]
        L.moe_set_wait_limit_ns.restype = None
        L.moe_pipeline_counters.argtypes = [P, P]
        L.moe_pipeline_counters.restype = S
        L.moe_profiler_enable.argtypes = [I]
        L.moe_profiler_enable.restype = None
        L.moe_profiler_read.argtypes = [P, P, P, I]
        L.moe_profiler_read.restype = I
        _lib = L
    return _lib


def _check(status: int, where: str) -> int:
    if status != MOE_OK:
        raise MoEError(status, where)
    return status


# --- same names as the C entry points -------------------------------------------------

def moe_workspace_bytes(cfg: MoeConfig) -> int:
    return int(lib().moe_workspace_bytes(C.byref(cfg)))


def moe_layer_create(cfg: MoeConfig, weights: MoeWeights, workspace: int, workspace_bytes: int) -> int:
    h = C.c_void_p()
    _check(lib().moe_layer_create(C.byref(cfg), C.byref(weights), C.c_void_p(workspace), workspace_bytes,
                                  C.byref(h)), "moe_layer_create")
    return h.value


def moe_route(layer: int, x: int, T: int, topk_idx: int = 0, topk_w: int = 0, counts: int = 0,
              offsets: int = 0, perm: int = 0, stream: int = 0) -> None:
    _check(lib().moe_route(layer, x, T, topk_idx or None, topk_w or None, counts or None, offsets or None,
                           perm or None, stream or None), "moe_route")


def moe_forward(layer: int, x: int, T: int, out: int, stream: int = 0) -> None:
    _check(lib().moe_forward(layer, x, T, out, stream or None), "moe_forward")


def moe_forward_residual(layer: int, x: int, T: int, out: int, stream: int = 0) -> None:
    _check(lib().moe_forward_residual(layer, x, T, out, stream or None), "moe_forward_residual")


def _handles(layers):
    arr = (C.c_void_p * len(layers))(*layers)
    return arr


def moe_stack_forward(layers, x_io: int, T: int, stream: int = 0) -> None:
    arr = _handles(layers)
    _check(lib().moe_stack_forward(C.cast(arr, C.c_void_p), len(layers), x_io, T, stream or None),
           "moe_stack_forward")


def moe_stack_forward_host(layers, x_host: int, T: int, out_host: int, stream: int = 0) -> None:
    arr = _handles(layers)
    _check(lib().moe_stack_forward_host(C.cast(arr, C.c_void_p), len(layers), x_host, T, out_host,
                                        stream or None), "moe_stack_forward_host")


def moe_forward_launches(layer: int, T: int) -> int:
    return int(lib().moe_forward_launches(layer, T))


def moe_stack_forward_launches(layers, T: int) -> int:
    arr = (C.c_void_p * len(layers))(*layers)
    return int(lib().moe_stack_forward_launches(arr, len(layers), T))


def moe_layer_get_error(layer: int) -> int:
    return int(lib().moe_layer_get_error(layer))


def moe_layer_destroy(layer: int) -> None:
    lib().moe_layer_destroy(layer)


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def moe_decode_forward_static(weights: MoeWeights, x: int, T: int, out: int, residual: bool = False,
                              stream: int = 0) -> None:
    _check(lib().moe_decode_forward_static(C.byref(weights), x, T, out, 1 if residual else 0, stream or None),
           "moe_decode_forward_static")


def moe_decode_static_get_error() -> int:
    return int(lib().moe_decode_static_get_error())


DEC_TRACE_CTAS, DEC_TRACE_STAMPS = 256, 16


def moe_decode_trace(layer: int, n_layers: int):
    """Phase timestamps of the last decode launch (MOE_DECODE_TRACE=1), as a uint64 array
    [n_layers][256 CTAs][16 stamps]."""
    import numpy as np
    n = n_layers * DEC_TRACE_CTAS * DEC_TRACE_STAMPS
    buf = np.zeros(n, np.uint64)
    _check(lib().moe_decode_trace(layer, buf.ctypes.data_as(C.c_void_p), n), "moe_decode_trace")
    return buf.reshape(n_layers, DEC_TRACE_CTAS, DEC_TRACE_STAMPS)


def moe_set_wait_limit_ns(ns: int) -> None:
    lib().moe_set_wait_limit_ns(int(ns))


PIPE_SLOTS = ["mma_wait_acc_drain", "mma_wait_dequant", "mma_wait_tma", "mma_total", "producer_wait_stage",
              "producer_total", "dequant_wait_tma", "dequant_total", "epilogue_wait_acc", "epilogue_total",
              "tiles"]


def moe_pipeline_counters(layer: int) -> dict:
    """{'gateup': {slot: cycles}, 'down': {...}} since the last read (MOE_PIPE_PROF=1)."""
    buf = (C.c_ulonglong * 32)()
    _check(lib().moe_pipeline_counters(layer, C.cast(buf, C.c_void_p)), "moe_pipeline_counters")
    return {k: {n: int(buf[16 * j + i]) for i, n in enumerate(PIPE_SLOTS)} for j, k in enumerate(("gateup", "down"))}


def moe_profiler_enable(on: bool) -> None:
    lib().moe_profiler_enable(1 if on else 0)


def moe_profiler_read() -> dict:
    """{kernel name: (total ms, launches)} since the last read."""
    n = 32
    names = (C.c_char_p * n)()
    tot = (C.c_double * n)()
    cnt = (C.c_longlong * n)()
    k = lib().moe_profiler_read(C.cast(names, C.c_void_p), C.cast(tot, C.c_void_p), C.cast(cnt, C.c_void_p), n)
    return {names[i].decode(): (tot[i], cnt[i]) for i in range(min(k, n))}


def gqa_decode_workspace_bytes(B: int) -> int:
    return int(lib().gqa_decode_workspace_bytes(int(B)))


def gqa_decode_attention(q: int, k: int, v: int, lens, B: int, S_max: int, out: int, workspace: int,
                         workspace_bytes: int, stream: int = 0) -> None:
    """lens: a sequence of B ints (host memory, as the C entry takes it)."""
    vals = [int(x) for x in lens]
    arr = (C.c_int32 * max(1, len(vals)))(*vals)
    _check(lib().gqa_decode_attention(q, k, v, C.cast(arr, C.c_void_p), B, S_max, out, workspace, workspace_bytes,
                                      stream or None), "gqa_decode_attention")


def gqa_decode_get_error(workspace: int) -> int:
    return int(lib().gqa_decode_get_error(workspace))


def declared_functions() -> list[str]:
    """Names of the functions declared in include/*.h."""
    import re
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b((?:moe|gqa)_[a-z_0-9]+)\s*\(", text))
    return sorted(names)
