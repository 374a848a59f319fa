"""Torch-facing wrappers over the C ABI: device weights, workspace, layers and stacks.

PyTorch supplies device memory and streams only.  ``MoELayer.forward`` is one C call
(``moe_forward`` / ``moe_forward_residual``); ``MoEStack.forward`` is one
``moe_stack_forward`` call.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import _abi
from ._abi import MoeConfig, MoeQMat, MoeWeights

HIDDEN, N_EXPERTS, TOP_K, INTER, SHARED_INTER, GROUP = 2048, 256, 8, 512, 512, 64


def config(max_tokens: int) -> MoeConfig:
    return MoeConfig(HIDDEN, N_EXPERTS, TOP_K, INTER, SHARED_INTER, GROUP, 4, int(max_tokens))


def _dev(a: np.ndarray, device) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    elif a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device, non_blocking=False)


@dataclass
class DeviceQMat:
    q: torch.Tensor
    scales: torch.Tensor
    biases: torch.Tensor

    def c(self) -> MoeQMat:
        return MoeQMat(self.q.data_ptr(), self.scales.data_ptr(), self.biases.data_ptr())


class DeviceWeights:
    """One layer's weights resident on the GPU, in the MLX affine 4-bit layout.

    ``host`` is any object with the attributes ``gate, up, down, sh_gate, sh_up,
    sh_down`` (each with numpy ``q`` uint32, ``scales``/``biases`` uint16 bf16 bits),
    ``router_w`` (uint16), ``shared_gate_w`` (uint16) and ``router_bias`` (float32 or
    None)."""

    def __init__(self, host, device="cuda"):
        self.mats = {n: DeviceQMat(_dev(getattr(host, n).q, device), _dev(getattr(host, n).scales, device),
                                   _dev(getattr(host, n).biases, device))
                     for n in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down")}
        self.router_w = _dev(host.router_w, device)
        self.shared_gate_w = _dev(host.shared_gate_w, device)
        rb = getattr(host, "router_bias", None)
        self.router_bias = None if rb is None else _dev(np.asarray(rb, np.float32), device)
        nw = getattr(host, "norm_w", None)
        self.norm_w = None if nw is None else _dev(np.asarray(nw, np.uint16), device)

    def c(self) -> MoeWeights:
        m = self.mats
        return MoeWeights(m["gate"].c(), m["up"].c(), m["down"].c(), m["sh_gate"].c(), m["sh_up"].c(),
                          m["sh_down"].c(), self.router_w.data_ptr(),
                          None if self.router_bias is None else self.router_bias.data_ptr(),
                          self.shared_gate_w.data_ptr(),
                          None if self.norm_w is None else self.norm_w.data_ptr())

    @property
    def nbytes(self) -> int:
        n = sum(t.numel() * t.element_size() for m in self.mats.values() for t in (m.q, m.scales, m.biases))
        n += self.router_w.numel() * 2 + self.shared_gate_w.numel() * 2
        return n


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def workspace_bytes(max_tokens: int) -> int:
    return _abi.moe_workspace_bytes(config(max_tokens))


def new_workspace(max_tokens: int, device="cuda") -> torch.Tensor:
    n = workspace_bytes(max_tokens)
    if n == 0:
        raise ValueError("configuration refused")
    return torch.empty(n, dtype=torch.uint8, device=device)


class MoELayer:
    """One MoE layer bound to a caller-owned workspace (allocated here if not given)."""

    def __init__(self, weights: DeviceWeights, max_tokens: int, workspace: torch.Tensor | None = None):
        self.weights = weights
        self.max_tokens = int(max_tokens)
        self.workspace = workspace if workspace is not None else new_workspace(max_tokens, weights.router_w.device)
        self._cw = weights.c()
        self.handle = _abi.moe_layer_create(config(max_tokens), self._cw, self.workspace.data_ptr(),
                                            self.workspace.numel())

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            try:
                _abi.moe_layer_destroy(h)
            except Exception:
                pass
            self.handle = None

    def forward(self, x: torch.Tensor, out: torch.Tensor | None = None, residual: bool = False,
                stream=None) -> torch.Tensor:
        assert x.dtype == torch.bfloat16 and x.is_contiguous() and x.dim() == 2
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        fn = _abi.moe_forward_residual if residual else _abi.moe_forward
        fn(self.handle, x.data_ptr(), T, out.data_ptr(), _stream_handle(stream))
        return out

    def route(self, x: torch.Tensor, stream=None) -> dict:
        T = x.shape[0]
        dev = x.device
        r = dict(idx=torch.empty((T, TOP_K), dtype=torch.int32, device=dev),
                 w=torch.empty((T, TOP_K), dtype=torch.float32, device=dev),
                 counts=torch.empty(N_EXPERTS, dtype=torch.int32, device=dev),
                 offsets=torch.empty(N_EXPERTS + 1, dtype=torch.int32, device=dev),
                 perm=torch.empty(T * TOP_K, dtype=torch.int32, device=dev))
        _abi.moe_route(self.handle, x.data_ptr(), T, r["idx"].data_ptr(), r["w"].data_ptr(), r["counts"].data_ptr(),
                       r["offsets"].data_ptr(), r["perm"].data_ptr(), _stream_handle(stream))
        return r

    def get_error(self) -> int:
        return _abi.moe_layer_get_error(self.handle)


class MoEStack:
    """Layers applied in sequence with a residual add, in place, one C call."""

    def __init__(self, layers: list[MoELayer]):
        self.layers = layers
        self.handles = [l.handle for l in layers]

    def forward_(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        _abi.moe_stack_forward(self.handles, x.data_ptr(), x.shape[0], _stream_handle(stream))
        return x

    def forward_host(self, x_host: torch.Tensor, out_host: torch.Tensor, stream=None) -> torch.Tensor:
        _abi.moe_stack_forward_host(self.handles, x_host.data_ptr(), x_host.shape[0], out_host.data_ptr(),
                                    _stream_handle(stream))
        return out_host
