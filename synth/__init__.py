"""Seeded synthetic inputs for the Qwen3.6-35B-A3B mixture-of-experts layer.

This module draws the inputs that both the CPU oracle and the CUDA library read:
4-bit expert weights in the MLX affine layout, the bf16 router matrix, the bf16
shared-expert gate vector, the optional fp32 per-expert router bias of the
skewed-routing workload, and bf16 activations.  It holds none of the layer's
arithmetic (no dequantisation, no routing, no expert maths): it only draws random
numbers and rounds them to the storage types.

Distributions (the layer as used by Lily, an engine for exactly this model; the
pages name the format "MLX affine 4-bit, group size 64" -- aimanavo.com, "Why is
Perplexity's local AI Lily faster than MLX", section "Only one 4-bit checkpoint of
a pinned revision runs"):

* packed weights: uniform uint32 words.  Every nibble of a uniform word is an
  independent draw from U{0..15}, the same law as drawing each 4-bit code and
  packing eight per word low nibble first.
* scales: ``bf16_rne(float32(U[0.002, 0.006]))``, one per group of 64 inputs.
* biases: ``bf16_rne(-8 * scale_bf16 + float32(N(0, 1e-3)))`` (1e-3 is the
  standard deviation), computed in float32.
* router matrix ``W_r[256, 2048]``: ``bf16_rne(float32(N(0, 0.02)))``.
* shared-expert gate vector ``g_s[2048]``: same law as the router (no law is given
  for it; this is the plainest reading).
* activations ``x[T, 2048]``: ``bf16_rne(float32(N(0, 1)))``.
* skewed workload: a random permutation ``pi`` of the experts gives each expert a
  rank ``r_e = pi(e) + 1``; its logit bias is
  ``1.5 * ln(r_e^-1.2 / H_{256,1.2})`` (a log-Zipf(s=1.2) law), in float32.

Random streams.  Every array has its own ``numpy.random.SeedSequence(seed,
spawn_key=(layer, stream))`` feeding a PCG64 generator, so layers, matrices and
activations are independent and each can be regenerated alone.  Layer ``l`` of a
stack uses ``layer=l``; activations use ``spawn_key=(X_STREAM,)``.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
import os

import numpy as np

__all__ = [
    "Dims", "QMat", "LayerWeights", "QWEN36_DIMS",
    "bf16_bits_from_f32", "f32_from_bf16_bits",
    "make_layer", "make_x", "make_skew_bias", "make_stack", "stack_layer", "make_gqa",
]

# stream ids (second element of spawn_key)
_S_ROUTER = 1
_S_SHARED_GATE = 2
_S_SKEW = 3
_S_MAT_BASE = 16          # + 4*matrix_index + {0: codes, 1: scales, 2: bias noise}
X_STREAM = 0x7800


@dataclass(frozen=True)
class Dims:
    """Layer dimensions.  The defaults are Qwen3.6-35B-A3B's MoE layer."""
    hidden: int = 2048
    n_experts: int = 256
    top_k: int = 8
    inter: int = 512
    shared_inter: int = 512
    group: int = 64


QWEN36_DIMS = Dims()


@dataclass
class QMat:
    """One MLX affine 4-bit matrix (or a stack of them along a leading axis).

    ``q``: uint32 ``[..., out, in/8]`` (eight 4-bit codes per word, low nibble
    first); ``scales`` / ``biases``: bf16 bits as uint16 ``[..., out, in/group]``.
    """
    q: np.ndarray
    scales: np.ndarray
    biases: np.ndarray

    @property
    def nbytes(self) -> int:
        return self.q.nbytes + self.scales.nbytes + self.biases.nbytes


@dataclass
class LayerWeights:
    dims: Dims
    gate: QMat          # [E, inter, hidden]
    up: QMat            # [E, inter, hidden]
    down: QMat          # [E, hidden, inter]
    sh_gate: QMat       # [shared_inter, hidden]
    sh_up: QMat         # [shared_inter, hidden]
    sh_down: QMat       # [hidden, shared_inter]
    router_w: np.ndarray                    # uint16 bf16 bits [E, hidden]
    shared_gate_w: np.ndarray               # uint16 bf16 bits [hidden]
    router_bias: np.ndarray | None = None   # float32 [E] or None
    norm_w: np.ndarray | None = None        # uint16 bf16 bits [hidden]: input RMSNorm, or None
    seed: int = 0
    layer: int = 0
    extra: dict = field(default_factory=dict)

    def qmats(self):
        return [self.gate, self.up, self.down, self.sh_gate, self.sh_up, self.sh_down]

    @property
    def nbytes(self) -> int:
        n = sum(m.nbytes for m in self.qmats()) + self.router_w.nbytes + self.shared_gate_w.nbytes
        if self.router_bias is not None:
            n += self.router_bias.nbytes
        return n


def bf16_bits_from_f32(a) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even); return the bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    r = ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)
    return r


def f32_from_bf16_bits(b) -> np.ndarray:
    """Widen bfloat16 bits (uint16) to float32 exactly."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=tuple(key))))


def _qmat(seed: int, layer: int, mat_index: int, lead: tuple, out_dim: int, in_dim: int, group: int) -> QMat:
    base = _S_MAT_BASE + 4 * mat_index
    q = _rng(seed, layer, base + 0).integers(0, 2**32, size=lead + (out_dim, in_dim // 8), dtype=np.uint32)
    gshape = lead + (out_dim, in_dim // group)
    s32 = _rng(seed, layer, base + 1).uniform(0.002, 0.006, size=gshape).astype(np.float32)
    scales = bf16_bits_from_f32(s32)
    noise = _rng(seed, layer, base + 2).normal(0.0, 1e-3, size=gshape).astype(np.float32)
    b32 = (np.float32(-8.0) * f32_from_bf16_bits(scales) + noise).astype(np.float32)
    biases = bf16_bits_from_f32(b32)
    return QMat(q, scales, biases)


def make_skew_bias(seed: int, n_experts: int = 256, layer: int = 0) -> np.ndarray:
    """Per-expert fp32 router-logit bias 1.5*log-Zipf(s=1.2) over a random expert permutation."""
    perm = _rng(seed, layer, _S_SKEW).permutation(n_experts)
    rank = perm.astype(np.float64) + 1.0
    h = np.sum(np.arange(1, n_experts + 1, dtype=np.float64) ** -1.2)
    return (1.5 * np.log(rank ** -1.2 / h)).astype(np.float32)


def make_layer(seed: int = 0, layer: int = 0, dims: Dims = QWEN36_DIMS, skew: bool = False,
               threads: int | None = None) -> LayerWeights:
    """Draw one layer's weights.  ``skew`` adds the log-Zipf router bias."""
    d = dims
    if d.hidden % d.group or d.inter % d.group or d.shared_inter % d.group or d.group % 8:
        raise ValueError("dimensions must be multiples of the group, and the group of 8")
    E = d.n_experts
    jobs = [
        (0, (E,), d.inter, d.hidden),
        (1, (E,), d.inter, d.hidden),
        (2, (E,), d.hidden, d.inter),
        (3, (), d.shared_inter, d.hidden),
        (4, (), d.shared_inter, d.hidden),
        (5, (), d.hidden, d.shared_inter),
    ]
    nthreads = threads or min(6, os.cpu_count() or 1)
    with ThreadPoolExecutor(nthreads) as ex:
        mats = list(ex.map(lambda j: _qmat(seed, layer, j[0], j[1], j[2], j[3], d.group), jobs))
    rw = bf16_bits_from_f32(_rng(seed, layer, _S_ROUTER).normal(0.0, 0.02, size=(E, d.hidden)).astype(np.float32))
    gs = bf16_bits_from_f32(_rng(seed, layer, _S_SHARED_GATE).normal(0.0, 0.02, size=(d.hidden,)).astype(np.float32))
    bias = make_skew_bias(seed, E, layer) if skew else None
    return LayerWeights(d, *mats, router_w=rw, shared_gate_w=gs, router_bias=bias, seed=seed, layer=layer)


BF16_ONE = 0x3F80


def stack_layer(l: int, dims: Dims = QWEN36_DIMS, threads: int | None = None) -> LayerWeights:
    """Layer l of a stack: seed l, with an input RMSNorm of weight 1 (see ``make_stack``)."""
    L = make_layer(seed=l, layer=l, dims=dims, threads=threads)
    L.norm_w = np.full(dims.hidden, BF16_ONE, np.uint16)
    return L


def make_stack(n_layers: int, dims: Dims = QWEN36_DIMS, threads: int | None = None):
    """A stack of independently seeded layers: layer l uses seed l, and every layer
    RMS-normalises its input (weight 1) before the mixture of experts; the residual adds
    the un-normalised input.  Without the norm such a stack diverges within a few
    layers (the SwiGLU output grows with the square of its input)."""
    return [stack_layer(l, dims, threads) for l in range(n_layers)]


def make_x(seed: int, T: int, hidden: int = 2048) -> np.ndarray:
    """Activations x[T, hidden] as bf16 bits (uint16), N(0, 1)."""
    return bf16_bits_from_f32(_rng(seed, X_STREAM).normal(0.0, 1.0, size=(T, hidden)).astype(np.float32))


GQA_STREAM = 0x7900


def make_gqa(seed: int, B: int, S_max: int, lens=None, Hq: int = 16, Hkv: int = 2, D: int = 128,
             needles: int = 4, needle_scale: float = 1.0, threads: int | None = None):
    """Inputs of one grouped-query decode-attention step: the new query token of each of
    B sequences and their key/value caches, as bf16 bits (uint16).

    q [B, Hq, D], k and v [B, Hkv, S_max, D] ~ N(0, 1); lens [B] int32 (all S_max unless
    given).  The pages give no law for these tensors; N(0, 1) is the plainest reading.
    ``needles`` planted keys per (sequence, query head) copy that head's query, times
    ``needle_scale``, into a random cached position of its KV head, so every head has a
    few keys it attends to sharply and heads sharing a KV head attend to different
    positions (real attention is peaked rather than uniform).  Rows at or beyond a
    sequence's length are drawn too (the kernels must not read them)."""
    B, S_max = int(B), int(S_max)
    lens = np.full(B, S_max, np.int32) if lens is None else np.asarray(lens, np.int32)
    g = Hq // Hkv
    rq = _rng(seed, GQA_STREAM)
    q = rq.normal(0.0, 1.0, size=(B, Hq, D)).astype(np.float32)
    k = np.empty((B, Hkv, S_max, D), np.float32)
    v = np.empty((B, Hkv, S_max, D), np.float32)

    def fill(args):
        b, j = args
        r = _rng(seed, GQA_STREAM + 1 + b * Hkv + j)
        k[b, j] = r.normal(0.0, 1.0, size=(S_max, D))
        v[b, j] = r.normal(0.0, 1.0, size=(S_max, D))
        if needles and lens[b] > 0:
            pos = r.integers(0, lens[b], size=(g, needles))
            for hh in range(g):
                k[b, j, pos[hh]] = needle_scale * q[b, j * g + hh]
    with ThreadPoolExecutor(threads or min(8, os.cpu_count() or 1)) as ex:
        list(ex.map(fill, [(b, j) for b in range(B) for j in range(Hkv)]))
    return (bf16_bits_from_f32(q), bf16_bits_from_f32(k), bf16_bits_from_f32(v), lens)


def expected_touched(T: int, n_experts: int = 256, top_k: int = 8) -> float:
    """Expected number of distinct experts hit by T tokens under uniform routing."""
    return n_experts * (1.0 - ((n_experts - top_k) / n_experts) ** T)

