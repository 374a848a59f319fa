"""CPU oracle for the 4-bit mixture-of-experts layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it, and it
imports nothing from the library: the two share only the seeded inputs of
``synth``.

The arithmetic lives in ``moe_oracle.c`` (plain C, double precision, one token and
one output at a time); this module compiles it with gcc and wraps it with ctypes.
Every function cites, in the C file, the passage it follows.

Pinned by ``tests/test_oracle_pins.py`` (hand-built words, exact dequant cases,
brute-force top-k, closed forms of identity-like experts, permutation invariance,
a float64 dense NumPy special case) and ``tests/test_oracle_mutants.py`` (each
planted mistake fails at least one pin).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_SRC_GQA = os.path.join(_HERE, "gqa_oracle.c")
_LOCK = threading.Lock()
_LIBS: dict[int, C.CDLL] = {}


def lib_path(mutant: int = 0) -> str:
    name = "libmoe_oracle.so" if mutant == 0 else f"libmoe_oracle_m{mutant}.so"
    return os.path.join(_HERE, "_build", name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (or a planted-mistake variant) with gcc; return the .so path."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= max(
            os.path.getmtime(_SRC), os.path.getmtime(_SRC_GQA), os.path.getmtime(os.path.join(_HERE, "moe_oracle.h"))):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
           f"-DORACLE_MUTANT={int(mutant)}", _SRC, _SRC_GQA, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class Dims(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("hidden", "n_experts", "top_k", "inter", "shared_inter", "group")]


class QMat(C.Structure):
    _fields_ = [("q", C.c_void_p), ("scales", C.c_void_p), ("biases", C.c_void_p)]


class Weights(C.Structure):
    _fields_ = [("gate", QMat), ("up", QMat), ("down", QMat),
                ("sh_gate", QMat), ("sh_up", QMat), ("sh_down", QMat),
                ("router_w", C.c_void_p), ("router_bias", C.c_void_p), ("shared_gate_w", C.c_void_p),
                ("norm_w", C.c_void_p)]


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def load(mutant: int = 0) -> C.CDLL:
    with _LOCK:
        if mutant in _LIBS:
            return _LIBS[mutant]
        lib = C.CDLL(build(mutant))
        P = C.c_void_p
        lib.oracle_bf16_to_double.argtypes = [C.c_uint16]
        lib.oracle_bf16_to_double.restype = C.c_double
        lib.oracle_double_to_bf16.argtypes = [C.c_double]
        lib.oracle_double_to_bf16.restype = C.c_uint16
        lib.oracle_unpack4.argtypes = [C.c_uint32, P]
        lib.oracle_dequant_row.argtypes = [P, P, P, C.c_int, C.c_int, P]
        lib.oracle_qmatvec.argtypes = [C.POINTER(QMat), C.c_long, C.c_int, C.c_int, C.c_int, P, P]
        lib.oracle_router_logits.argtypes = [C.POINTER(Dims), P, P, P, P]
        lib.oracle_layer_logits.argtypes = [C.POINTER(Dims), C.POINTER(Weights), P, P]
        lib.oracle_rmsnorm.argtypes = [C.c_int, P, P, P]
        lib.oracle_route_logits.argtypes = [C.POINTER(Dims), P, P, P, P, P, P]
        lib.oracle_expert.argtypes = [C.POINTER(Dims), C.POINTER(QMat), C.POINTER(QMat), C.POINTER(QMat),
                                      C.c_long, C.c_int, P, P]
        lib.oracle_shared_gate.argtypes = [C.POINTER(Dims), P, P]
        lib.oracle_shared_gate.restype = C.c_double
        lib.oracle_token_forward.argtypes = [C.POINTER(Dims), C.POINTER(Weights), P, P, P, C.c_int, P]
        lib.oracle_route.argtypes = [C.POINTER(Dims), C.POINTER(Weights), P, C.c_int, C.c_int, P, P, P, P, P, P]
        lib.oracle_layer_forward.argtypes = [C.POINTER(Dims), C.POINTER(Weights), P, C.c_int, C.c_int, C.c_int,
                                             P, P, P, P]
        lib.oracle_token_forward_choice.argtypes = [C.POINTER(Dims), C.POINTER(Weights), P, P, C.c_int, P, P]
        lib.oracle_mutant.restype = C.c_int
        lib.oracle_gqa_decode.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, P, P, P, P, C.c_double,
                                          C.c_int, P, P]
        lib.oracle_gqa_decode.restype = None
        _LIBS[mutant] = lib
        return lib


def default_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


class Oracle:
    """ctypes front end over one compiled oracle (``mutant`` 0 is the real one)."""

    def __init__(self, mutant: int = 0):
        self.lib = load(mutant)
        self.mutant = mutant

    # --- small pieces --------------------------------------------------------
    def bf16_to_double(self, b: int) -> float:
        return self.lib.oracle_bf16_to_double(int(b))

    def double_to_bf16(self, v: float) -> int:
        return int(self.lib.oracle_double_to_bf16(float(v)))

    def unpack4(self, word: int) -> list[int]:
        q = np.zeros(8, np.int32)
        self.lib.oracle_unpack4(C.c_uint32(word & 0xFFFFFFFF), _p(q))
        return q.tolist()

    def dequant_row(self, q_row, s_row, b_row, group: int) -> np.ndarray:
        q_row = np.ascontiguousarray(q_row, np.uint32)
        s_row = np.ascontiguousarray(s_row, np.uint16)
        b_row = np.ascontiguousarray(b_row, np.uint16)
        w = np.zeros(q_row.size * 8, np.float64)
        self.lib.oracle_dequant_row(_p(q_row), _p(s_row), _p(b_row), q_row.size * 8, group, _p(w))
        return w

    @staticmethod
    def _dims(d) -> Dims:
        return Dims(d.hidden, d.n_experts, d.top_k, d.inter, d.shared_inter, d.group)

    @staticmethod
    def _qmat(m) -> QMat:
        return QMat(_p(m.q), _p(m.scales), _p(m.biases))

    def _weights(self, L) -> Weights:
        for m in L.qmats():
            assert m.q.flags.c_contiguous and m.scales.flags.c_contiguous and m.biases.flags.c_contiguous
        return Weights(*(self._qmat(m) for m in L.qmats()), _p(L.router_w), _p(L.router_bias),
                       _p(L.shared_gate_w), _p(getattr(L, "norm_w", None)))

    def router_logits(self, L, x_row) -> np.ndarray:
        """The layer's fp32 router logits for one token (after the layer's input norm, if any)."""
        x_row = np.ascontiguousarray(x_row, np.uint16)
        out = np.zeros(L.dims.n_experts, np.float32)
        d, W = self._dims(L.dims), self._weights(L)
        self.lib.oracle_layer_logits(C.byref(d), C.byref(W), _p(x_row), _p(out))
        return out

    def rmsnorm(self, x_row, norm_w) -> np.ndarray:
        x_row = np.ascontiguousarray(x_row, np.uint16)
        norm_w = np.ascontiguousarray(norm_w, np.uint16)
        out = np.zeros_like(x_row)
        self.lib.oracle_rmsnorm(x_row.size, _p(x_row), _p(norm_w), _p(out))
        return out

    def route_logits(self, dims, logits):
        """Route one token from its fp32 logits: (idx, w, gap, p_sorted, order)."""
        logits = np.ascontiguousarray(logits, np.float32)
        K, E = dims.top_k, dims.n_experts
        idx = np.zeros(K, np.int32)
        w = np.zeros(K, np.float64)
        gap = np.zeros(1, np.float64)
        ps = np.zeros(E, np.float64)
        order = np.zeros(E, np.int32)
        d = self._dims(dims)
        self.lib.oracle_route_logits(C.byref(d), _p(logits), _p(idx), _p(w), _p(gap), _p(ps), _p(order))
        return idx, w, float(gap[0]), ps, order

    def expert(self, L, e: int, x: np.ndarray, shared: bool = False) -> np.ndarray:
        d = self._dims(L.dims)
        x = np.ascontiguousarray(x, np.float64)
        y = np.zeros(L.dims.hidden, np.float64)
        if shared:
            mats = (self._qmat(L.sh_gate), self._qmat(L.sh_up), self._qmat(L.sh_down))
            inter = L.dims.shared_inter
        else:
            mats = (self._qmat(L.gate), self._qmat(L.up), self._qmat(L.down))
            inter = L.dims.inter
        self.lib.oracle_expert(C.byref(d), *(C.byref(m) for m in mats), e, inter, _p(x), _p(y))
        return y

    def shared_gate(self, L, x_row) -> float:
        d = self._dims(L.dims)
        x_row = np.ascontiguousarray(x_row, np.uint16)
        return self.lib.oracle_shared_gate(C.byref(d), _p(L.shared_gate_w), _p(x_row))

    # --- whole layer ---------------------------------------------------------
    def route(self, L, x, nthreads: int | None = None):
        """Routing of every token: dict of idx [T,K], w [T,K] (float64), gap [T],
        counts [E], offsets [E+1], perm [T*K]."""
        x = np.ascontiguousarray(x, np.uint16)
        T = x.shape[0]
        K, E = L.dims.top_k, L.dims.n_experts
        idx = np.zeros((T, K), np.int32)
        w = np.zeros((T, K), np.float64)
        gap = np.zeros(T, np.float64)
        counts = np.zeros(E, np.int32)
        offsets = np.zeros(E + 1, np.int32)
        perm = np.zeros(T * K, np.int32)
        d, W = self._dims(L.dims), self._weights(L)
        self.lib.oracle_route(C.byref(d), C.byref(W), _p(x), T, nthreads or default_threads(),
                              _p(idx), _p(w), _p(gap), _p(counts), _p(offsets), _p(perm))
        return dict(idx=idx, w=w, gap=gap, counts=counts, offsets=offsets, perm=perm)

    def forward(self, L, x, residual: bool = False, nthreads: int | None = None):
        """The layer on every token: dict of out (bf16 bits [T,H]), idx, w, gap."""
        x = np.ascontiguousarray(x, np.uint16)
        T = x.shape[0]
        K = L.dims.top_k
        out = np.zeros((T, L.dims.hidden), np.uint16)
        idx = np.zeros((T, K), np.int32)
        w = np.zeros((T, K), np.float64)
        gap = np.zeros(T, np.float64)
        d, W = self._dims(L.dims), self._weights(L)
        self.lib.oracle_layer_forward(C.byref(d), C.byref(W), _p(x), T, int(residual), nthreads or default_threads(),
                                      _p(out), _p(idx), _p(w), _p(gap))
        return dict(out=out, idx=idx, w=w, gap=gap)

    def token_forward_choice(self, L, x_row, experts, residual: bool = False):
        """One token with an oracle-chosen alternative expert list: (out bits [H], w [K])."""
        x_row = np.ascontiguousarray(x_row, np.uint16)
        ex = np.ascontiguousarray(experts, np.int32)
        out = np.zeros(L.dims.hidden, np.uint16)
        w = np.zeros(L.dims.top_k, np.float64)
        d, W = self._dims(L.dims), self._weights(L)
        self.lib.oracle_token_forward_choice(C.byref(d), C.byref(W), _p(x_row), _p(ex), int(residual),
                                             _p(out), _p(w))
        return out, w

    def gqa_decode(self, q, k, v, lens, scale=None, nthreads: int | None = None):
        """Grouped-query decode attention (gqa_oracle.c): q bf16 bits [B, Hq, D], k and v
        bf16 bits [B, Hkv, S_max, D], lens [B].  Returns (out, abs_out), float64 [B, Hq, D]."""
        q = np.ascontiguousarray(q, np.uint16)
        k = np.ascontiguousarray(k, np.uint16)
        v = np.ascontiguousarray(v, np.uint16)
        lens = np.ascontiguousarray(lens, np.int32)
        B, Hq, D = q.shape
        _, Hkv, S_max, _ = k.shape
        assert k.shape == v.shape == (B, Hkv, S_max, D) and lens.shape == (B,)
        assert Hq % Hkv == 0 and np.all(lens >= 1) and np.all(lens <= S_max)
        out = np.zeros((B, Hq, D), np.float64)
        aout = np.zeros((B, Hq, D), np.float64)
        sc = 1.0 / np.sqrt(D) if scale is None else float(scale)
        self.lib.oracle_gqa_decode(B, Hq, Hkv, D, S_max, _p(lens), _p(q), _p(k), _p(v), sc,
                                   nthreads or default_threads(), _p(out), _p(aout))
        return out, aout

    def token_forward(self, L, x_row, experts, wts, residual: bool = False) -> np.ndarray:
        """One token, experts and weights given, unrounded double output [H]."""
        x_row = np.ascontiguousarray(x_row, np.uint16)
        ex = np.ascontiguousarray(experts, np.int32)
        wt = np.ascontiguousarray(wts, np.float64)
        out = np.zeros(L.dims.hidden, np.float64)
        d, W = self._dims(L.dims), self._weights(L)
        self.lib.oracle_token_forward(C.byref(d), C.byref(W), _p(x_row), _p(ex), _p(wt), int(residual), _p(out))
        return out


def valid_sets(ps, order, own, K: int, tol: float = 1e-4, max_choices: int = 8, mutant: int = 0):
    """The top-K expert sets that count as correct for one token, from its probabilities
    sorted in descending order (``ps``, with the expert ids ``order`` in the same order)
    and the oracle's own choice ``own``.

    The near-tie reading of the parity rule: with S the mass of the K largest
    probabilities and p_K the K-th largest, an expert whose probability exceeds
    p_K + tol*S must be chosen, and the slots left over may hold any experts whose
    probability is within tol*S of p_K (both bounds inclusive).  Returns the oracle's
    own set first, then the other such sets, at most ``max_choices`` in all.

    ``mutant`` plants a mistake for the pin tests (0 = none): 1 drops the factor S from
    the band, 2 builds the must-choose set with >= instead of >."""
    from itertools import combinations
    ps = np.asarray(ps, np.float64)
    S = float(np.sum(ps[:K]))
    pk = ps[K - 1]
    band_w = tol if mutant == 1 else tol * S
    if mutant == 2:
        sure = [int(order[r]) for r in range(len(order)) if ps[r] >= pk + band_w]
    else:
        sure = [int(order[r]) for r in range(len(order)) if ps[r] > pk + band_w]
    band = [int(order[r]) for r in range(len(order)) if abs(ps[r] - pk) <= band_w]
    need = K - len(sure)
    out = [[int(e) for e in own]]
    if need <= 0:
        return out
    for comb in combinations(band, need):
        cand = sure + list(comb)
        if sorted(cand) != sorted(out[0]):
            out.append(cand)
        if len(out) >= max_choices:
            break
    return out


def valid_choices(oracle: Oracle, dims, logits, tol: float = 1e-4, max_choices: int = 8):
    """Every top-k expert set that is valid for a near-tie token (``valid_sets``), from
    the oracle's own routing of the token's fp32 logits.  Returns a list of expert lists
    (the oracle's own choice first)."""
    idx, w, gap, ps, order = oracle.route_logits(dims, logits)
    return valid_sets(ps, order, idx, dims.top_k, tol, max_choices)
