"""ctypes front end of the C++ float64 oracle (oracle/moe_oracle_ref.cpp).

TEST INFRASTRUCTURE (see oracle/__init__.py). Numpy arrays in, numpy arrays out;
the arithmetic is all in the C++ library. The functions mirror the numpy
restatement in ``moe_oracle`` (same names and argument order), so the same pins
run against both.

Expert weights are handed over per expert by a callable ``e -> weights``:
  * ``(w13, w2)`` float64 arrays [2I, H], [H, I] (any values), or
  * ``(w13, w2)`` uint16 arrays of bf16 bit patterns, or
  * an :class:`NVFP4Expert` of codes, e4m3 scale bytes and tensor scales, or
  * an :class:`FP8Expert` of e4m3 codes and float32 128 x 128 block scales.
Only the experts some row selects (and the shared ones) are requested.
"""

from __future__ import annotations

import ctypes
from collections import namedtuple

import numpy as np

from . import build as _build

SCORE_SOFTMAX = 0
SCORE_SIGMOID_BIAS = 1
FMT_F64, FMT_BF16, FMT_NVFP4, FMT_FP8 = 0, 1, 2, 3

# gate/up codes [2I, H/2], scales [2I, H/16], tensor scales (gate, up); down
# codes [H, I/2], scales [H, I/16], tensor scale
NVFP4Expert = namedtuple("NVFP4Expert", "q13 s13 gs13 q2 s2 gs2")
# e4m3 gate/up codes [2I, H], float32 scales [2I/128, H/128]; down codes [H, I],
# scales [H/128, I/128]
FP8Expert = namedtuple("FP8Expert", "q13 s13 q2 s2")


class _Experts(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("w13", ctypes.POINTER(ctypes.c_void_p)),
                ("w2", ctypes.POINTER(ctypes.c_void_p)), ("w13_scale", ctypes.POINTER(ctypes.c_void_p)),
                ("w2_scale", ctypes.POINTER(ctypes.c_void_p)), ("w13_gscale", ctypes.c_void_p),
                ("w2_gscale", ctypes.c_void_p)]


class _Shape(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("num_shared", ctypes.c_int32), ("rows", ctypes.c_int32),
                ("score", ctypes.c_int32), ("router_fmt", ctypes.c_int32), ("routed_scale", ctypes.c_double),
                ("threads", ctypes.c_int32)]


_libs: dict = {}


def load(mutant: int = 0) -> ctypes.CDLL:
    """The oracle library (built first when missing or stale)."""
    if mutant not in _libs:
        lib = ctypes.CDLL(_build.build(mutant))
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.moe_oracle_bf16_to_f64.argtypes = [vp, vp, i64]
        lib.moe_oracle_bf16_to_f64.restype = None
        lib.moe_oracle_f64_to_bf16.argtypes = [vp, vp, i64]
        lib.moe_oracle_f64_to_bf16.restype = None
        lib.moe_oracle_e2m1.argtypes = [i32]
        lib.moe_oracle_e2m1.restype = dbl
        lib.moe_oracle_e4m3.argtypes = [i32]
        lib.moe_oracle_e4m3.restype = dbl
        lib.moe_oracle_silu.argtypes = [vp, vp, i64]
        lib.moe_oracle_silu.restype = None
        lib.moe_oracle_rmsnorm_bf16.argtypes = [vp, vp, i32, i32, dbl]
        lib.moe_oracle_rmsnorm_bf16.restype = None
        lib.moe_oracle_select.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        lib.moe_oracle_select.restype = i32
        lib.moe_oracle_router.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp]
        lib.moe_oracle_router.restype = i32
        lib.moe_oracle_layer.argtypes = [ctypes.POINTER(_Shape), vp, vp, vp, vp, ctypes.POINTER(_Experts),
                                         ctypes.POINTER(_Experts), vp, vp, vp, vp]
        lib.moe_oracle_layer.restype = i32
        lib.moe_oracle_max_threads.restype = i32
        _libs[mutant] = lib
    return _libs[mutant]


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def max_threads(lib=None) -> int:
    return int((lib or load()).moe_oracle_max_threads())


# ----------------------------------------------------------------------------- number formats


def bf16_bits_to_f64(bits, lib=None) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, np.float64)
    (lib or load()).moe_oracle_bf16_to_f64(_ptr(b), _ptr(out), b.size)
    return out


def f64_to_bf16_bits(v, lib=None) -> np.ndarray:
    a = _f64(v)
    out = np.empty(a.shape, np.uint16)
    (lib or load()).moe_oracle_f64_to_bf16(_ptr(a), _ptr(out), a.size)
    return out


def e2m1_value(code, lib=None) -> float:
    return float((lib or load()).moe_oracle_e2m1(int(code)))


def e4m3_value(byte, lib=None) -> float:
    return float((lib or load()).moe_oracle_e4m3(int(byte)))


def silu(g, lib=None) -> np.ndarray:
    a = _f64(g)
    out = np.empty(a.shape, np.float64)
    (lib or load()).moe_oracle_silu(_ptr(a), _ptr(out), a.size)
    return out


def stack_layer_input(hidden_bits, eps: float = 1e-6, lib=None) -> np.ndarray:
    """bf16 bits of bf16(RMSNorm(hidden)) per row, gamma = 1."""
    h = np.ascontiguousarray(hidden_bits, dtype=np.uint16)
    m, hd = h.shape
    out = np.empty_like(h)
    (lib or load()).moe_oracle_rmsnorm_bf16(_ptr(h), _ptr(out), m, hd, eps)
    return out


# ----------------------------------------------------------------------------- routing


def _router_arg(router_w):
    r = np.asarray(router_w)
    if r.dtype == np.uint16:
        return np.ascontiguousarray(r), FMT_BF16
    return _f64(r), FMT_F64


def router_logits(x, router_w, threads: int = 0, lib=None) -> np.ndarray:
    xa = _f64(np.atleast_2d(x))
    r, fmt = _router_arg(router_w)
    out = np.empty((xa.shape[0], r.shape[0]), np.float64)
    st = (lib or load()).moe_oracle_router(_ptr(xa), _ptr(r), fmt, xa.shape[0], xa.shape[1], r.shape[0], threads,
                                           _ptr(out))
    assert st == 0, st
    return out


def select(logits_row, k: int, score: int = SCORE_SOFTMAX, bias=None, lib=None):
    """(idx int64 [k], w float64 [k]) of one row of logits."""
    l = _f64(logits_row)
    b = None if bias is None else _f64(bias)
    idx = np.empty(k, np.int64)
    w = np.empty(k, np.float64)
    st = (lib or load()).moe_oracle_select(_ptr(l), l.size, k, score, _ptr(b), _ptr(idx), _ptr(w))
    if st != 0:
        raise ValueError(f"moe_oracle_select: status {st}")
    return idx, w


def topk_renorm(logits_row, k: int, lib=None):
    return select(logits_row, k, SCORE_SOFTMAX, None, lib)


def route(x, router_w, k: int, score: int = SCORE_SOFTMAX, bias=None, threads: int = 0, lib=None):
    logits = router_logits(x, router_w, threads, lib)
    idx = np.zeros((logits.shape[0], k), np.int64)
    w = np.zeros((logits.shape[0], k), np.float64)
    for m in range(logits.shape[0]):
        idx[m], w[m] = select(logits[m], k, score, bias, lib)
    return logits, idx, w


# ----------------------------------------------------------------------------- the layer


def _inter_of(w) -> int:
    """The expert intermediate size I from one expert's weights."""
    if isinstance(w, NVFP4Expert):
        return np.asarray(w.q2).shape[1] * 2
    if isinstance(w, FP8Expert):
        return np.asarray(w.q2).shape[1]
    return np.asarray(w[1]).shape[1]


class _ExpertTable:
    """ctypes pointer tables for a set of experts (keeps the arrays alive)."""

    def __init__(self, n: int, entries: dict):
        self.keep = []
        arr = lambda: (ctypes.c_void_p * max(n, 1))()  # noqa: E731
        self.w13, self.w2, self.s13, self.s2 = arr(), arr(), arr(), arr()
        self.gs13 = np.zeros((max(n, 1), 2), np.float32)
        self.gs2 = np.zeros(max(n, 1), np.float32)
        fmt = None
        for e, wts in entries.items():
            if isinstance(wts, FP8Expert):
                f = FMT_FP8
                q13, q2 = (np.ascontiguousarray(a, dtype=np.uint8) for a in (wts.q13, wts.q2))
                s13, s2 = (np.ascontiguousarray(a, dtype=np.float32) for a in (wts.s13, wts.s2))
                self.keep += [q13, s13, q2, s2]
                self.w13[e], self.w2[e] = q13.ctypes.data, q2.ctypes.data
                self.s13[e], self.s2[e] = s13.ctypes.data, s2.ctypes.data
            elif isinstance(wts, NVFP4Expert):
                f = FMT_NVFP4
                q13, s13, q2, s2 = (np.ascontiguousarray(a, dtype=np.uint8) for a in (wts.q13, wts.s13, wts.q2, wts.s2))
                self.keep += [q13, s13, q2, s2]
                self.w13[e], self.w2[e] = q13.ctypes.data, q2.ctypes.data
                self.s13[e], self.s2[e] = s13.ctypes.data, s2.ctypes.data
                self.gs13[e] = np.asarray(wts.gs13, np.float32).reshape(2)
                self.gs2[e] = np.float32(wts.gs2)
            else:
                w13, w2 = (np.asarray(a) for a in wts)
                f = FMT_BF16 if w13.dtype == np.uint16 else FMT_F64
                dt = np.uint16 if f == FMT_BF16 else np.float64
                w13, w2 = np.ascontiguousarray(w13, dtype=dt), np.ascontiguousarray(w2, dtype=dt)
                self.keep += [w13, w2]
                self.w13[e], self.w2[e] = w13.ctypes.data, w2.ctypes.data
            if fmt is not None and f != fmt:
                raise ValueError("all experts of one table must share a storage format")
            fmt = f
        self.struct = _Experts(FMT_F64 if fmt is None else fmt, self.w13, self.w2, self.s13, self.s2,
                               self.gs13.ctypes.data, self.gs2.ctypes.data)


def moe_layer(x, residual, router_w, expert_weights, shared_weights, top_k, routed_scale: float = 1.0,
              score: int = SCORE_SOFTMAX, bias=None, threads: int = 0, lib=None, return_logits: bool = False):
    """One layer step for M rows (same contract as ``moe_oracle.moe_layer``).

    x, residual float64 [M, H]; router_w float64 or bf16 bits [E, H];
    expert_weights(e) -> the weights of routed expert e (see the module doc);
    shared_weights: a list of the same for the shared experts.
    Returns (out float64 [M, H], idx int64 [M, k], w float64 [M, k]).
    """
    lib = lib or load()
    xa, ra = _f64(np.atleast_2d(x)), _f64(np.atleast_2d(residual))
    r, rfmt = _router_arg(router_w)
    m, h = xa.shape
    e_count = r.shape[0]
    b = None if bias is None else _f64(bias)
    _, idx0, _ = route(xa, r, top_k, score, b, threads, lib)
    needed = sorted(set(int(v) for v in idx0.ravel()))
    routed = _ExpertTable(e_count, {e: expert_weights(e) for e in needed})
    shared = _ExpertTable(len(shared_weights), dict(enumerate(shared_weights)))
    any_w = expert_weights(needed[0]) if needed else shared_weights[0]
    inter = _inter_of(any_w)
    shape = _Shape(h, inter, e_count, top_k, len(shared_weights), m, score, rfmt, float(routed_scale), threads)
    out = np.empty((m, h), np.float64)
    idx = np.empty((m, top_k), np.int64)
    w = np.empty((m, top_k), np.float64)
    logits = np.empty((m, e_count), np.float64)
    st = lib.moe_oracle_layer(ctypes.byref(shape), _ptr(xa), _ptr(ra), _ptr(r), _ptr(b), ctypes.byref(routed.struct),
                              ctypes.byref(shared.struct), _ptr(out), _ptr(idx), _ptr(w), _ptr(logits))
    if st != 0:
        raise RuntimeError(f"moe_oracle_layer: status {st}")
    return (out, idx, w, logits) if return_logits else (out, idx, w)


class Prepared:
    """A layer step with every needed expert's weights already in pointer tables,
    so that timing one call measures the oracle's arithmetic alone."""

    def __init__(self, x, residual, router_w, expert_weights, shared_weights, top_k, routed_scale=1.0,
                 score=SCORE_SOFTMAX, bias=None, lib=None):
        self.lib = lib or load()
        self.xa, self.ra = _f64(np.atleast_2d(x)), _f64(np.atleast_2d(residual))
        self.r, rfmt = _router_arg(router_w)
        self.b = None if bias is None else _f64(bias)
        m, h = self.xa.shape
        _, idx0, _ = route(self.xa, self.r, top_k, score, self.b, 0, self.lib)
        needed = sorted(set(int(v) for v in idx0.ravel()))
        self.needed = needed
        self.routed = _ExpertTable(self.r.shape[0], {e: expert_weights(e) for e in needed})
        self.shared = _ExpertTable(len(shared_weights), dict(enumerate(shared_weights)))
        any_w = expert_weights(needed[0])
        inter = _inter_of(any_w)
        self.shape = _Shape(h, inter, self.r.shape[0], top_k, len(shared_weights), m, score, rfmt,
                            float(routed_scale), 0)
        self.out = np.empty((m, h), np.float64)
        self.idx = np.empty((m, top_k), np.int64)
        self.w = np.empty((m, top_k), np.float64)

    def run(self, threads: int = 0):
        self.shape.threads = threads
        st = self.lib.moe_oracle_layer(ctypes.byref(self.shape), _ptr(self.xa), _ptr(self.ra), _ptr(self.r),
                                       _ptr(self.b), ctypes.byref(self.routed.struct),
                                       ctypes.byref(self.shared.struct), _ptr(self.out), _ptr(self.idx),
                                       _ptr(self.w), None)
        if st != 0:
            raise RuntimeError(f"moe_oracle_layer: status {st}")
        return self.out, self.idx, self.w
