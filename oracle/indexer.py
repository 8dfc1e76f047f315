"""fp64 CPU oracle for the lightning-indexer backward -- TEST INFRASTRUCTURE.

Binding of ``indexer_oracle.c`` (built into the same ``liboracle.so`` as the
selected-attention oracle).  Only the tests, ``smoke()`` and the bench's CPU
baseline may use it.  What it follows: "aclnnLightningIndexerGrad", formula
section (S = Relu(Query . Gather(Key, Indices)), Y = Dy * Weights,
dW = Reduce(S * dy), dQ = ReluGrad(Y, S) . Gather(Key, Indices),
dK = ScatterAdd(ReluGrad(Y, S)^T . Q, Indices)); the readings taken where the
page is silent are listed at the top of the C file.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np

from . import _load, as_array, _Tensor, F64

OK, EARG, EINDEX = 0, -1, -2


class _Lio(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("n1", ctypes.c_int32), ("n2", ctypes.c_int32), ("d", ctypes.c_int32),
        ("topk", ctypes.c_int32), ("layout", ctypes.c_int32), ("s1_max", ctypes.c_int32),
        ("s2_max", ctypes.c_int32), ("cu_q", ctypes.c_void_p), ("cu_kv", ctypes.c_void_p),
        ("idx", ctypes.c_void_p), ("q", _Tensor), ("k", _Tensor), ("w", _Tensor), ("dy", _Tensor),
    ]


@dataclass
class Problem:
    """One lightning-indexer backward problem (host arrays).

    query [T1, n1, d], key [T2, n2, d], weights [T1, n1], indices and dy
    [T1, n2, topk]; T1 / T2 are the rows of the query / key axis (packed TND,
    or BSND padded to s1_max / s2_max rows per batch, layout = 1).
    """
    cu_q: np.ndarray
    cu_kv: np.ndarray
    n1: int
    n2: int
    d: int
    topk: int
    idx: np.ndarray
    q: object
    k: object
    w: object
    dy: object
    kind: str | None = None
    layout: int = 0
    s1_max: int = 0
    s2_max: int = 0

    @property
    def batch(self) -> int:
        return len(self.cu_q) - 1

    @property
    def t1(self) -> int:
        return self.batch * self.s1_max if self.layout else int(self.cu_q[-1])

    @property
    def t2(self) -> int:
        return self.batch * self.s2_max if self.layout else int(self.cu_kv[-1])

    def _c(self):
        keep = []

        def arr(x, dt):
            a = np.ascontiguousarray(x, dtype=dt)
            keep.append(a)
            return a.ctypes.data

        def ten(x):
            a, code = as_array(x, self.kind)
            keep.append(a)
            return _Tensor(a.ctypes.data, code, 0)

        c = _Lio(batch=self.batch, n1=self.n1, n2=self.n2, d=self.d, topk=self.topk, layout=int(self.layout),
                 s1_max=int(self.s1_max), s2_max=int(self.s2_max), cu_q=arr(self.cu_q, np.int32),
                 cu_kv=arr(self.cu_kv, np.int32), idx=arr(self.idx, np.int32), q=ten(self.q), k=ten(self.k),
                 w=ten(self.w), dy=ten(self.dy))
        return c, keep


def _lib():
    lib = _load()
    if not getattr(lib, "_lio_ready", False):
        P, dp = ctypes.POINTER(_Lio), ctypes.c_void_p
        lib.lio_backward.argtypes = [P, dp, dp, dp]
        lib.lio_backward_range.argtypes = [P, ctypes.c_int64, ctypes.c_int64, dp, dp, dp]
        lib.lio_backward_range.restype = ctypes.c_int
        lib.lio_scores.argtypes = [P, dp]
        lib.lio_q_rows.argtypes = [P, ctypes.c_int64, dp, dp, dp]
        lib.lio_k_rows.argtypes = [P, ctypes.c_int64, dp, dp, dp]
        for f in (lib.lio_backward, lib.lio_scores, lib.lio_q_rows, lib.lio_k_rows):
            f.restype = ctypes.c_int
        lib._lio_ready = True
    return lib


def _check(rc, what):
    if rc != OK:
        raise RuntimeError(f"indexer oracle {what} failed with status {rc}")


def backward(p: Problem):
    """Full fp64 (dq [T1,n1,d], dk [T2,n2,d], dw [T1,n1])."""
    dq = np.zeros((p.t1, p.n1, p.d))
    dk = np.zeros((p.t2, p.n2, p.d))
    dw = np.zeros((p.t1, p.n1))
    c, _keep = p._c()
    _check(_lib().lio_backward(ctypes.byref(c), dq.ctypes.data, dk.ctypes.data, dw.ctypes.data), "backward")
    return dq, dk, dw


def backward_range(p: Problem, t_lo: int, t_hi: int):
    """The backward of the query rows [t_lo, t_hi) only (dk holds their
    contributions); the ranges of a partition sum to ``backward``."""
    dq = np.zeros((p.t1, p.n1, p.d))
    dk = np.zeros((p.t2, p.n2, p.d))
    dw = np.zeros((p.t1, p.n1))
    c, _keep = p._c()
    _check(_lib().lio_backward_range(ctypes.byref(c), int(t_lo), int(t_hi), dq.ctypes.data, dk.ctypes.data,
                                     dw.ctypes.data), "backward_range")
    return dq, dk, dw


def scores(p: Problem):
    """Index scores of the selected positions [T1, n2, topk] (the forward)."""
    out = np.zeros((p.t1, p.n2, p.topk))
    c, _keep = p._c()
    _check(_lib().lio_scores(ctypes.byref(c), out.ctypes.data), "scores")
    return out


def q_rows(p: Problem, tokens):
    """dQ [n, n1, d] and dW [n, n1] of the query rows `tokens`."""
    t = np.ascontiguousarray(np.asarray(tokens, np.int64))
    dq = np.zeros((len(t), p.n1, p.d))
    dw = np.zeros((len(t), p.n1))
    c, _keep = p._c()
    _check(_lib().lio_q_rows(ctypes.byref(c), len(t), t.ctypes.data, dq.ctypes.data, dw.ctypes.data), "q_rows")
    return dq, dw


def k_rows(p: Problem, key_rows, heads):
    """dK [n, d] of the key rows (key_rows[i], key head heads[i])."""
    r = np.ascontiguousarray(np.asarray(key_rows, np.int64))
    h = np.ascontiguousarray(np.asarray(heads, np.int32))
    dk = np.zeros((len(r), p.d))
    c, _keep = p._c()
    _check(_lib().lio_k_rows(ctypes.byref(c), len(r), r.ctypes.data, h.ctypes.data, dk.ctypes.data), "k_rows")
    return dk
