"""fp64 CPU oracle for NSA selected-attention backward -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does: it has
no CPU path of any kind.

The arithmetic lives in ``selattn_oracle.c`` (plain single-threaded C, fp64
accumulation, no blocking or fusion); this module only compiles it with gcc and
marshals numpy arrays into it.  What each function follows on the pages:

* ``forward``     -- "aclnnFlashAttentionUnpaddingScoreGradV3", Formula
  (forward S, P, Y with no pse/mask/dropout) applied to the rows that the
  "NsaSelectedAttentionGrad" README's Gather formula selects; yields
  attentionOut and the softmaxMax / softmaxSum rows.
* ``backward``, ``dq_rows``, ``dkdv_block`` -- "NsaSelectedAttentionGrad"
  README, function description (dV = P^T dY, dQ = dS K / sqrt(d),
  dK = dS^T Q / sqrt(d) over the gathered rows, scatter-added back).
* ``oracle.indexer`` -- the lightning-indexer backward of the
  "aclnnLightningIndexerGrad" page (``indexer_oracle.c``).

Every function is pinned by tests that do not reuse its formulas: central
finite differences, torch fp64 autograd of the gathered and of the dense
attention, the dK / dV sum invariants and exhaustive 16-bit decoding checks.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "selattn_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "indexer_oracle.c")]
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

F64, BF16, F16, F32 = 0, 1, 2, 3
OK, EARG, EINDEX, ENOMEM = 0, -1, -2, -3


class _Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("pad_", ctypes.c_int32)]


class _Problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("n1", ctypes.c_int32), ("n2", ctypes.c_int32),
        ("d_qk", ctypes.c_int32), ("d_v", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("block_count", ctypes.c_int32), ("stat_stride", ctypes.c_int32), ("scale", ctypes.c_double),
        ("cu_q", ctypes.c_void_p), ("cu_kv", ctypes.c_void_p), ("topk", ctypes.c_void_p),
        ("q", _Tensor), ("k", _Tensor), ("v", _Tensor), ("o", _Tensor), ("dy", _Tensor),
        ("smax", _Tensor), ("ssum", _Tensor),
        ("layout", ctypes.c_int32), ("s1_max", ctypes.c_int32), ("s2_max", ctypes.c_int32),
        ("pad2_", ctypes.c_int32),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (host code only; same result on x86 and Arm)."""
    if (force or not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(f) for f in _SRCS)):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC",
                               "-o", tmp, *_SRCS, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER(_Problem)
        dp = ctypes.c_void_p
        lib.sao_forward.argtypes = [P, dp, dp, dp]
        lib.sao_forward_rows.argtypes = [P, ctypes.c_int64, dp, dp, dp, dp]
        lib.sao_backward.argtypes = [P, dp, dp, dp]
        lib.sao_dq_rows.argtypes = [P, ctypes.c_int64, dp, dp]
        lib.sao_dkdv_block.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp]
        lib.sao_dkdv_block_range.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int64, ctypes.c_int64, dp, dp]
        for f in (lib.sao_forward, lib.sao_forward_rows, lib.sao_backward, lib.sao_dq_rows, lib.sao_dkdv_block,
                  lib.sao_dkdv_block_range):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def as_array(x, kind: str | None = None):
    """Return (contiguous numpy array, oracle dtype code).

    Accepts numpy arrays or CPU torch tensors.  16-bit data is passed as raw
    bits; ``kind`` ("bf16" / "f16") names the format for uint16 numpy input.
    """
    if x is None:
        return None, F64
    if not isinstance(x, np.ndarray):  # torch tensor
        import torch
        t = x.detach().contiguous().cpu()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16), BF16
        if t.dtype == torch.float16:
            return t.view(torch.int16).numpy().view(np.uint16), F16
        x = t.numpy()
    x = np.ascontiguousarray(x)
    if x.dtype == np.float64:
        return x, F64
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.float16:
        return x.view(np.uint16), F16
    if x.dtype == np.uint16:
        if kind not in ("bf16", "f16"):
            raise ValueError("uint16 input needs kind='bf16' or 'f16'")
        return x, BF16 if kind == "bf16" else F16
    raise TypeError(f"unsupported oracle input dtype {x.dtype}")


@dataclass
class Problem:
    """One selected-attention problem (host arrays).

    Layout TND (0): rows of batch b are cu_q[b] .. cu_q[b+1]-1 (keys: cu_kv).
    Layout BSND (1): every batch padded to s1_max query / s2_max key rows,
    batch b starting at row b * s1_max (b * s2_max); cu_q / cu_kv then hold the
    prefix sums of the valid lengths.  The array shapes below use T1 / T2 for
    the rows of the query / key axis in either layout.
    """
    cu_q: np.ndarray
    cu_kv: np.ndarray
    n1: int
    n2: int
    d_qk: int
    d_v: int
    block_size: int
    block_count: int
    scale: float
    topk: object          # [T1, n2, block_count] int32
    q: object             # [T1, n1, d_qk]
    k: object             # [T2, n2, d_qk]
    v: object             # [T2, n2, d_v]
    o: object = None      # [T1, n1, d_v]
    dy: object = None     # [T1, n1, d_v]
    smax: object = None   # [T1, n1, stat_stride]
    ssum: object = None   # [T1, n1, stat_stride]
    stat_stride: int = 8
    kind: str | None = None   # "bf16"/"f16" when 16-bit data arrives as uint16
    layout: int = 0           # 0 TND, 1 BSND
    s1_max: int = 0           # BSND: padded query rows per batch
    s2_max: int = 0           # BSND: padded key rows per batch

    @property
    def batch(self) -> int:
        return len(self.cu_q) - 1

    @property
    def t1(self) -> int:
        """Rows of the query axis."""
        return self.batch * self.s1_max if self.layout else int(self.cu_q[-1])

    @property
    def t2(self) -> int:
        """Rows of the key axis."""
        return self.batch * self.s2_max if self.layout else int(self.cu_kv[-1])

    def _c(self):
        """(C struct, list of the arrays it points into).  The caller holds the
        list for the duration of the C call; nothing is stored on the object,
        so several threads may call into the oracle with one Problem."""
        keep = []

        def arr(x, dt=None):
            a = np.ascontiguousarray(x, dtype=dt) if dt else x
            keep.append(a)
            return a.ctypes.data

        def ten(x):
            a, code = as_array(x, self.kind)
            if a is None:
                return _Tensor(None, F64, 0)
            keep.append(a)
            return _Tensor(a.ctypes.data, code, 0)

        topk = self.topk
        if not isinstance(topk, np.ndarray):
            topk = topk.detach().cpu().numpy()
        c = _Problem(
            batch=self.batch, n1=self.n1, n2=self.n2, d_qk=self.d_qk, d_v=self.d_v,
            block_size=self.block_size, block_count=self.block_count,
            stat_stride=self.stat_stride, scale=float(self.scale),
            cu_q=arr(np.asarray(self.cu_q), np.int32), cu_kv=arr(np.asarray(self.cu_kv), np.int32),
            topk=arr(topk, np.int32),
            q=ten(self.q), k=ten(self.k), v=ten(self.v), o=ten(self.o), dy=ten(self.dy),
            smax=ten(self.smax), ssum=ten(self.ssum),
            layout=int(self.layout), s1_max=int(self.s1_max), s2_max=int(self.s2_max), pad2_=0,
        )
        return c, keep


def _check(rc: int, what: str):
    if rc != OK:
        raise RuntimeError(f"oracle {what} failed with status {rc}")


def forward(p: Problem):
    """attentionOut [T1,n1,d_v] and per-row softmax max / sum [T1,n1] (fp64)."""
    lib = _load()
    o = np.zeros((p.t1, p.n1, p.d_v))
    m = np.zeros((p.t1, p.n1))
    l = np.zeros((p.t1, p.n1))
    c, _keep = p._c()
    _check(lib.sao_forward(ctypes.byref(c), o.ctypes.data, m.ctypes.data, l.ctypes.data), "forward")
    return o, m, l


def forward_rows(p: Problem, rows_th):
    """Forward of the rows rows_th[i] = t * n1 + h: o [n, d_v], m [n], l [n]."""
    lib = _load()
    rows = np.ascontiguousarray(np.asarray(rows_th, dtype=np.int64))
    o = np.zeros((len(rows), p.d_v))
    m = np.zeros(len(rows))
    l = np.zeros(len(rows))
    c, _keep = p._c()
    _check(lib.sao_forward_rows(ctypes.byref(c), len(rows), rows.ctypes.data, o.ctypes.data,
                                m.ctypes.data, l.ctypes.data), "forward_rows")
    return o, m, l


def backward(p: Problem):
    """Full fp64 (dq, dk, dv)."""
    lib = _load()
    dq = np.zeros((p.t1, p.n1, p.d_qk))
    dk = np.zeros((p.t2, p.n2, p.d_qk))
    dv = np.zeros((p.t2, p.n2, p.d_v))
    c, _keep = p._c()
    _check(lib.sao_backward(ctypes.byref(c), dq.ctypes.data, dk.ctypes.data, dv.ctypes.data), "backward")
    return dq, dk, dv


def dq_rows(p: Problem, rows_th):
    """dQ of the rows rows_th[i] = t * n1 + h, shape [len(rows_th), d_qk]."""
    lib = _load()
    rows = np.ascontiguousarray(np.asarray(rows_th, dtype=np.int64))
    dq = np.zeros((len(rows), p.d_qk))
    c, _keep = p._c()
    _check(lib.sao_dq_rows(ctypes.byref(c), len(rows), rows.ctypes.data, dq.ctypes.data), "dq_rows")
    return dq


def dkdv_block(p: Problem, b: int, n2: int, kb: int):
    """dK [block_size, d_qk] and dV [block_size, d_v] of key block kb of (b, n2)."""
    lib = _load()
    dk = np.zeros((p.block_size, p.d_qk))
    dv = np.zeros((p.block_size, p.d_v))
    c, _keep = p._c()
    _check(lib.sao_dkdv_block(ctypes.byref(c), b, n2, kb, dk.ctypes.data, dv.ctypes.data), "dkdv_block")
    return dk, dv


def dkdv_block_range(p: Problem, b: int, n2: int, kb: int, t_lo: int, t_hi: int):
    """Contribution of query tokens [t_lo, t_hi) of batch b to key block kb."""
    lib = _load()
    dk = np.zeros((p.block_size, p.d_qk))
    dv = np.zeros((p.block_size, p.d_v))
    c, _keep = p._c()
    _check(lib.sao_dkdv_block_range(ctypes.byref(c), b, n2, kb, t_lo, t_hi, dk.ctypes.data,
                                    dv.ctypes.data), "dkdv_block_range")
    return dk, dv
