"""Helpers for the parity tests: inputs, oracle fan-out, tolerance checks.

The oracle itself is single-threaded; for the larger parity cases its rows
are split over a pool of threads (each C call runs without the GIL).  Only
slicing and copying happen here: every number the tests compare against comes
from ``oracle/``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import torch

import oracle
import synth

# spec tolerance per output tensor for 16-bit outputs
REL_FRO = 5e-3
MAX_ABS_FRAC = 2e-2


def workers() -> int:
    return max(1, os.cpu_count() or 1)


def to_np16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def problem(w: synth.Workload, x: dict, stat_stride: int = 8, with_backward: bool = True) -> oracle.Problem:
    """oracle.Problem over host copies of the workload's tensors."""
    return oracle.Problem(
        cu_q=np.asarray(w.cu_q, np.int32), cu_kv=np.asarray(w.cu_kv, np.int32), n1=w.n1, n2=w.n2,
        d_qk=w.d_qk, d_v=w.d_v, block_size=w.block_size, block_count=w.block_count, scale=w.scale,
        topk=x["topk"].cpu().numpy(), q=to_np16(x["q"]), k=to_np16(x["k"]), v=to_np16(x["v"]),
        o=to_np16(x["o"]) if with_backward else None, dy=to_np16(x["dy"]),
        smax=x["softmax_max"].cpu().numpy() if with_backward else None,
        ssum=x["softmax_sum"].cpu().numpy() if with_backward else None,
        stat_stride=stat_stride, kind=w.dtype)


# ---------------------------------------------------------------- fan-out
# The oracle's C functions keep no global state and ctypes releases the GIL
# for the length of each call, so one process spreads the rows over threads:
# no worker start-up, no copies of the problem.
_EXEC = None


def _executor():
    global _EXEC
    if _EXEC is None:
        _EXEC = cf.ThreadPoolExecutor(max_workers=workers())
    return _EXEC


def _chunks(rows, n):
    return [c for c in np.array_split(np.asarray(rows, np.int64), max(1, n * 4)) if len(c)]


def par_forward_rows(p: oracle.Problem, rows, n=None):
    n = n or workers()
    parts = list(_executor().map(lambda r: oracle.forward_rows(p, r), _chunks(rows, n)))
    return (np.concatenate([a for a, _, _ in parts]), np.concatenate([b for _, b, _ in parts]),
            np.concatenate([c for _, _, c in parts]))


def par_dq_rows(p: oracle.Problem, rows, n=None):
    n = n or workers()
    return np.concatenate(list(_executor().map(lambda r: oracle.dq_rows(p, r), _chunks(rows, n))))


def par_dkdv_blocks(p: oracle.Problem, blocks, n=None):
    return list(_executor().map(lambda a: oracle.dkdv_block(p, *a), list(blocks)))


def par_dkdv_block(p: oracle.Problem, b: int, n2: int, kb: int, n=None):
    """One key block, its batch's query tokens split over the workers; the
    partial sums (each a plain oracle result) are added in fp64."""
    n = n or workers()
    q0, q1 = int(p.cu_q[b]), int(p.cu_q[b + 1])
    edges = np.linspace(q0, q1, n * 4 + 1).astype(np.int64)
    tasks = [(b, n2, kb, int(a), int(c)) for a, c in zip(edges[:-1], edges[1:]) if c > a]
    parts = list(_executor().map(lambda a: oracle.dkdv_block_range(p, *a), tasks))
    return sum(a for a, _ in parts), sum(c for _, c in parts)


def oracle_full_forward(w: synth.Workload, x: dict):
    """Oracle forward of every row: O [T1, n1, d_v], max and sum [T1, n1]."""
    p = problem(w, x, with_backward=False)
    o, m, l = par_forward_rows(p, np.arange(w.t1 * w.n1))
    return o.reshape(w.t1, w.n1, w.d_v), m.reshape(w.t1, w.n1), l.reshape(w.t1, w.n1)


def oracle_full_backward(w: synth.Workload, x: dict):
    """Oracle dq, dk, dv of the whole problem (rows and key blocks fanned out)."""
    p = problem(w, x)
    dq = par_dq_rows(p, np.arange(w.t1 * w.n1)).reshape(w.t1, w.n1, w.d_qk)
    blocks = [(b, j, kb) for b in range(w.batch) for j in range(w.n2)
              for kb in range((w.cu_kv[b + 1] - w.cu_kv[b]) // w.block_size)]
    dk = np.zeros((w.t2, w.n2, w.d_qk))
    dv = np.zeros((w.t2, w.n2, w.d_v))
    for (b, j, kb), (bk, bv) in zip(blocks, par_dkdv_blocks(p, blocks)):
        r0 = w.cu_kv[b] + kb * w.block_size
        dk[r0:r0 + w.block_size, j] = bk
        dv[r0:r0 + w.block_size, j] = bv
    return dq, dk, dv


# ------------------------------------------------------------------ inputs
def forward_inputs(w: synth.Workload, x: dict) -> dict:
    """attentionOut and [T1,N1,8] stats from the oracle forward (host)."""
    p = problem(w, x, with_backward=False)
    o, m, l = par_forward_rows(p, np.arange(w.t1 * w.n1))
    x = dict(x)
    x["o"] = torch.from_numpy(o.reshape(w.t1, w.n1, w.d_v)).to(w.torch_dtype)
    x["softmax_max"] = torch.from_numpy(m).float().view(w.t1, w.n1, 1).expand(-1, -1, 8).contiguous()
    x["softmax_sum"] = torch.from_numpy(l).float().view(w.t1, w.n1, 1).expand(-1, -1, 8).contiguous()
    return x


def workload_inputs(w: synth.Workload, device="cpu") -> dict:
    x = synth.make_inputs(w, device=device)
    if w.stats == "oracle":
        x = forward_inputs(w, {k: v.cpu() for k, v in x.items()})
    return x


def gpu_forward_inputs(w: synth.Workload, x: dict) -> dict:
    """attentionOut and [T1,N1,8] stats from the library's forward (device);
    the tests compare them with the oracle forward on the rows they sample."""
    import sparse_attention_backward_gb300 as sab
    o, m, l = sab.forward(x["q"], x["k"], x["v"], x["topk"], w.cu_q, w.cu_kv, w.scale, w.block_size,
                          w.block_count, check=True)
    return dict(x, o=o, softmax_max=m, softmax_sum=l)


def sub_problem(w: synth.Workload, x: dict, b: int, n2: int, tokens) -> oracle.Problem:
    """One batch, one KV head, a subset of its query tokens (row order kept).

    Its gradients equal the full problem's on those rows: every quantity of a
    query row depends only on that row and on its batch's key rows.
    """
    G = w.group
    t = torch.as_tensor(np.asarray(tokens, np.int64), device=x["q"].device)
    k0, k1 = w.cu_kv[b], w.cu_kv[b + 1]
    hs = slice(n2 * G, (n2 + 1) * G)
    sub = {
        "q": x["q"][t][:, hs], "dy": x["dy"][t][:, hs], "o": x["o"][t][:, hs],
        "softmax_max": x["softmax_max"][t][:, hs], "softmax_sum": x["softmax_sum"][t][:, hs],
        "topk": x["topk"][t][:, n2:n2 + 1], "k": x["k"][k0:k1, n2:n2 + 1], "v": x["v"][k0:k1, n2:n2 + 1],
    }
    sw = w.with_(cu_q=(0, len(tokens)), cu_kv=(0, k1 - k0), n1=G, n2=1)
    return problem(sw, sub)


def selecting_tokens(w: synth.Workload, x: dict, b: int, n2: int, kb: int) -> np.ndarray:
    q0, q1 = w.cu_q[b], w.cu_q[b + 1]
    hit = (x["topk"][q0:q1, n2] == kb).any(-1)
    return (torch.nonzero(hit).view(-1) + q0).cpu().numpy()


# --------------------------------------------------------------- tolerance
def metrics(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    nrm = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / nrm if nrm > 0 else np.linalg.norm(got - ref)
    mx = np.max(np.abs(ref)) if ref.size else 0.0
    err = np.max(np.abs(got - ref)) if ref.size else 0.0
    return rel, err, mx


def assert_close(name, got, ref):
    rel, err, mx = metrics(got, ref)
    assert np.all(np.isfinite(got)), f"{name}: non-finite output"
    assert rel <= REL_FRO, f"{name}: relative Frobenius error {rel:.3e} > {REL_FRO}"
    assert err <= MAX_ABS_FRAC * mx + 1e-30, f"{name}: max abs error {err:.3e} > {MAX_ABS_FRAC} * {mx:.3e}"
    return rel, err / mx if mx else 0.0


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()
