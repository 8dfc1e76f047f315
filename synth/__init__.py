"""Seeded synthetic inputs for selected-attention backward workloads.

This module is the only thing the oracle and the GPU library share: it draws
the tensors both of them consume.  It holds none of the backward's arithmetic.

Workloads follow the five configurations the method is benchmarked on (tiny,
varlen TND, long context, max selection, small-group stress).  Values are
drawn with torch's seeded generators on the requested device and rounded
(round-to-nearest-even) to bf16 / fp16; index lists are distinct block ids per
(token, KV head), sorted ascending, drawn as the top-``count`` of seeded
uniform keys (a uniformly random subset).

attentionOut and the softmax stats are forward outputs, so they are not
drawn here: the caller runs a forward over the drawn q, k, v and index lists.
For the two small workloads that is the fp64 oracle forward ("oracle"); for
the three large ones it is the library's own forward ("gpu"), which the tests
check against the oracle forward on sampled rows before the backward uses it.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    cu_q: tuple
    cu_kv: tuple
    n1: int
    n2: int
    d_qk: int
    d_v: int
    dtype: str            # "bf16" | "f16"
    block_size: int
    block_count: int
    scale: float
    std: float            # standard deviation of q, k, v, dy
    topk: str             # "uniform" | "skewed"
    stats: str            # forward that produces O and the stats: "oracle" | "gpu"
    seed: int

    @property
    def batch(self) -> int:
        return len(self.cu_q) - 1

    @property
    def t1(self) -> int:
        return self.cu_q[-1]

    @property
    def t2(self) -> int:
        return self.cu_kv[-1]

    @property
    def group(self) -> int:
        return self.n1 // self.n2

    @property
    def selected_keys(self) -> int:
        return self.block_size * self.block_count

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    def flops(self) -> float:
        """2 * L * (3 * d_qk + 2 * d_v) per query head per token."""
        return 2.0 * self.selected_keys * (3 * self.d_qk + 2 * self.d_v) * self.t1 * self.n1

    def algorithmic_bytes(self) -> float:
        """Every input read once and every output written once."""
        e = 2
        t1, t2 = self.t1, self.t2
        q = t1 * self.n1 * self.d_qk * e
        o = dy = t1 * self.n1 * self.d_v * e
        stats = 2 * t1 * self.n1 * 8 * 4
        topk = t1 * self.n2 * self.block_count * 4
        k = t2 * self.n2 * self.d_qk * e
        v = t2 * self.n2 * self.d_v * e
        return float(2 * q + o + dy + stats + topk + 2 * k + 2 * v)

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


def _cu(lengths):
    out = [0]
    for s in lengths:
        out.append(out[-1] + s)
    return tuple(out)


WORKLOADS = [
    Workload("tiny", (0, 256), (0, 256), 4, 1, 192, 128, "bf16", 16, 4, 1 / math.sqrt(192), 1.0,
             "uniform", "oracle", 20260000),
    Workload("varlen", (0, 1024, 4096), (0, 1024, 4096), 16, 1, 192, 128, "bf16", 64, 16,
             1 / math.sqrt(192), 1.0, "uniform", "oracle", 20260001),
    Workload("long_context", (0, 32768), (0, 32768), 64, 4, 192, 128, "bf16", 64, 16,
             1 / math.sqrt(192), 1.0, "uniform", "gpu", 20260002),
    Workload("max_selection", _cu([65536] * 4), _cu([65536] * 4), 128, 4, 192, 128, "bf16", 128, 63,
             1 / math.sqrt(192), 1.0, "uniform", "gpu", 20260003),
    Workload("small_group", _cu([16384] * 2), _cu([16384] * 2), 8, 8, 128, 128, "f16", 16, 128,
             1 / math.sqrt(128), math.sqrt(0.5), "skewed", "gpu", 20260004),
]


def _normal(shape, std, dtype, gen, device, chunk_rows=1 << 20):
    """N(0, std^2) rounded to dtype, drawn in row chunks (bounded temporaries)."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        x = torch.randn((r1 - r0, flat.shape[1]), generator=gen, device=device, dtype=torch.float32)
        flat[r0:r1] = (x * std).to(dtype)
    return out


def _distinct_sorted(nrows, n_out, n_from, gen, device, chunk_rows):
    """Per row: n_out distinct ids uniform over [0, n_from), sorted ascending."""
    out = torch.empty((nrows, n_out), dtype=torch.int32, device=device)
    for r0 in range(0, nrows, chunk_rows):
        r1 = min(nrows, r0 + chunk_rows)
        keys = torch.rand((r1 - r0, n_from), generator=gen, device=device)
        ids = torch.topk(keys, n_out, dim=1).indices
        out[r0:r1] = torch.sort(ids, dim=1).values.to(torch.int32)
    return out


def make_topk(w: Workload, gen, device) -> torch.Tensor:
    """topkIndices [T1, n2, block_count] int32 with batch-local block ids."""
    topk = torch.empty((w.t1, w.n2, w.block_count), dtype=torch.int32, device=device)
    for b in range(w.batch):
        q0, q1 = w.cu_q[b], w.cu_q[b + 1]
        nblk = (w.cu_kv[b + 1] - w.cu_kv[b]) // w.block_size
        rows = (q1 - q0) * w.n2
        if rows == 0:
            continue
        chunk = max(1, (1 << 28) // max(1, nblk * 4))
        if w.topk == "uniform":
            ids = _distinct_sorted(rows, w.block_count, nblk, gen, device, chunk)
        elif w.topk == "skewed":
            # a seeded quarter of the blocks is "hot"; each row takes 3/4 of its
            # ids from the hot set and 1/4 from the rest, so 75 % of all
            # selections land on 25 % of the blocks
            perm = torch.randperm(nblk, generator=gen, device=device).to(torch.int32)
            n_hot = nblk // 4
            hot, cold = perm[:n_hot], perm[n_hot:]
            k_hot = (w.block_count * 3) // 4
            k_cold = w.block_count - k_hot
            ih = _distinct_sorted(rows, k_hot, n_hot, gen, device, chunk)
            ic = _distinct_sorted(rows, k_cold, nblk - n_hot, gen, device, chunk)
            ids = torch.cat([hot[ih.long()], cold[ic.long()]], dim=1)
            ids = torch.sort(ids, dim=1).values
        else:
            raise ValueError(w.topk)
        topk[q0:q1] = ids.view(q1 - q0, w.n2, w.block_count)
    return topk


def make_inputs(w: Workload, device="cpu", seed: int | None = None) -> dict:
    """q, k, v, dy and topk; attentionOut and the stats come from a forward."""
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    dt = w.torch_dtype
    return {
        "q": _normal((w.t1, w.n1, w.d_qk), w.std, dt, gen, device),
        "k": _normal((w.t2, w.n2, w.d_qk), w.std, dt, gen, device),
        "v": _normal((w.t2, w.n2, w.d_v), w.std, dt, gen, device),
        "dy": _normal((w.t1, w.n1, w.d_v), w.std, dt, gen, device),
        "topk": make_topk(w, gen, device),
    }


# ------------------------------------------------------------ lightning indexer
@dataclass(frozen=True)
class IndexerWorkload:
    """A lightning-indexer backward problem: query [T1, n1, d], key [T2, n2, d],
    weights [T1, n1], indices / dy [T1, n2, topk] (dy fp32)."""
    name: str
    cu_q: tuple
    cu_kv: tuple
    n1: int
    n2: int
    d: int
    topk: int
    dtype: str
    empty_frac: float     # fraction of slots set to -1 (empty)
    seed: int

    @property
    def batch(self) -> int:
        return len(self.cu_q) - 1

    @property
    def t1(self) -> int:
        return self.cu_q[-1]

    @property
    def t2(self) -> int:
        return self.cu_kv[-1]

    @property
    def group(self) -> int:
        return self.n1 // self.n2

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    def flops(self) -> float:
        """Three contractions of 2 * d flops per (query head, selected key):
        scores, dQ and dK."""
        return 3 * 2.0 * self.d * self.topk * self.t1 * self.n1

    def with_(self, **kw) -> "IndexerWorkload":
        d = dict(self.__dict__)
        d.update(kw)
        return IndexerWorkload(**d)


INDEXER_WORKLOADS = [
    IndexerWorkload("indexer_tiny", (0, 256), (0, 256), 16, 1, 128, 64, "bf16", 0.0, 20261000),
    IndexerWorkload("indexer_varlen", (0, 300, 1000), (0, 300, 1000), 32, 1, 128, 128, "f16", 0.05, 20261001),
    IndexerWorkload("indexer_long", (0, 8192), (0, 8192), 64, 1, 128, 2048, "bf16", 0.0, 20261002),
]


def make_indexer_inputs(w: IndexerWorkload, device="cpu", seed: int | None = None) -> dict:
    """q, k, weights ~ N(0, 1) rounded to the dtype; dy ~ N(0, 1) fp32; per
    (token, key head) topk distinct key positions of the token's batch, sorted,
    a seeded fraction of slots then set to -1 (empty)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    dt = w.torch_dtype
    x = {
        "q": _normal((w.t1, w.n1, w.d), 1.0, dt, gen, device),
        "k": _normal((w.t2, w.n2, w.d), 1.0, dt, gen, device),
        "w": _normal((w.t1, w.n1), 1.0, dt, gen, device),
        "dy": torch.randn((w.t1, w.n2, w.topk), generator=gen, device=device, dtype=torch.float32),
    }
    idx = torch.full((w.t1, w.n2, w.topk), -1, dtype=torch.int32, device=device)
    for b in range(w.batch):
        q0, q1 = w.cu_q[b], w.cu_q[b + 1]
        s2 = w.cu_kv[b + 1] - w.cu_kv[b]
        rows = (q1 - q0) * w.n2
        if rows == 0:
            continue
        chunk = max(1, (1 << 28) // max(1, s2 * 4))
        idx[q0:q1] = _distinct_sorted(rows, w.topk, s2, gen, device, chunk).view(q1 - q0, w.n2, w.topk)
    if w.empty_frac > 0:
        drop = torch.rand((w.t1, w.n2, w.topk), generator=gen, device=device) < w.empty_frac
        idx = torch.where(drop, torch.full_like(idx, -1), idx)
    x["idx"] = idx
    return x
