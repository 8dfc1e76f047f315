"""GPU parity of the lightning-indexer backward ("aclnnLightningIndexerGrad",
formula section) against the fp64 oracle.

Small workloads are compared in full (dq, dk, dweights), including empty
slots (-1), a position selected twice, the BSND layout with junk in every
padding row, and out-of-range ids reported; the long workload (8192 tokens,
64 heads, 2048 selections per token) at full size on sampled query rows (dq,
dweights) and sampled key rows (dk).  Tolerance per output tensor as for the
attention backward: relative Frobenius error <= 5e-3 and max abs error
<= 2e-2 * max|ref|.
"""
import numpy as np
import pytest
import torch

import oracle.indexer as li
import sparse_attention_backward_gb300 as sab
import synth
from tests import _support as S

pytestmark = pytest.mark.gpu


def _problem(w, x, layout=0, s1=0, s2=0):
    return li.Problem(cu_q=np.asarray(w.cu_q, np.int32), cu_kv=np.asarray(w.cu_kv, np.int32), n1=w.n1, n2=w.n2,
                      d=w.d, topk=w.topk, idx=x["idx"].cpu().numpy(), q=S.to_np16(x["q"]), k=S.to_np16(x["k"]),
                      w=S.to_np16(x["w"]), dy=x["dy"].cpu().numpy(), kind=w.dtype, layout=layout, s1_max=s1,
                      s2_max=s2)


def _oracle_full(p):
    """oracle backward with the query rows split over threads (fp64 sum of
    the dK contributions)."""
    edges = np.linspace(0, p.t1, 4 * S.workers() + 1).astype(np.int64)
    parts = list(S._executor().map(lambda ab: li.backward_range(p, int(ab[0]), int(ab[1])),
                                   [(a, b) for a, b in zip(edges[:-1], edges[1:]) if b > a]))
    return tuple(sum(x[i] for x in parts) for i in range(3))


def _run(w, x, check=True):
    t = {k: v.cuda() for k, v in x.items()}
    return sab.indexer_backward(t["q"], t["k"], t["w"], t["dy"], t["idx"], w.cu_q, w.cu_kv, check=check)


def _close(name, outs, refs):
    for nm, got, ref in zip(("dq", "dk", "dweights"), outs, refs):
        S.assert_close(f"{name} {nm}", S.f64(got).reshape(ref.shape), ref)


@pytest.mark.parametrize("idx", [0, 1])
def test_indexer_full_parity_small(idx):
    w = synth.INDEXER_WORKLOADS[idx]
    x = synth.make_indexer_inputs(w)
    _close(w.name, _run(w, x), _oracle_full(_problem(w, x)))


@pytest.mark.parametrize("shape", [
    # one query head per key head; 5 heads per key head; a single selection; 300 selections (three
    # chunks, the last one ragged) in fp16 with empty slots
    dict(name="indexer_g1", cu_q=(0, 90), cu_kv=(0, 200), n1=4, n2=4, topk=64, seed=31),
    dict(name="indexer_g5", cu_q=(0, 37, 100), cu_kv=(0, 150, 260), n1=10, n2=2, topk=96, seed=32),
    dict(name="indexer_topk1", cu_q=(0, 50), cu_kv=(0, 64), n1=16, n2=1, topk=1, seed=33),
    dict(name="indexer_topk300", cu_q=(0, 40), cu_kv=(0, 512), n1=8, n2=1, topk=300, kind="f16",
         empty_frac=0.1, seed=34),
])
def test_indexer_shapes(shape):
    shape = dict(shape)
    kind = shape.pop("kind", None)
    if kind is not None:
        shape["dtype"] = kind
    w = synth.INDEXER_WORKLOADS[0].with_(**shape)
    x = synth.make_indexer_inputs(w)
    _close(w.name, _run(w, x), _oracle_full(_problem(w, x)))


def test_indexer_position_selected_twice_and_two_key_heads():
    w = synth.INDEXER_WORKLOADS[0].with_(name="indexer_dup", cu_q=(0, 70, 130), cu_kv=(0, 96, 200), n1=32, n2=2,
                                         topk=40, seed=7)
    x = synth.make_indexer_inputs(w)
    x["idx"] = x["idx"].clone()
    x["idx"][:, :, 1] = x["idx"][:, :, 0]            # every list names its first position twice
    _close(w.name, _run(w, x), _oracle_full(_problem(w, x)))


def test_indexer_bsnd_with_junk_padding():
    w = synth.INDEXER_WORKLOADS[1]
    x = synth.make_indexer_inputs(w)
    s1, s2 = 760, 720
    g = torch.Generator().manual_seed(9)

    def pad(t, cu, smax, fill):
        out = fill((w.batch, smax) + tuple(t.shape[1:]), t.dtype)
        for b in range(w.batch):
            out[b, :cu[b + 1] - cu[b]] = t[cu[b]:cu[b + 1]]
        return out.contiguous()
    junk = lambda shape, dt: (torch.full(shape, 10 ** 6, dtype=dt) if dt == torch.int32
                              else (torch.randn(shape, generator=g) * 9).to(dt))
    xb = {k: pad(v, w.cu_q if k != "k" else w.cu_kv, s1 if k != "k" else s2, junk) for k, v in x.items()}
    outs = _run(w, xb)
    refs = _oracle_full(_problem(w, {k: v.reshape((-1,) + tuple(v.shape[2:])) for k, v in xb.items()}, 1, s1, s2))
    _close("indexer bsnd", outs, refs)
    for b in range(w.batch):
        n = w.cu_q[b + 1] - w.cu_q[b]
        assert not S.f64(outs[0][b, n:]).any() and not S.f64(outs[2][b, n:]).any()


def test_indexer_out_of_range_id_is_reported():
    w = synth.INDEXER_WORKLOADS[0]
    x = synth.make_indexer_inputs(w)
    x["idx"] = x["idx"].clone()
    x["idx"][3, 0, 5] = 256          # one past the batch's keys
    with pytest.raises(sab.SagError) as e:
        _run(w, x)
    assert e.value.status == sab.SAG_ERR_INDEX


def test_indexer_long_sampled():
    """8192 tokens x 64 heads x 2048 selections at full size: 128 sampled
    query rows (dq, dweights) and 64 sampled key rows (dk)."""
    w = synth.INDEXER_WORKLOADS[2]
    x = synth.make_indexer_inputs(w, device="cuda")
    dq, dk, dw = sab.indexer_backward(x["q"], x["k"], x["w"], x["dy"], x["idx"], w.cu_q, w.cu_kv, check=True)
    p = _problem(w, x)
    rng = np.random.default_rng(3)
    toks = np.sort(rng.choice(w.t1, 128, replace=False))
    parts = list(S._executor().map(lambda c: li.q_rows(p, c), np.array_split(toks, 4 * S.workers())))
    rdq = np.concatenate([a for a, _ in parts])
    rdw = np.concatenate([b for _, b in parts])
    ti = torch.as_tensor(toks, device=dq.device)
    S.assert_close("indexer long dq (sampled rows)", S.f64(dq[ti]), rdq)
    S.assert_close("indexer long dweights (sampled rows)", S.f64(dw[ti]), rdw)
    rows = np.sort(rng.choice(w.t2, 64, replace=False))
    rdk = np.concatenate(list(S._executor().map(lambda c: li.k_rows(p, c, np.zeros(len(c), np.int32)),
                                                np.array_split(rows, 4 * S.workers()))))
    S.assert_close("indexer long dk (sampled rows)", S.f64(dk[torch.as_tensor(rows, device=dk.device), 0]), rdk)
