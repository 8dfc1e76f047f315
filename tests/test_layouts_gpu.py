"""GPU parity of the other layouts the pages describe.

* Rope split ("aclnnFlashAttentionUnpaddingScoreGradV3", formula section:
  Q = [query, queryRope], K = [key, keyRope]; dqRope = dS kRope / sqrt(d),
  dkRope = dS^T qRope / sqrt(d)): the 192-wide heads are passed as 128 + 64
  columns in separate tensors.  The oracle runs the concatenated problem and
  its dQ / dK are compared column slice by column slice.
* BSND ("aclnnLightningIndexerGrad": TND or BSND layouts; the
  "NsaSelectedAttentionGrad" README's calling section has a non-TND sample):
  every batch padded to S1 / S2 rows.  Padding rows hold junk, their index
  lists block ids far out of range (a read of them would be reported); the
  oracle runs the same padded tensors in its BSND mode, and padding rows
  must come back as exact zeros.
Tolerance per output tensor: relative Frobenius error <= 5e-3 and max abs
error <= 2e-2 * max|ref|.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_backward_gb300 as sab
import synth
from tests import _support as S
from tests.test_parity_gpu import SMALL

pytestmark = pytest.mark.gpu

ROPE_CASES = ["tiny", "varlen", "g32_bs128", "bs16_cnt127"]


@pytest.fixture(scope="module")
def rope_data():
    cache = {}

    def get(name):
        if name not in cache:
            w = SMALL[name]
            x = S.workload_inputs(w, "cpu")
            cache[name] = (w, x, S.oracle_full_backward(w, x), S.oracle_full_forward(w, x))
        return cache[name]
    return get


def _split(t):
    return t[..., :128].contiguous(), t[..., 128:].contiguous()


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("name", ROPE_CASES)
def test_rope_split_backward(rope_data, name, deterministic):
    w, x, (rdq, rdk, rdv), _ = rope_data(name)
    t = {k: v.cuda() for k, v in x.items()}
    q, qr = _split(t["q"])
    k, kr = _split(t["k"])
    dq, dk, dv, dqr, dkr = sab.backward(q, k, t["v"], t["o"], t["dy"], t["softmax_max"], t["softmax_sum"],
                                        t["topk"], w.cu_q, w.cu_kv, w.scale, w.block_size, w.block_count,
                                        deterministic=deterministic, check=True, q_rope=qr, k_rope=kr)
    assert dq.shape[-1] == 128 and dqr.shape[-1] == 64
    S.assert_close(f"{name} dq", S.f64(dq), rdq[..., :128])
    S.assert_close(f"{name} dq_rope", S.f64(dqr), rdq[..., 128:])
    S.assert_close(f"{name} dk", S.f64(dk), rdk[..., :128])
    S.assert_close(f"{name} dk_rope", S.f64(dkr), rdk[..., 128:])
    S.assert_close(f"{name} dv", S.f64(dv), rdv)


@pytest.mark.parametrize("name", ["varlen", "g32_bs128"])
def test_rope_split_chunked_deterministic_is_bitwise_stable(rope_data, name, monkeypatch):
    monkeypatch.setenv("SELATTN_DS_CHUNK_TOKENS", "7" if name == "g32_bs128" else "1000")
    w, x, (rdq, rdk, rdv), _ = rope_data(name)
    t = {k: v.cuda() for k, v in x.items()}
    q, qr = _split(t["q"])
    k, kr = _split(t["k"])
    run = lambda: sab.backward(q, k, t["v"], t["o"], t["dy"], t["softmax_max"], t["softmax_sum"], t["topk"],
                               w.cu_q, w.cu_kv, w.scale, w.block_size, w.block_count, deterministic=True,
                               check=True, q_rope=qr, k_rope=kr)
    a, b = run(), run()
    S.assert_close(f"{name} chunks dq_rope", S.f64(a[3]), rdq[..., 128:])
    S.assert_close(f"{name} chunks dk_rope", S.f64(a[4]), rdk[..., 128:])
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.int16), v.view(torch.int16))


@pytest.mark.parametrize("name", ROPE_CASES)
def test_rope_split_forward(rope_data, name):
    w, x, _, (ro, rm, rl) = rope_data(name)
    t = {k: v.cuda() for k, v in x.items()}
    q, qr = _split(t["q"])
    k, kr = _split(t["k"])
    o, m, l = sab.forward(q, k, t["v"], t["topk"], w.cu_q, w.cu_kv, w.scale, w.block_size, w.block_count,
                          check=True, q_rope=qr, k_rope=kr)
    S.assert_close(f"{name} rope attention_out", S.f64(o), ro)
    S.assert_close(f"{name} rope softmax_max", m[..., 0].double().cpu().numpy(), rm)
    S.assert_close(f"{name} rope softmax_sum", l[..., 0].double().cpu().numpy(), rl)


# ------------------------------------------------------------------- BSND
def _pad(x, cu, smax, junk):
    """[T, ...] packed -> [B, smax, ...] with junk in the padding rows."""
    B = len(cu) - 1
    out = junk((B, smax) + tuple(x.shape[1:]), x.dtype)
    for b in range(B):
        out[b, :cu[b + 1] - cu[b]] = x[cu[b]:cu[b + 1]]
    return out.contiguous()


def _bsnd_case(name, s1_extra, s2_extra, seed):
    """A small workload in BSND: inputs, forward outputs from the oracle in
    its BSND mode, and the padded problem the oracle runs."""
    w = SMALL[name]
    x = synth.make_inputs(w)
    g = torch.Generator().manual_seed(seed)

    def junk(shape, dt):
        if dt == torch.int32:
            return torch.full(shape, 10 ** 6, dtype=dt)
        return (torch.randn(shape, generator=g) * 5).to(dt)
    s1 = max(np.diff(w.cu_q)) + s1_extra
    s2 = max(np.diff(w.cu_kv)) + s2_extra
    xb = {k: _pad(v, w.cu_q if k in ("q", "dy", "topk") else w.cu_kv, s1 if k in ("q", "dy", "topk") else s2, junk)
          for k, v in x.items()}

    def problem(xs, with_backward=True):
        flat = lambda t: S.to_np16(t) if t.dtype != torch.float32 else t.numpy()
        return oracle.Problem(
            cu_q=np.asarray(w.cu_q, np.int32), cu_kv=np.asarray(w.cu_kv, np.int32), n1=w.n1, n2=w.n2,
            d_qk=w.d_qk, d_v=w.d_v, block_size=w.block_size, block_count=w.block_count, scale=w.scale,
            topk=xs["topk"].numpy(), q=flat(xs["q"]), k=flat(xs["k"]), v=flat(xs["v"]), dy=flat(xs["dy"]),
            o=flat(xs["o"]) if with_backward else None, smax=xs["softmax_max"].numpy() if with_backward else None,
            ssum=xs["softmax_sum"].numpy() if with_backward else None, kind=w.dtype, layout=1, s1_max=s1,
            s2_max=s2)
    # forward outputs over the padded rows (zeros on padding rows), as the op would be given them
    p = problem(xb, with_backward=False)
    rows = np.concatenate([np.arange(b * s1 + 0, b * s1 + w.cu_q[b + 1] - w.cu_q[b])
                           for b in range(w.batch)]).astype(np.int64)
    B = w.batch
    o = torch.zeros((B, s1, w.n1, w.d_v), dtype=w.torch_dtype)
    m = torch.zeros((B, s1, w.n1, 8))
    l = torch.zeros((B, s1, w.n1, 8))
    if rows.size:
        fo, fm, fl = S.par_forward_rows(p, (rows[:, None] * w.n1 + np.arange(w.n1)).reshape(-1))
        idx = torch.as_tensor(rows)
        o.view(-1, w.n1, w.d_v)[idx] = torch.from_numpy(fo.reshape(-1, w.n1, w.d_v)).to(w.torch_dtype)
        m.view(-1, w.n1, 8)[idx] = torch.from_numpy(fm.reshape(-1, w.n1, 1)).float().expand(-1, -1, 8)
        l.view(-1, w.n1, 8)[idx] = torch.from_numpy(fl.reshape(-1, w.n1, 1)).float().expand(-1, -1, 8)
    xb.update(o=o, softmax_max=m, softmax_sum=l)
    return w, xb, s1, s2, problem(xb), (o, m, l)


@pytest.fixture(scope="module")
def bsnd_data():
    cache = {}

    def get(name):
        if name not in cache:
            w, xb, s1, s2, p, fwd = _bsnd_case(name, s1_extra=5, s2_extra=2 * SMALL[name].block_size, seed=41)
            dq, dk, dv = oracle.backward(p) if p.t1 * p.n1 < 20000 else _par_backward(p, w, s1, s2)
            cache[name] = (w, xb, s1, s2, (dq, dk, dv), fwd)
        return cache[name]
    return get


def _par_backward(p, w, s1, s2):
    """oracle.backward of a BSND problem with its rows and blocks fanned out."""
    rows = np.concatenate([np.arange(b * s1, b * s1 + w.cu_q[b + 1] - w.cu_q[b]) for b in range(w.batch)])
    dq = np.zeros((p.t1, w.n1, w.d_qk))
    flat = (rows[:, None] * w.n1 + np.arange(w.n1)).reshape(-1)
    dq.reshape(-1, w.d_qk)[flat] = S.par_dq_rows(p, flat)
    blocks = [(b, j, kb) for b in range(w.batch) for j in range(w.n2)
              for kb in range((w.cu_kv[b + 1] - w.cu_kv[b]) // w.block_size)]
    dk = np.zeros((p.t2, w.n2, w.d_qk))
    dv = np.zeros((p.t2, w.n2, w.d_v))
    for (b, j, kb), (bk, bv) in zip(blocks, S.par_dkdv_blocks(p, blocks)):
        r0 = b * s2 + kb * w.block_size
        dk[r0:r0 + w.block_size, j] = bk
        dv[r0:r0 + w.block_size, j] = bv
    return dq, dk, dv


BSND_CASES = ["ragged_fp16", "varlen", "g32_bs128"]


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("name", BSND_CASES)
def test_bsnd_backward(bsnd_data, name, deterministic):
    w, xb, s1, s2, (rdq, rdk, rdv), _ = bsnd_data(name)
    t = {k: v.cuda() for k, v in xb.items()}
    dq, dk, dv = sab.backward(t["q"], t["k"], t["v"], t["o"], t["dy"], t["softmax_max"], t["softmax_sum"], t["topk"],
                              w.cu_q, w.cu_kv, w.scale, w.block_size, w.block_count, deterministic=deterministic,
                              check=True)
    assert dq.shape == (w.batch, s1, w.n1, w.d_qk) and dk.shape == (w.batch, s2, w.n2, w.d_qk)
    S.assert_close(f"{name} bsnd dq", S.f64(dq).reshape(rdq.shape), rdq)
    S.assert_close(f"{name} bsnd dk", S.f64(dk).reshape(rdk.shape), rdk)
    S.assert_close(f"{name} bsnd dv", S.f64(dv).reshape(rdv.shape), rdv)
    for b in range(w.batch):   # padding rows: exact zeros
        assert not S.f64(dq[b, w.cu_q[b + 1] - w.cu_q[b]:]).any()
        assert not S.f64(dk[b, w.cu_kv[b + 1] - w.cu_kv[b]:]).any()
        assert not S.f64(dv[b, w.cu_kv[b + 1] - w.cu_kv[b]:]).any()


@pytest.mark.parametrize("name", BSND_CASES)
def test_bsnd_forward(bsnd_data, name):
    w, xb, s1, s2, _, (ro, rm, rl) = bsnd_data(name)
    t = {k: v.cuda() for k, v in xb.items()}
    o, m, l = sab.forward(t["q"], t["k"], t["v"], t["topk"], w.cu_q, w.cu_kv, w.scale, w.block_size,
                          w.block_count, check=True)
    S.assert_close(f"{name} bsnd attention_out", S.f64(o), S.f64(ro))
    S.assert_close(f"{name} bsnd softmax_max", m.cpu().double().numpy(), rm.double().numpy())
    S.assert_close(f"{name} bsnd softmax_sum", l.cpu().double().numpy(), rl.double().numpy())
    for b in range(w.batch):   # padding rows: exact zeros
        n = w.cu_q[b + 1] - w.cu_q[b]
        assert not S.f64(o[b, n:]).any() and not m[b, n:].any() and not l[b, n:].any()


@pytest.mark.parametrize("slots", ["0", "1"])
def test_bsnd_with_rope_split_chunked_deterministic(bsnd_data, slots, monkeypatch):
    """Both at once, in the deterministic mode's chunked path, with dQ from
    the stored dS or from per-slot partials."""
    monkeypatch.setenv("SELATTN_DS_CHUNK_TOKENS", "900")
    monkeypatch.setenv("SELATTN_DQ_SLOTS", slots)
    w, xb, s1, s2, (rdq, rdk, rdv), _ = bsnd_data("varlen")
    t = {k: v.cuda() for k, v in xb.items()}
    q, qr = _split(t["q"])
    k, kr = _split(t["k"])
    dq, dk, dv, dqr, dkr = sab.backward(q, k, t["v"], t["o"], t["dy"], t["softmax_max"], t["softmax_sum"],
                                        t["topk"], w.cu_q, w.cu_kv, w.scale, w.block_size, w.block_count,
                                        deterministic=True, check=True, q_rope=qr, k_rope=kr)
    S.assert_close("bsnd rope dq", S.f64(dq).reshape(rdq[..., :128].shape), rdq[..., :128])
    S.assert_close("bsnd rope dq_rope", S.f64(dqr).reshape(rdq[..., 128:].shape), rdq[..., 128:])
    S.assert_close("bsnd rope dk", S.f64(dk).reshape(rdk[..., :128].shape), rdk[..., :128])
    S.assert_close("bsnd rope dk_rope", S.f64(dkr).reshape(rdk[..., 128:].shape), rdk[..., 128:])
    S.assert_close("bsnd rope dv", S.f64(dv).reshape(rdv.shape), rdv)
