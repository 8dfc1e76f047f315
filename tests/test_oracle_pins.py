"""Pins of the fp64 oracle against things other than itself (CPU only).

* central finite differences of L = sum(dY * O(Q, K, V)) (the backward is the
  gradient of the forward the op documentation states);
* torch fp64 autograd of the gathered attention, duplicates included (the
  gather's adjoint is a scatter-add);
* torch fp64 autograd of dense, unmasked attention when every block is
  selected ("aclnnFlashAttentionUnpaddingScoreGradV3" formulas, no pse, mask
  or dropout);
* the dK / dV sum invariants;
* exhaustive decoding of every bf16 and fp16 bit pattern;
* the stat-lane, list-order and index-range readings.
"""
import numpy as np
import pytest
import torch

import oracle


def _rand_problem(rng, lens_q=(5, 7), lens_kv=(32, 24), n1=4, n2=2, dqk=8, dv=6, bs=8, cnt=2,
                  scale=0.35, duplicates=False, order="sorted"):
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_kv = np.concatenate([[0], np.cumsum(lens_kv)]).astype(np.int32)
    t1, t2 = int(cu_q[-1]), int(cu_kv[-1])
    topk = np.zeros((t1, n2, cnt), np.int32)
    for b in range(len(lens_q)):
        nblk = lens_kv[b] // bs
        for t in range(cu_q[b], cu_q[b + 1]):
            for j in range(n2):
                if duplicates:
                    ids = rng.integers(0, nblk, cnt)
                else:
                    ids = rng.choice(nblk, cnt, replace=False)
                    ids = np.sort(ids) if order == "sorted" else ids
                topk[t, j] = ids
    q = rng.standard_normal((t1, n1, dqk))
    k = rng.standard_normal((t2, n2, dqk))
    v = rng.standard_normal((t2, n2, dv))
    dy = rng.standard_normal((t1, n1, dv))
    return oracle.Problem(cu_q=cu_q, cu_kv=cu_kv, n1=n1, n2=n2, d_qk=dqk, d_v=dv, block_size=bs,
                          block_count=cnt, scale=scale, topk=topk, q=q, k=k, v=v, dy=dy,
                          stat_stride=1)


def _with_forward(p):
    o, m, l = oracle.forward(p)
    p.o, p.smax, p.ssum = o, m[..., None].copy(), l[..., None].copy()
    return p


def _loss(p):
    o, _, _ = oracle.forward(p)
    return float(np.sum(o * p.dy))


def test_finite_differences():
    rng = np.random.default_rng(1)
    p = _with_forward(_rand_problem(rng, lens_q=(3, 4), lens_kv=(64, 48)))
    dq, dk, dv = oracle.backward(p)
    eps = 1e-6
    for name, grad in (("q", dq), ("k", dk), ("v", dv)):
        base = getattr(p, name)
        fd = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = base.copy(); plus[idx] += eps
            minus = base.copy(); minus[idx] -= eps
            setattr(p, name, plus); lp = _loss(p)
            setattr(p, name, minus); lm = _loss(p)
            fd[idx] = (lp - lm) / (2 * eps)
        setattr(p, name, base)
        err = np.max(np.abs(fd - grad)) / max(1e-12, np.max(np.abs(fd)))
        assert err < 1e-6, (name, err)
    # keys of blocks nobody selected get exactly zero gradient
    assert np.count_nonzero(np.all(dk == 0, axis=-1)) > 0


def _torch_gathered(p):
    """Autograd of the gathered attention, one (t, h) at a time (fp64)."""
    q = torch.tensor(p.q, requires_grad=True)
    k = torch.tensor(p.k, requires_grad=True)
    v = torch.tensor(p.v, requires_grad=True)
    dy = torch.tensor(p.dy)
    G = p.n1 // p.n2
    loss = 0.0
    outs, lses, maxes = [], [], []
    for b in range(p.batch):
        for t in range(p.cu_q[b], p.cu_q[b + 1]):
            for h in range(p.n1):
                j = h // G
                ids = torch.tensor(p.topk[t, j], dtype=torch.long)
                rows = (p.cu_kv[b] + ids[:, None] * p.block_size +
                        torch.arange(p.block_size)[None, :]).reshape(-1)
                ks = k[:, j].index_select(0, rows)
                vs = v[:, j].index_select(0, rows)
                s = p.scale * (ks @ q[t, h])
                o = torch.softmax(s, 0) @ vs
                outs.append(o)
                maxes.append(s.max())
                lses.append(torch.logsumexp(s, 0))
                loss = loss + (o * dy[t, h]).sum()
    loss.backward()
    o = torch.stack(outs).reshape(p.t1, p.n1, p.d_v)
    mx = torch.stack(maxes).reshape(p.t1, p.n1)
    lse = torch.stack(lses).reshape(p.t1, p.n1)
    return (o.detach().numpy(), mx.detach().numpy(), lse.detach().numpy(),
            q.grad.numpy(), k.grad.numpy(), v.grad.numpy())


@pytest.mark.parametrize("duplicates", [False, True])
def test_against_torch_autograd_gathered(duplicates):
    rng = np.random.default_rng(2 + duplicates)
    p = _rand_problem(rng, n1=6, n2=2, dqk=16, dv=12, bs=4, cnt=3, lens_kv=(24, 16),
                      duplicates=duplicates, order="shuffled")
    o, m, l = oracle.forward(p)
    to, tm, tlse, tdq, tdk, tdv = _torch_gathered(p)
    np.testing.assert_allclose(o, to, rtol=0, atol=1e-12)
    np.testing.assert_allclose(m, tm, rtol=0, atol=1e-12)
    np.testing.assert_allclose(m + np.log(l), tlse, rtol=0, atol=1e-12)
    _with_forward(p)
    dq, dk, dv = oracle.backward(p)
    np.testing.assert_allclose(dq, tdq, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, tdk, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, tdv, rtol=0, atol=1e-11)


def test_dense_case_matches_dense_attention():
    """All S2/bs blocks selected (in shuffled order) == dense unmasked attention."""
    rng = np.random.default_rng(4)
    bs, lens = 8, (40, 40)
    p = _rand_problem(rng, lens_q=(9, 6), lens_kv=lens, n1=4, n2=2, dqk=16, dv=8, bs=bs,
                      cnt=lens[0] // bs, order="shuffled", scale=1 / np.sqrt(16))
    _with_forward(p)
    dq, dk, dv = oracle.backward(p)
    fo, fm, fl = oracle.forward(p)
    q = torch.tensor(p.q, requires_grad=True)
    k = torch.tensor(p.k, requires_grad=True)
    v = torch.tensor(p.v, requires_grad=True)
    G = p.n1 // p.n2
    loss = 0.0
    for b in range(p.batch):
        qs = q[p.cu_q[b]:p.cu_q[b + 1]].transpose(0, 1)                      # [n1, S1, d]
        ks = k[p.cu_kv[b]:p.cu_kv[b + 1]].transpose(0, 1).repeat_interleave(G, 0)
        vs = v[p.cu_kv[b]:p.cu_kv[b + 1]].transpose(0, 1).repeat_interleave(G, 0)
        sc = p.scale * qs @ ks.transpose(1, 2)
        o = torch.softmax(sc, -1) @ vs
        # the forward's outputs: dense attention, its row maxima and row sums
        rows = slice(p.cu_q[b], p.cu_q[b + 1])
        np.testing.assert_allclose(fo[rows], o.transpose(0, 1).detach().numpy(), rtol=0, atol=1e-12)
        mx = sc.max(-1).values
        np.testing.assert_allclose(fm[rows], mx.transpose(0, 1).detach().numpy(), rtol=0, atol=1e-12)
        sm = torch.exp(sc - mx[..., None]).sum(-1)
        np.testing.assert_allclose(fl[rows], sm.transpose(0, 1).detach().numpy(), rtol=1e-12, atol=0)
        loss = loss + (o.transpose(0, 1) * torch.tensor(p.dy[p.cu_q[b]:p.cu_q[b + 1]])).sum()
    loss.backward()
    np.testing.assert_allclose(dq, q.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, k.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, v.grad.numpy(), rtol=0, atol=1e-11)


def test_invariants_dk_sums_to_zero_dv_sums_to_dy():
    rng = np.random.default_rng(5)
    p = _with_forward(_rand_problem(rng, n1=6, n2=3, dqk=12, dv=10, lens_q=(11, 4),
                                    lens_kv=(48, 32)))
    dq, dk, dv = oracle.backward(p)
    G = p.n1 // p.n2
    for b in range(p.batch):
        ks = slice(p.cu_kv[b], p.cu_kv[b + 1])
        qs = slice(p.cu_q[b], p.cu_q[b + 1])
        for j in range(p.n2):
            # sum_j dS_j = sum_j P_j dP_j - Delta = 0 when O and the stats are exact
            np.testing.assert_allclose(dk[ks, j].sum(0), 0.0, atol=1e-12)
            # sum_j P_j = 1
            want = p.dy[qs, j * G:(j + 1) * G].sum((0, 1))
            np.testing.assert_allclose(dv[ks, j].sum(0), want, atol=1e-12)


def test_sampled_entry_points_match_full_backward():
    rng = np.random.default_rng(6)
    p = _with_forward(_rand_problem(rng))
    dq, dk, dv = oracle.backward(p)
    rows = np.array([0, 3, 17, p.t1 * p.n1 - 1])
    np.testing.assert_array_equal(oracle.dq_rows(p, rows), dq.reshape(-1, p.d_qk)[rows])
    G = p.n1 // p.n2
    for (b, j, kb) in [(0, 0, 1), (1, 1, 2), (0, 1, 3)]:
        bk, bv = oracle.dkdv_block(p, b, j, kb)
        r0 = p.cu_kv[b] + kb * p.block_size
        np.testing.assert_allclose(bk, dk[r0:r0 + p.block_size, j], rtol=0, atol=1e-14)
        np.testing.assert_allclose(bv, dv[r0:r0 + p.block_size, j], rtol=0, atol=1e-14)
    assert G == 2
    # a token range split of one block adds up to the whole block
    b, j, kb = 1, 0, 1
    mid = (p.cu_q[b] + p.cu_q[b + 1]) // 2
    k1, v1 = oracle.dkdv_block_range(p, b, j, kb, 0, mid)
    k2, v2 = oracle.dkdv_block_range(p, b, j, kb, mid, p.t1)
    wk, wv = oracle.dkdv_block(p, b, j, kb)
    np.testing.assert_allclose(k1 + k2, wk, rtol=0, atol=1e-14)
    np.testing.assert_allclose(v1 + v2, wv, rtol=0, atol=1e-14)
    # the row-subset forward equals the full forward on those rows
    o, m, l = oracle.forward(p)
    o2, m2, l2 = oracle.forward_rows(p, rows)
    np.testing.assert_array_equal(o2, o.reshape(-1, p.d_v)[rows])
    np.testing.assert_array_equal(m2, m.reshape(-1)[rows])
    np.testing.assert_array_equal(l2, l.reshape(-1)[rows])


def test_list_order_does_not_matter():
    rng = np.random.default_rng(7)
    p = _with_forward(_rand_problem(rng))
    ref = oracle.backward(p)
    perm_rng = np.random.default_rng(8)
    flat = p.topk.reshape(-1, p.block_count)
    p.topk = np.stack([perm_rng.permutation(r) for r in flat]).reshape(p.topk.shape)
    got = oracle.backward(p)
    for a, b in zip(ref, got):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_stat_lane_zero_is_read():
    rng = np.random.default_rng(9)
    p = _with_forward(_rand_problem(rng))
    ref = oracle.backward(p)
    m8 = np.repeat(p.smax, 8, axis=-1)
    l8 = np.repeat(p.ssum, 8, axis=-1)
    m8[..., 1:] = 1e30
    l8[..., 1:] = -7.0
    p.smax, p.ssum, p.stat_stride = m8, l8, 8
    got = oracle.backward(p)
    for a, b in zip(ref, got):
        np.testing.assert_array_equal(a, b)


def test_out_of_range_block_id_is_an_error():
    rng = np.random.default_rng(10)
    p = _with_forward(_rand_problem(rng))
    p.topk = p.topk.copy()
    p.topk[3, 0, 0] = 4   # batch 0 has 32 / 8 = 4 blocks: ids 0..3
    with pytest.raises(RuntimeError):
        oracle.backward(p)


@pytest.mark.parametrize("kind", ["bf16", "f16"])
def test_every_16bit_pattern_decodes_exactly(kind):
    """One key per token, each token selects its own one-row block: O = v."""
    bits = np.arange(65536, dtype=np.uint16)
    n = bits.size
    cu = np.array([0, n], np.int32)
    topk = np.arange(n, dtype=np.int32).reshape(n, 1, 1)
    one = np.zeros((n, 1, 1), np.uint16)  # q = k = +0: P = 1 for the single key
    p = oracle.Problem(cu_q=cu, cu_kv=cu, n1=1, n2=1, d_qk=1, d_v=1, block_size=1, block_count=1,
                       scale=1.0, topk=topk, q=one, k=one, v=bits.reshape(n, 1, 1), kind=kind)
    # block ids are batch local and the batch spans all n rows
    o, m, l = oracle.forward(p)
    if kind == "f16":
        want = bits.view(np.float16).astype(np.float64)
    else:
        want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = o.reshape(-1)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])
    assert np.all(m == 0.0) and np.all(l == 1.0)


def _to_bsnd(p, s1_max, s2_max, rng):
    """The same problem in the padded BSND layout; every padding row holds
    junk (random values, and block ids far out of range) that must not reach
    the result."""
    B = p.batch
    lq, lk = np.diff(p.cu_q), np.diff(p.cu_kv)

    def pad(x, lens, cu, smax, fill):
        out = fill((B * smax,) + x.shape[1:])
        for b in range(B):
            out[b * smax:b * smax + lens[b]] = x[cu[b]:cu[b + 1]]
        return out

    junk = lambda shape: rng.standard_normal(shape) * 7.0
    bad_ids = lambda shape: np.full(shape, 10 ** 6, np.int32)
    return oracle.Problem(
        cu_q=p.cu_q, cu_kv=p.cu_kv, n1=p.n1, n2=p.n2, d_qk=p.d_qk, d_v=p.d_v, block_size=p.block_size,
        block_count=p.block_count, scale=p.scale, topk=pad(p.topk, lq, p.cu_q, s1_max, bad_ids),
        q=pad(p.q, lq, p.cu_q, s1_max, junk), k=pad(p.k, lk, p.cu_kv, s2_max, junk),
        v=pad(p.v, lk, p.cu_kv, s2_max, junk), dy=pad(p.dy, lq, p.cu_q, s1_max, junk),
        o=pad(p.o, lq, p.cu_q, s1_max, junk), smax=pad(p.smax, lq, p.cu_q, s1_max, junk),
        ssum=pad(p.ssum, lq, p.cu_q, s1_max, junk), stat_stride=p.stat_stride, layout=1, s1_max=s1_max,
        s2_max=s2_max)


def test_bsnd_layout_is_the_packed_problem_with_padding_ignored():
    """BSND (every batch padded to s1_max / s2_max rows) against the same
    data packed in TND: equal forward and gradients on the valid rows, zero
    gradients on padding rows, and padding rows never read (their block ids
    are out of range and would fail the call)."""
    rng = np.random.default_rng(31)
    p = _with_forward(_rand_problem(rng, lens_q=(5, 0, 7), lens_kv=(32, 16, 24)))
    pb = _to_bsnd(p, s1_max=9, s2_max=40, rng=rng)
    o, m, l = oracle.forward(p)
    ob, mb, lb = oracle.forward(pb)
    dq, dk, dv = oracle.backward(p)
    dqb, dkb, dvb = oracle.backward(pb)
    for b in range(p.batch):
        q0, q1 = p.cu_q[b], p.cu_q[b + 1]
        k0, k1 = p.cu_kv[b], p.cu_kv[b + 1]
        r = slice(b * 9, b * 9 + q1 - q0)
        kr = slice(b * 40, b * 40 + k1 - k0)
        np.testing.assert_array_equal(ob[r], o[q0:q1])
        np.testing.assert_array_equal(mb[r], m[q0:q1])
        np.testing.assert_array_equal(lb[r], l[q0:q1])
        np.testing.assert_array_equal(dqb[r], dq[q0:q1])
        np.testing.assert_array_equal(dkb[kr], dk[k0:k1])
        np.testing.assert_array_equal(dvb[kr], dv[k0:k1])
        assert not dqb[b * 9 + q1 - q0:(b + 1) * 9].any()
        assert not dkb[b * 40 + k1 - k0:(b + 1) * 40].any() and not dvb[b * 40 + k1 - k0:(b + 1) * 40].any()
    # row-wise entry points address padded rows too
    tok_bsnd = np.array([9 * 2 + 3, 0, 4])             # batch 2 token 3, batch 0 tokens 0 and 4
    tok_tnd = np.array([p.cu_q[2] + 3, 0, 4])
    np.testing.assert_array_equal(oracle.dq_rows(pb, tok_bsnd * p.n1 + 1), oracle.dq_rows(p, tok_tnd * p.n1 + 1))
    np.testing.assert_array_equal(oracle.dkdv_block(pb, 2, 1, 2)[0], oracle.dkdv_block(p, 2, 1, 2)[0])
    with pytest.raises(RuntimeError):
        oracle.dq_rows(pb, np.array([9 * 0 + 6]) * p.n1)   # a padding row of batch 0 is not a query
