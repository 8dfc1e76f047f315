"""Pins of the lightning-indexer oracle (CPU only), none reusing its code:

* central finite differences of L = sum(dy * scores(q, k, w)), the loss
  whose gradient the backward is (scores = the index scores of the selected
  positions, sum over heads of w * relu(q . k));
* torch fp64 autograd of an independent formulation of those scores, with a
  position selected twice (the ScatterAdd counts it twice) and empty slots;
* the identities that come from relu being positively homogeneous:
  <q[t,h], dQ[t,h]> = w[t,h] * dW[t,h] per row, and
  sum over key rows of <k, dK> = sum of w * dW;
* row entry points against the full backward; BSND against the packed
  problem with junk in the padding rows; an id out of range is an error.
"""
import numpy as np
import pytest
import torch

import oracle.indexer as li


def _problem(rng, lens_q=(5, 4), lens_kv=(20, 12), n1=4, n2=2, d=6, topk=5, dup=False, empty=False):
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_kv = np.concatenate([[0], np.cumsum(lens_kv)]).astype(np.int32)
    t1, t2 = int(cu_q[-1]), int(cu_kv[-1])
    idx = np.zeros((t1, n2, topk), np.int32)
    for b in range(len(lens_q)):
        for t in range(cu_q[b], cu_q[b + 1]):
            for j in range(n2):
                ids = rng.choice(lens_kv[b], topk, replace=False)
                if dup:
                    ids[1] = ids[0]
                if empty:
                    ids[-1] = -1
                idx[t, j] = ids
    return li.Problem(cu_q=cu_q, cu_kv=cu_kv, n1=n1, n2=n2, d=d, topk=topk, idx=idx,
                      q=rng.standard_normal((t1, n1, d)), k=rng.standard_normal((t2, n2, d)),
                      w=rng.standard_normal((t1, n1)), dy=rng.standard_normal((t1, n2, topk)))


def _torch_scores(p, q, k, w):
    G = p.n1 // p.n2
    out = torch.zeros((p.t1, p.n2, p.topk), dtype=torch.float64)
    for b in range(p.batch):
        for t in range(p.cu_q[b], p.cu_q[b + 1]):
            for j in range(p.n2):
                ids = torch.as_tensor(p.idx[t, j].astype(np.int64))
                keep = ids != -1
                kk = k[p.cu_kv[b] + ids[keep], j]                 # [m, d]
                qq = q[t, j * G:(j + 1) * G]                       # [G, d]
                s = torch.relu(qq @ kk.T)                          # [G, m]
                row = torch.zeros(p.topk, dtype=torch.float64)
                row[keep] = (w[t, j * G:(j + 1) * G, None] * s).sum(0)
                out[t, j] = row
    return out


def test_finite_differences():
    rng = np.random.default_rng(1)
    p = _problem(rng)
    dq, dk, dw = li.backward(p)
    eps = 1e-6

    def loss():
        return float(np.sum(li.scores(p) * p.dy))

    for name, arr, grad in (("q", p.q, dq), ("k", p.k, dk), ("w", p.w, dw)):
        flat = arr.reshape(-1)
        for i in rng.choice(flat.size, 12, replace=False):
            old = flat[i]
            flat[i] = old + eps
            lp = loss()
            flat[i] = old - eps
            lm = loss()
            flat[i] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad.reshape(-1)[i]) <= 1e-6 * max(1.0, abs(fd)), (name, i, fd, grad.reshape(-1)[i])


@pytest.mark.parametrize("dup,empty", [(False, False), (True, True)])
def test_torch_autograd(dup, empty):
    rng = np.random.default_rng(2)
    p = _problem(rng, dup=dup, empty=empty)
    q = torch.tensor(p.q, requires_grad=True)
    k = torch.tensor(p.k, requires_grad=True)
    w = torch.tensor(p.w, requires_grad=True)
    (torch.tensor(p.dy) * _torch_scores(p, q, k, w)).sum().backward()
    dq, dk, dw = li.backward(p)
    np.testing.assert_allclose(dq, q.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dk, k.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dw, w.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(li.scores(p), _torch_scores(p, q, k, w).detach().numpy(), rtol=1e-12, atol=1e-12)


def test_relu_homogeneity_identities():
    rng = np.random.default_rng(3)
    p = _problem(rng, lens_q=(9, 7), lens_kv=(40, 24), n1=8, n2=2, d=16, topk=6)
    dq, dk, dw = li.backward(p)
    lhs = np.einsum("thd,thd->th", p.q, dq)
    np.testing.assert_allclose(lhs, p.w * dw, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(np.einsum("sjd,sjd->", p.k, dk), np.sum(p.w * dw), rtol=1e-10)


def test_row_entry_points_match_the_full_backward():
    rng = np.random.default_rng(4)
    p = _problem(rng, dup=True, empty=True)
    dq, dk, dw = li.backward(p)
    toks = np.array([0, 3, 7, 8])
    rq, rw = li.q_rows(p, toks)
    np.testing.assert_array_equal(rq, dq[toks])
    np.testing.assert_array_equal(rw, dw[toks])
    rows, heads = np.array([0, 5, 19, 20, 31]), np.array([0, 1, 1, 0, 1])
    np.testing.assert_array_equal(li.k_rows(p, rows, heads), dk[rows, heads])


def test_token_ranges_sum_to_the_full_backward():
    rng = np.random.default_rng(6)
    p = _problem(rng, dup=True, empty=True)
    full = li.backward(p)
    parts = [li.backward_range(p, a, b) for a, b in ((0, 3), (3, 7), (7, p.t1))]
    for i in range(3):
        np.testing.assert_allclose(sum(x[i] for x in parts), full[i], rtol=1e-13, atol=1e-13)


def test_bsnd_is_the_packed_problem_and_bad_ids_fail():
    rng = np.random.default_rng(5)
    p = _problem(rng, lens_q=(5, 0, 4), lens_kv=(20, 8, 12))
    s1, s2 = 7, 24

    def pad(x, cu, smax, fill):
        out = np.full((p.batch * smax,) + x.shape[1:], fill, dtype=x.dtype)
        for b in range(p.batch):
            out[b * smax:b * smax + cu[b + 1] - cu[b]] = x[cu[b]:cu[b + 1]]
        return out
    pb = li.Problem(cu_q=p.cu_q, cu_kv=p.cu_kv, n1=p.n1, n2=p.n2, d=p.d, topk=p.topk,
                    idx=pad(p.idx, p.cu_q, s1, 10 ** 6), q=pad(p.q, p.cu_q, s1, 3.5), k=pad(p.k, p.cu_kv, s2, -2.5),
                    w=pad(p.w, p.cu_q, s1, 7.0), dy=pad(p.dy, p.cu_q, s1, 9.0), layout=1, s1_max=s1, s2_max=s2)
    dq, dk, dw = li.backward(p)
    dqb, dkb, dwb = li.backward(pb)
    for b in range(p.batch):
        nq, nk = p.cu_q[b + 1] - p.cu_q[b], p.cu_kv[b + 1] - p.cu_kv[b]
        np.testing.assert_array_equal(dqb[b * s1:b * s1 + nq], dq[p.cu_q[b]:p.cu_q[b + 1]])
        np.testing.assert_array_equal(dwb[b * s1:b * s1 + nq], dw[p.cu_q[b]:p.cu_q[b + 1]])
        np.testing.assert_array_equal(dkb[b * s2:b * s2 + nk], dk[p.cu_kv[b]:p.cu_kv[b + 1]])
        assert not dqb[b * s1 + nq:(b + 1) * s1].any() and not dkb[b * s2 + nk:(b + 1) * s2].any()
    p.idx[2, 1, 0] = p.cu_kv[1] - p.cu_kv[0]          # one past batch 0's keys
    with pytest.raises(RuntimeError):
        li.backward(p)
