"""The synthetic input recipe (CPU): index lists are distinct, sorted and in
their batch's block range; the small-group workload's skew puts exactly 3/4 of
every list on a fixed quarter of each batch's blocks; draws are reproducible
from the seed and differ between seeds."""
import torch

import synth


def _lists(w, seed=None):
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    return synth.make_topk(w, gen, "cpu")


def _check_distinct_sorted_in_range(w, topk):
    for b in range(w.batch):
        q0, q1 = w.cu_q[b], w.cu_q[b + 1]
        nblk = (w.cu_kv[b + 1] - w.cu_kv[b]) // w.block_size
        ids = topk[q0:q1].reshape(-1, w.block_count)
        if ids.numel() == 0:
            continue
        assert int(ids.min()) >= 0 and int(ids.max()) < nblk
        assert torch.all(ids[:, 1:] > ids[:, :-1])            # strictly increasing: sorted and distinct


def test_uniform_lists_are_distinct_sorted_and_batch_local():
    for w in (synth.WORKLOADS[0], synth.WORKLOADS[1], synth.WORKLOADS[2].with_(cu_q=(0, 2048), cu_kv=(0, 4096))):
        _check_distinct_sorted_in_range(w, _lists(w))


def test_skewed_lists_put_three_quarters_on_a_quarter_of_the_blocks():
    w = synth.WORKLOADS[4]
    assert w.topk == "skewed"
    # same per-batch block range and list length, fewer query tokens
    w = w.with_(cu_q=(0, 512, 1024))
    topk = _lists(w)
    _check_distinct_sorted_in_range(w, topk)
    for b in range(w.batch):
        nblk = (w.cu_kv[b + 1] - w.cu_kv[b]) // w.block_size
        ids = topk[w.cu_q[b]:w.cu_q[b + 1]].reshape(-1, w.block_count).long()
        counts = torch.bincount(ids.reshape(-1), minlength=nblk)
        hot = torch.argsort(counts, descending=True)[:nblk // 4]
        is_hot = torch.zeros(nblk, dtype=torch.bool)
        is_hot[hot] = True
        per_row_hot = is_hot[ids].sum(1)
        # every list: exactly 3/4 of its ids from the hot quarter
        assert torch.all(per_row_hot == (w.block_count * 3) // 4)
        assert float(counts[hot].sum()) / ids.numel() == 0.75


def test_draws_follow_the_seed():
    w = synth.WORKLOADS[1]
    assert torch.equal(_lists(w), _lists(w))
    assert not torch.equal(_lists(w), _lists(w, seed=w.seed + 1))
