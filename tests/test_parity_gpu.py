"""GPU parity: the CUDA library against the fp64 oracle, element by element.

Small cases (the tiny and varlen workloads plus ragged / edge shapes) are
compared in full; the three large workloads are run at full size in the
launch configuration the benchmark times and compared on sampled dQ rows and
sampled key blocks (dK, dV) that the oracle computes one by one.  Tolerance
per output tensor: relative Frobenius error <= 5e-3 and max abs error
<= 2e-2 * max|ref|.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_backward_gb300 as sab
import synth
from tests import _support as S

pytestmark = pytest.mark.gpu


def _run(w, x, deterministic):
    t = {k: v.cuda() for k, v in x.items()}
    return sab.backward(t["q"], t["k"], t["v"], t["o"], t["dy"], t["softmax_max"], t["softmax_sum"],
                        t["topk"], w.cu_q, w.cu_kv, w.scale, w.block_size, w.block_count,
                        deterministic=deterministic, check=True)


def _oracle_full(w, x):
    p = S.problem(w, x)
    rows = np.arange(w.t1 * w.n1)
    big = w.t1 * w.n1 * w.selected_keys > 2_000_000
    dq = (S.par_dq_rows(p, rows) if big else oracle.dq_rows(p, rows)).reshape(w.t1, w.n1, w.d_qk)
    blocks = [(b, j, kb) for b in range(w.batch) for j in range(w.n2)
              for kb in range((w.cu_kv[b + 1] - w.cu_kv[b]) // w.block_size)]
    res = S.par_dkdv_blocks(p, blocks) if big else [oracle.dkdv_block(p, *a) for a in blocks]
    dk = np.zeros((w.t2, w.n2, w.d_qk))
    dv = np.zeros((w.t2, w.n2, w.d_v))
    for (b, j, kb), (bk, bv) in zip(blocks, res):
        r0 = w.cu_kv[b] + kb * w.block_size
        dk[r0:r0 + w.block_size, j] = bk
        dv[r0:r0 + w.block_size, j] = bv
    return dq, dk, dv


def _small_cases():
    base = synth.WORKLOADS[0]
    return {
        "tiny": base,
        "varlen": synth.WORKLOADS[1],
        # empty first batch, ragged query lengths, fp16, G = 2, Dqk = Dv = 128
        "ragged_fp16": base.with_(name="ragged_fp16", cu_q=(0, 0, 37, 100), cu_kv=(0, 128, 320, 448),
                                  n1=6, n2=3, d_qk=128, d_v=128, dtype="f16", block_size=32,
                                  block_count=3, scale=128 ** -0.5, seed=11),
        # largest group (G = 32), largest block (128), two KV heads
        "g32_bs128": base.with_(name="g32_bs128", cu_q=(0, 9, 21), cu_kv=(0, 512, 768), n1=64, n2=2,
                                block_size=128, block_count=2, seed=12),
        # many small blocks: block_count = 127
        "bs16_cnt127": base.with_(name="bs16_cnt127", cu_q=(0, 13), cu_kv=(0, 2048), n1=2, n2=1,
                                  block_size=16, block_count=127, seed=13),
        # value head dim 192 (K and V head dims may differ)
        "dv192": base.with_(name="dv192", cu_q=(0, 40), cu_kv=(0, 384), n1=8, n2=2, d_qk=128, d_v=192,
                            block_size=64, block_count=3, scale=128 ** -0.5, seed=14),
    }


SMALL = _small_cases()


@pytest.fixture(scope="module")
def small_data():
    cache = {}

    def get(name):
        if name not in cache:
            w = SMALL[name]
            x = S.workload_inputs(w, "cpu")
            cache[name] = (w, x, _oracle_full(w, x))
        return cache[name]
    return get


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("name", list(SMALL))
def test_full_parity_small(small_data, name, deterministic):
    w, x, (rdq, rdk, rdv) = small_data(name)
    dq, dk, dv = _run(w, x, deterministic)
    S.assert_close(f"{name} dq", S.f64(dq), rdq)
    S.assert_close(f"{name} dk", S.f64(dk), rdk)
    S.assert_close(f"{name} dv", S.f64(dv), rdv)
    # rows of blocks nobody selected are exactly zero
    unsel = np.all(rdk == 0, axis=-1)
    assert np.all(S.f64(dk)[unsel] == 0) and np.all(S.f64(dv)[unsel] == 0)


@pytest.mark.parametrize("window", [37, 300])
@pytest.mark.parametrize("name", ["varlen", "ragged_fp16", "g32_bs128", "bs16_cnt127"])
def test_token_windows_parity(small_data, name, window, monkeypatch):
    """Default mode with the work split into token windows (dK/dV as partials)."""
    monkeypatch.setenv("SELATTN_WINDOW_TOKENS", str(window))
    w, x, (rdq, rdk, rdv) = small_data(name)
    desc = sab.make_desc(w.cu_q, w.cu_kv, w.n1, w.n2, w.d_qk, w.d_v, w.block_size, w.block_count, w.scale,
                         sab.SAG_FP16 if w.dtype == "f16" else sab.SAG_BF16, False)
    assert sab.plan_info(desc).launches == 10   # windowed: the dK/dV cast runs too
    dq, dk, dv = _run(w, x, False)
    S.assert_close(f"{name} w{window} dq", S.f64(dq), rdq)
    S.assert_close(f"{name} w{window} dk", S.f64(dk), rdk)
    S.assert_close(f"{name} w{window} dv", S.f64(dv), rdv)


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("split", ["0", "1"])
@pytest.mark.parametrize("name", ["tiny", "varlen", "ragged_fp16", "g32_bs128", "bs16_cnt127"])
def test_both_tensor_core_schedules(small_data, name, split, deterministic, monkeypatch):
    """Both tensor-core schedules (softmax between the MMA groups, or split in
    two phases beside them) forced on shapes either can take, both modes."""
    monkeypatch.setenv("SELATTN_SPLIT_SOFTMAX", split)
    w, x, (rdq, rdk, rdv) = small_data(name)
    dq, dk, dv = _run(w, x, deterministic)
    S.assert_close(f"{name} split={split} dq", S.f64(dq), rdq)
    S.assert_close(f"{name} split={split} dk", S.f64(dk), rdk)
    S.assert_close(f"{name} split={split} dv", S.f64(dv), rdv)


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("name", ["tiny", "varlen", "g32_bs128"])
def test_cuda_core_kernel_parity(small_data, name, deterministic, monkeypatch):
    """The CUDA-core kernel on shapes the tensor-core kernel also takes."""
    monkeypatch.setenv("SELATTN_FORCE_CUDA_CORE", "1")
    w, x, (rdq, rdk, rdv) = small_data(name)
    desc = sab.make_desc(w.cu_q, w.cu_kv, w.n1, w.n2, w.d_qk, w.d_v, w.block_size, w.block_count, w.scale,
                         sab.SAG_FP16 if w.dtype == "f16" else sab.SAG_BF16, deterministic)
    assert sab.plan_info(desc).main_kernel == 0
    dq, dk, dv = _run(w, x, deterministic)
    S.assert_close(f"{name} cuda-core dq", S.f64(dq), rdq)
    S.assert_close(f"{name} cuda-core dk", S.f64(dk), rdk)
    S.assert_close(f"{name} cuda-core dv", S.f64(dv), rdv)


def test_tensor_core_kernel_is_selected():
    for w in synth.WORKLOADS:
        desc = sab.make_desc(w.cu_q, w.cu_kv, w.n1, w.n2, w.d_qk, w.d_v, w.block_size, w.block_count,
                             w.scale, sab.SAG_FP16 if w.dtype == "f16" else sab.SAG_BF16, False)
        assert sab.plan_info(desc).main_kernel == 1, w.name


def test_duplicate_ids_count_twice():
    w = SMALL["tiny"].with_(name="dups", cu_q=(0, 20), cu_kv=(0, 128), n1=4, n2=2, block_size=16,
                           block_count=4, seed=15)
    x = synth.make_inputs(w)
    topk = x["topk"].clone()
    topk[:, :, 1] = topk[:, :, 0]          # every list repeats its first id
    topk[5, 1, :] = 3                      # one list names the same block four times
    x["topk"] = topk
    x = S.forward_inputs(w, x)
    rdq, rdk, rdv = _oracle_full(w, x)
    for det in (False, True):
        dq, dk, dv = _run(w, x, det)
        S.assert_close("dups dq", S.f64(dq), rdq)
        S.assert_close("dups dk", S.f64(dk), rdk)
        S.assert_close("dups dv", S.f64(dv), rdv)


def test_out_of_range_id_is_reported_not_read():
    w = SMALL["tiny"]
    x = synth.make_inputs(w)
    x = S.forward_inputs(w, x)
    x["topk"] = x["topk"].clone()
    x["topk"][7, 0, 2] = 16                # 256 / 16 = 16 blocks: ids 0..15
    x["topk"][9, 0, 0] = -1
    for det in (False, True):
        with pytest.raises(sab.SagError) as e:
            _run(w, x, det)
        assert e.value.status == sab.SAG_ERR_INDEX


@pytest.mark.parametrize("name", list(SMALL))
def test_deterministic_mode_is_bitwise_reproducible(small_data, name):
    w, x, _ = small_data(name)
    a = _run(w, x, True)
    b = _run(w, x, True)
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.int16), v.view(torch.int16))


# ---------------------------------------------------------------- full size
def _sampled_parity(w, x, outs, n_rows=512, n_blocks=4, seed=0):
    dq, dk, dv = outs
    rng = np.random.default_rng(seed)
    # dQ rows: grouped by (batch, KV head) into sub-problems the oracle can run
    rows = rng.choice(w.t1 * w.n1, n_rows, replace=False)
    ref, got = [], []
    tb = np.searchsorted(np.asarray(w.cu_q), rows // w.n1, side="right") - 1
    for b in np.unique(tb):
        for j in range(w.n2):
            sel = rows[(tb == b) & ((rows % w.n1) // w.group == j)]
            if sel.size == 0:
                continue
            toks = np.unique(sel // w.n1)
            sub = S.sub_problem(w, x, int(b), j, toks)
            pos = np.searchsorted(toks, sel // w.n1)
            sub_rows = pos * w.group + (sel % w.n1) % w.group
            ref.append(S.par_dq_rows(sub, sub_rows))
            got.append(S.f64(dq.view(-1, w.d_qk)[torch.as_tensor(sel, device=dq.device)]))
    S.assert_close(f"{w.name} dq (sampled rows)", np.concatenate(got), np.concatenate(ref))
    # key blocks: random ones plus the most selected one
    blocks = []
    for i in range(n_blocks):
        b = int(rng.integers(w.batch))
        j = int(rng.integers(w.n2))
        nblk = (w.cu_kv[b + 1] - w.cu_kv[b]) // w.block_size
        kb = int(rng.integers(nblk))
        if i == n_blocks - 1:
            q0, q1 = w.cu_q[b], w.cu_q[b + 1]
            cnt = torch.bincount(x["topk"][q0:q1, j].reshape(-1).long(), minlength=nblk)
            kb = int(torch.argmax(cnt))
        blocks.append((b, j, kb))
    rk, rv, gk, gv = [], [], [], []
    for (b, j, kb) in blocks:
        toks = S.selecting_tokens(w, x, b, j, kb)
        sub = S.sub_problem(w, x, b, j, toks)
        bk, bv = S.par_dkdv_block(sub, 0, 0, kb)
        r0 = w.cu_kv[b] + kb * w.block_size
        rk.append(bk)
        rv.append(bv)
        gk.append(S.f64(dk[r0:r0 + w.block_size, j]))
        gv.append(S.f64(dv[r0:r0 + w.block_size, j]))
    S.assert_close(f"{w.name} dk (sampled blocks)", np.concatenate(gk), np.concatenate(rk))
    S.assert_close(f"{w.name} dv (sampled blocks)", np.concatenate(gv), np.concatenate(rv))


def _full_size(idx, deterministic):
    w = synth.WORKLOADS[idx]
    x = synth.make_inputs(w, device="cuda")
    outs = sab.backward(x["q"], x["k"], x["v"], x["o"], x["dy"], x["softmax_max"], x["softmax_sum"],
                        x["topk"], w.cu_q, w.cu_kv, w.scale, w.block_size, w.block_count,
                        deterministic=deterministic, check=True)
    torch.cuda.synchronize()
    _sampled_parity(w, x, outs)
    return w, x, outs


@pytest.mark.parametrize("deterministic", [False, True])
def test_long_context_sampled(deterministic):
    _full_size(2, deterministic)


@pytest.mark.parametrize("deterministic", [False, True])
def test_max_selection_sampled(deterministic):
    _full_size(3, deterministic)


def test_small_group_stress_sampled():
    _full_size(4, False)
