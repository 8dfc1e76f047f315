"""GPU parity: the CUDA library against the fp64 oracle, element by element.

Small cases (the tiny and varlen workloads plus ragged / edge shapes) are
compared in full, in both modes and under every schedule and switch the
library has (the three large workloads are in test_fullsize_gpu.py).
Tolerance per output tensor: relative Frobenius error <= 5e-3 and max abs
error <= 2e-2 * max|ref|.
"""
import numpy as np
import pytest
import torch

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
    return S.oracle_full_backward(w, x)


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
        # groups that do not divide a 128-row tile (126 rows used, 2 zero-filled): G = 6, and G = 3
        # (too large for gathers of four rows, so per-token boxes of 3 rows)
        "g6": base.with_(name="g6", cu_q=(0, 50, 97), cu_kv=(0, 256, 512), n1=12, n2=2, block_size=32,
                         block_count=5, seed=17),
        "g3_fp16": base.with_(name="g3_fp16", cu_q=(0, 90), cu_kv=(0, 320), n1=3, n2=1, d_qk=128, d_v=128,
                              dtype="f16", block_size=64, block_count=3, scale=128 ** -0.5, seed=18),
        # G = 8 with two KV heads
        "g8": base.with_(name="g8", cu_q=(0, 70), cu_kv=(0, 512), n1=16, n2=2, block_size=64, block_count=4,
                         seed=19),
        # 128-key blocks with 128-wide heads; 48-key blocks (N = 48 MMAs); 96-key blocks (the CUDA-core
        # kernel: no tensor-core tile for them)
        "d128_bs128": base.with_(name="d128_bs128", cu_q=(0, 33, 60), cu_kv=(0, 512, 768), n1=16, n2=2,
                                 d_qk=128, d_v=128, block_size=128, block_count=2, scale=128 ** -0.5, seed=20),
        "bs48": base.with_(name="bs48", cu_q=(0, 64), cu_kv=(0, 480), n1=16, n2=1, block_size=48, block_count=3,
                           seed=21),
        "bs96": base.with_(name="bs96", cu_q=(0, 40), cu_kv=(0, 384), n1=4, n2=1, block_size=96, block_count=2,
                           seed=22),
        # a single selected block per token; the largest group with the smallest blocks
        "cnt1": base.with_(name="cnt1", cu_q=(0, 45, 100), cu_kv=(0, 128, 320), n1=16, n2=1, block_size=64,
                           block_count=1, seed=23),
        "g32_bs16": base.with_(name="g32_bs16", cu_q=(0, 30), cu_kv=(0, 256), n1=32, n2=1, block_size=16,
                               block_count=6, seed=24),
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
    """Default mode with the work split into token windows (dK/dV as partials);
    windows belong to the in-kernel dQ reductions, forced on."""
    monkeypatch.setenv("SELATTN_WINDOW_TOKENS", str(window))
    monkeypatch.setenv("SELATTN_DQ_PASS", "0")
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
@pytest.mark.parametrize("name", ["tiny", "varlen", "ragged_fp16", "g32_bs128", "bs16_cnt127", "g6", "g3_fp16",
                                  "d128_bs128", "bs48"])
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


@pytest.mark.parametrize("name,chunk", [("varlen", 1000), ("g32_bs128", 7), ("ragged_fp16", 30)])
def test_deterministic_token_chunks(small_data, name, chunk, monkeypatch):
    """Deterministic mode run in several token chunks (dK / dV carried across
    them in fp32): parity with the oracle, and bit-identical over two runs."""
    monkeypatch.setenv("SELATTN_DS_CHUNK_TOKENS", str(chunk))
    w, x, (rdq, rdk, rdv) = small_data(name)
    desc = sab.make_desc(w.cu_q, w.cu_kv, w.n1, w.n2, w.d_qk, w.d_v, w.block_size, w.block_count, w.scale,
                         sab.SAG_FP16 if w.dtype == "f16" else sab.SAG_BF16, True)
    assert sab.plan_info(desc).token_chunks == -(-w.t1 // chunk) >= 3
    a = _run(w, x, True)
    S.assert_close(f"{name} chunks dq", S.f64(a[0]), rdq)
    S.assert_close(f"{name} chunks dk", S.f64(a[1]), rdk)
    S.assert_close(f"{name} chunks dv", S.f64(a[2]), rdv)
    b = _run(w, x, True)
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.int16), v.view(torch.int16))


@pytest.mark.parametrize("slots", ["0", "1"])
@pytest.mark.parametrize("name", ["tiny", "varlen", "ragged_fp16", "g32_bs128", "bs16_cnt127", "g6", "g8",
                                  "d128_bs128", "bs48"])
def test_deterministic_dq_sources(small_data, name, slots, monkeypatch):
    """Deterministic mode with dQ summed from per-slot fp32 partials (the
    plan's choice for small blocks and groups) or from the stored dS, each
    forced on: parity with the oracle, bit-identical over two runs."""
    monkeypatch.setenv("SELATTN_DQ_SLOTS", slots)
    w, x, (rdq, rdk, rdv) = small_data(name)
    desc = sab.make_desc(w.cu_q, w.cu_kv, w.n1, w.n2, w.d_qk, w.d_v, w.block_size, w.block_count, w.scale,
                         sab.SAG_FP16 if w.dtype == "f16" else sab.SAG_BF16, True)
    assert sab.plan_info(desc).dq_path == (2 if slots == "1" else 1)
    a = _run(w, x, True)
    S.assert_close(f"{name} slots={slots} dq", S.f64(a[0]), rdq)
    S.assert_close(f"{name} slots={slots} dk", S.f64(a[1]), rdk)
    S.assert_close(f"{name} slots={slots} dv", S.f64(a[2]), rdv)
    b = _run(w, x, True)
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.int16), v.view(torch.int16))


@pytest.mark.parametrize("name,chunk", [("varlen", 1000), ("g32_bs128", 7), ("ragged_fp16", 30)])
def test_slot_partials_in_token_chunks(small_data, name, chunk, monkeypatch):
    """The per-slot dQ partials of a token chunk indexed from the chunk's first
    token: several chunks, parity and bit-identical repeats."""
    monkeypatch.setenv("SELATTN_DQ_SLOTS", "1")
    monkeypatch.setenv("SELATTN_DS_CHUNK_TOKENS", str(chunk))
    w, x, (rdq, rdk, rdv) = small_data(name)
    desc = sab.make_desc(w.cu_q, w.cu_kv, w.n1, w.n2, w.d_qk, w.d_v, w.block_size, w.block_count, w.scale,
                         sab.SAG_FP16 if w.dtype == "f16" else sab.SAG_BF16, True)
    info = sab.plan_info(desc)
    assert info.dq_path == 2 and info.token_chunks == -(-w.t1 // chunk) >= 3
    a = _run(w, x, True)
    S.assert_close(f"{name} slot chunks dq", S.f64(a[0]), rdq)
    S.assert_close(f"{name} slot chunks dk", S.f64(a[1]), rdk)
    S.assert_close(f"{name} slot chunks dv", S.f64(a[2]), rdv)
    b = _run(w, x, True)
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.int16), v.view(torch.int16))


def test_bucket_beyond_the_shared_memory_sort():
    """Every one of 40000 query tokens selects block 0 (as NSA's always-kept
    first block would be): a bucket of 40000 entries, sorted in place through
    global memory.  Both modes against the oracle; the deterministic mode
    bit-identical over two calls."""
    w = SMALL["tiny"].with_(name="hot_block", cu_q=(0, 40000), cu_kv=(0, 512), n1=2, n2=1, d_qk=128, d_v=128,
                            block_size=16, block_count=2, scale=128 ** -0.5, seed=16)
    x = synth.make_inputs(w)
    g = torch.Generator().manual_seed(17)
    other = torch.randint(1, 32, (w.t1, 1), generator=g, dtype=torch.int32)
    x["topk"] = torch.cat([torch.zeros_like(other), other], dim=1).view(w.t1, 1, 2).contiguous()
    x = S.forward_inputs(w, x)
    rdq, rdk, rdv = _oracle_full(w, x)
    outs = {}
    for det in (False, True):
        dq, dk, dv = _run(w, x, det)
        S.assert_close(f"hot block det={det} dq", S.f64(dq), rdq)
        S.assert_close(f"hot block det={det} dk", S.f64(dk), rdk)
        S.assert_close(f"hot block det={det} dv", S.f64(dv), rdv)
        outs[det] = (dq, dk, dv)
    again = _run(w, x, True)
    for u, v in zip(outs[True], again):
        assert torch.equal(u.view(torch.int16), v.view(torch.int16))


@pytest.mark.parametrize("slots", ["0", "1"])
@pytest.mark.parametrize("name", ["varlen", "ragged_fp16", "g32_bs128", "bs16_cnt127"])
def test_default_mode_with_the_dq_pass(small_data, name, slots, monkeypatch):
    """The default mode with dQ formed by a fixed-order pass (the plan's other
    dQ paths: from the stored dS or from per-slot partials), forced on."""
    monkeypatch.setenv("SELATTN_DQ_PASS", "1")
    monkeypatch.setenv("SELATTN_DQ_SLOTS", slots)
    w, x, (rdq, rdk, rdv) = small_data(name)
    desc = sab.make_desc(w.cu_q, w.cu_kv, w.n1, w.n2, w.d_qk, w.d_v, w.block_size, w.block_count, w.scale,
                         sab.SAG_FP16 if w.dtype == "f16" else sab.SAG_BF16, False)
    assert sab.plan_info(desc).dq_path == (2 if slots == "1" else 1)
    dq, dk, dv = _run(w, x, False)
    S.assert_close(f"{name} dq pass slots={slots} dq", S.f64(dq), rdq)
    S.assert_close(f"{name} dq pass slots={slots} dk", S.f64(dk), rdk)
    S.assert_close(f"{name} dq pass slots={slots} dv", S.f64(dv), rdv)


@pytest.mark.parametrize("name", ["varlen", "bs48", "cnt1", "g32_bs16", "g32_bs128", "g6"])
def test_default_mode_with_the_reductions(small_data, name, monkeypatch):
    """The default mode with dQ reduced in the main kernel, forced; varlen,
    cnt1 and G = 32 with 16- and 128-key blocks are shapes whose plan takes
    the fixed-order pass."""
    monkeypatch.setenv("SELATTN_DQ_PASS", "0")
    w, x, (rdq, rdk, rdv) = small_data(name)
    desc = sab.make_desc(w.cu_q, w.cu_kv, w.n1, w.n2, w.d_qk, w.d_v, w.block_size, w.block_count, w.scale,
                         sab.SAG_FP16 if w.dtype == "f16" else sab.SAG_BF16, False)
    assert sab.plan_info(desc).dq_path == 0
    dq, dk, dv = _run(w, x, False)
    S.assert_close(f"{name} reductions dq", S.f64(dq), rdq)
    S.assert_close(f"{name} reductions dk", S.f64(dk), rdk)
    S.assert_close(f"{name} reductions dv", S.f64(dv), rdv)


def test_bounded_wait_runs_out_and_the_context_stays_usable(small_data):
    """A wait that nothing completes gives up after its limit, the device
    reports SAG_ERR_TIMEOUT through the workspace, and the next backward on the
    same context is still correct."""
    import time
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    t0 = time.perf_counter()
    sab.selftest_wait_timeout(ws.data_ptr(), 50_000_000, stream.cuda_stream)    # 50 ms
    assert sab.query_error(ws.data_ptr(), stream.cuda_stream) == sab.SAG_ERR_TIMEOUT
    assert time.perf_counter() - t0 >= 0.05
    w, x, (rdq, rdk, rdv) = small_data("tiny")
    dq, dk, dv = _run(w, x, False)
    S.assert_close("after timeout dq", S.f64(dq), rdq)
    S.assert_close("after timeout dk", S.f64(dk), rdk)
    S.assert_close("after timeout dv", S.f64(dv), rdv)
