"""GPU parity of the forward (attention_out, softmax_max, softmax_sum) against
the fp64 oracle forward, and the forward feeding the backward.

Small cases are compared in full here; the three large workloads are run at
full size in test_fullsize_gpu.py and compared on sampled query rows.  Tolerance per output tensor as for the backward:
relative Frobenius error <= 5e-3 and max abs error <= 2e-2 * max|ref|.
"""
import pytest
import torch

import sparse_attention_backward_gb300 as sab
import synth
from tests import _support as S
from tests.test_parity_gpu import SMALL

pytestmark = pytest.mark.gpu

FWD_CASES = ["tiny", "varlen", "ragged_fp16", "g32_bs128", "bs16_cnt127", "g6", "g3_fp16", "g8", "d128_bs128", "bs48"]


def _gpu_forward(w, x):
    t = {k: v.cuda() for k, v in x.items()}
    return sab.forward(t["q"], t["k"], t["v"], t["topk"], w.cu_q, w.cu_kv, w.scale, w.block_size,
                       w.block_count, check=True)


def _check_forward(o, smax, ssum, ref_o, ref_m, ref_l, shape):
    t1, n1, d_v = shape
    smax, ssum = smax.cpu(), ssum.cpu()
    # the 8 lanes of each statistic are equal
    assert torch.equal(smax, smax[..., :1].expand_as(smax))
    assert torch.equal(ssum, ssum[..., :1].expand_as(ssum))
    S.assert_close("attention_out", S.f64(o).reshape(-1, d_v), ref_o.reshape(-1, d_v))
    S.assert_close("softmax_max", smax[..., 0].double().numpy().reshape(-1), ref_m.reshape(-1))
    S.assert_close("softmax_sum", ssum[..., 0].double().numpy().reshape(-1), ref_l.reshape(-1))


@pytest.mark.parametrize("name", FWD_CASES)
def test_forward_parity_small(name):
    w = SMALL[name]
    x = synth.make_inputs(w, device="cpu")
    ref_o, ref_m, ref_l = S.oracle_full_forward(w, x)
    o, smax, ssum = _gpu_forward(w, x)
    _check_forward(o, smax, ssum, ref_o, ref_m, ref_l, (w.t1, w.n1, w.d_v))


def test_forward_rejects_unsupported_value_dim():
    w = SMALL["dv192"]
    x = synth.make_inputs(w, device="cpu")
    with pytest.raises(sab.SagError) as e:
        _gpu_forward(w, x)
    assert e.value.status == sab.SAG_ERR_UNSUPPORTED


def test_forward_then_backward():
    """The GPU forward's outputs as the backward's inputs: the GPU backward
    matches the oracle backward given the same (GPU-produced) O and stats."""
    w = SMALL["varlen"]
    x = synth.make_inputs(w, device="cpu")
    o, smax, ssum = _gpu_forward(w, x)
    x = dict(x, o=o.cpu(), softmax_max=smax.cpu(), softmax_sum=ssum.cpu())
    t = {k: v.cuda() for k, v in x.items()}
    dq, dk, dv = sab.backward(t["q"], t["k"], t["v"], t["o"], t["dy"], t["softmax_max"], t["softmax_sum"],
                              t["topk"], w.cu_q, w.cu_kv, w.scale, w.block_size, w.block_count, check=True)
    ref = S.oracle_full_backward(w, x)
    for nm, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        S.assert_close(nm, S.f64(got), r)


def test_forward_reports_out_of_range_ids():
    w = SMALL["tiny"]
    x = synth.make_inputs(w, device="cpu")
    x["topk"] = x["topk"].clone()
    x["topk"][5, 0, 1] = 10 ** 6
    with pytest.raises(sab.SagError) as e:
        _gpu_forward(w, x)
    assert e.value.status == sab.SAG_ERR_INDEX


@pytest.mark.parametrize("window", [37, 300])
@pytest.mark.parametrize("name", ["varlen", "ragged_fp16", "g32_bs128"])
def test_forward_token_windows_parity(name, window, monkeypatch):
    """Token windows (the default on problems whose O accumulator is far
    beyond L2) forced small on small problems."""
    monkeypatch.setenv("SELATTN_FWD_WINDOW_TOKENS", str(window))
    w = SMALL[name]
    x = synth.make_inputs(w, device="cpu")
    ref_o, ref_m, ref_l = S.oracle_full_forward(w, x)
    o, smax, ssum = _gpu_forward(w, x)
    _check_forward(o, smax, ssum, ref_o, ref_m, ref_l, (w.t1, w.n1, w.d_v))
