"""The allocation-free entry point against the workspace entry point.

sel_attn_grad_noalloc serves callers that cannot allocate device memory when
they call the backward (a framework memory pool that forbids raw cudaMalloc,
a plug-in handed only tensors): its scratch is a fixed array inside the
library.  Here it is called through the C ABI twice in a row (the second call
finds the first call's leftovers in the shared array) and must agree with
sel_attn_grad on a caller-owned workspace within the parity tolerance.  The
file is collected last so that a stop-at-first-failure run has already run
every other test.
"""
import ctypes
import os
import re

import pytest
import torch

import sparse_attention_backward_gb300 as sab
import synth
from tests import _support as S

pytestmark = pytest.mark.gpu


def _entry(lib):
    f = lib.sel_attn_grad_noalloc
    f.argtypes = [ctypes.POINTER(sab.SagDesc)] + [ctypes.c_void_p] * 12
    f.restype = ctypes.c_int
    return f


def _inputs(w, dev, seed):
    x = S.gpu_forward_inputs(w, synth.make_inputs(w, device=dev, seed=seed))
    return [x[k] for k in ("q", "k", "v", "o", "dy", "softmax_max", "softmax_sum", "topk")]


def _scratch_limit() -> int:
    """SEL_ATTN_GRAD_NOALLOC_MAX_SCRATCH as the library's header defines it."""
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "selattn.h")
    with open(hdr) as f:
        m = re.search(r"#define SEL_ATTN_GRAD_NOALLOC_MAX_SCRATCH \(\(size_t\)(\d+) << (\d+)\)", f.read())
    assert m, "limit not found in include/selattn.h"
    return int(m.group(1)) << int(m.group(2))


def _desc(w, det):
    return sab.make_desc(w.cu_q, w.cu_kv, w.n1, w.n2, w.d_qk, w.d_v, w.block_size, w.block_count, w.scale,
                         sab.SAG_FP16 if w.dtype == "f16" else sab.SAG_BF16, det)


@pytest.mark.parametrize("deterministic", [False, True])
def test_noalloc_matches_workspace_entry_point(deterministic):
    lib = sab.load()
    f = _entry(lib)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    w = synth.WORKLOADS[0]
    # two calls in a row on different inputs: the second must not see the first
    for call, seed in enumerate((101, 202)):
        ins = _inputs(w, dev, seed)
        want = sab.backward(*ins, w.cu_q, w.cu_kv, w.scale, w.block_size, w.block_count,
                            deterministic=deterministic, check=True)
        got = [torch.full_like(t, float("nan")) for t in (ins[0], ins[1], ins[2])]
        desc = _desc(w, deterministic)
        st = f(ctypes.byref(desc), *[t.data_ptr() for t in ins], *[t.data_ptr() for t in got],
               stream.cuda_stream)
        assert st == sab.SAG_OK, sab.status_string(st)
        torch.cuda.synchronize()
        for name, g, r in zip(("dq", "dk", "dv"), got, want):
            S.assert_close(f"call {call} {name}", S.f64(g), S.f64(r))


def test_noalloc_reports_out_of_range_ids():
    """An id past the batch's blocks is skipped and reported; the status is
    read back from the fixed scratch, and a clean call clears it."""
    lib = sab.load()
    f = _entry(lib)
    q_err = lib.sel_attn_grad_noalloc_query_error
    q_err.argtypes = [ctypes.c_void_p]
    q_err.restype = ctypes.c_int
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    w = synth.WORKLOADS[0]
    ins = _inputs(w, dev, 303)
    bad = ins[7].clone()
    bad[3, 0, 1] = 10 ** 6
    outs = [torch.empty_like(t) for t in (ins[0], ins[1], ins[2])]
    desc = _desc(w, False)
    for topk, want in ((bad, sab.SAG_ERR_INDEX), (ins[7], sab.SAG_OK)):
        st = f(ctypes.byref(desc), *[t.data_ptr() for t in ins[:7]], topk.data_ptr(),
               *[t.data_ptr() for t in outs], stream.cuda_stream)
        assert st == sab.SAG_OK, sab.status_string(st)
        assert q_err(stream.cuda_stream) == want


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = sab.load()
    f = _entry(lib)
    w = synth.WORKLOADS[2]   # long context: its workspace is far above the fixed scratch
    need = sab.workspace_size(_desc(w, False))
    assert need > _scratch_limit()
    dev = torch.device("cuda", 0)
    dummy = torch.empty(16, dtype=torch.uint8, device=dev)
    st = f(ctypes.byref(_desc(w, False)), *([dummy.data_ptr()] * 11),
           torch.cuda.current_stream(dev).cuda_stream)
    assert st == sab.SAG_ERR_WORKSPACE
