"""GB300 (sm_103a) selected-attention backward: thin Python binding.

Every step of the backward runs in the CUDA kernels of ``libselattn.so``; this
module only marshals arguments into its C ABI (``include/selattn.h``) with
ctypes.  PyTorch is used for device memory and streams.  There is no CPU path:
if the library is missing, importing the binding's entry points raises.

    import sparse_attention_backward_gb300 as sab
    dq, dk, dv = sab.backward(q, k, v, o, dy, softmax_max, softmax_sum, topk,
                              cu_seqlens_q, cu_seqlens_kv, scale,
                              block_size, block_count, deterministic=False)

Tensors are TND ([T, N, D]) or, given as 4-D tensors, BSND ([B, S, N, D] with
every batch padded to S rows; cu_seqlens then give the valid lengths).  With
``q_rope`` / ``k_rope`` the head dim is split (Q = [q, q_rope] along D) and
the gradients come back as (dq, dk, dv, dq_rope, dk_rope).
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libselattn.so")

SAG_OK, SAG_ERR_NULL, SAG_ERR_SHAPE, SAG_ERR_DTYPE, SAG_ERR_UNSUPPORTED = 0, 1, 2, 3, 4
SAG_ERR_WORKSPACE, SAG_ERR_ALIGN, SAG_ERR_CUDA, SAG_ERR_INDEX, SAG_ERR_TIMEOUT = 5, 6, 7, 8, 9
SAG_BF16, SAG_FP16 = 0, 1
SAG_LAYOUT_TND, SAG_LAYOUT_BSND = 0, 1

EXPORTED = ("sel_attn_grad_workspace_size", "sel_attn_grad", "sel_attn_grad_timed", "sel_attn_grad_ex",
            "sel_attn_grad_plan_info", "sel_attn_grad_query_error", "sel_attn_grad_status_string",
            "sel_attn_fwd_workspace_size", "sel_attn_fwd", "sel_attn_fwd_timed", "sel_attn_fwd_ex",
            "lightning_indexer_grad_workspace_size", "lightning_indexer_grad", "sel_attn_selftest_wait_timeout")


class SagDesc(ctypes.Structure):
    """Mirror of ``sag_desc`` in include/selattn.h."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("n1", ctypes.c_int32), ("n2", ctypes.c_int32),
        ("d_qk", ctypes.c_int32), ("d_v", ctypes.c_int32),
        ("block_size", ctypes.c_int32), ("block_count", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("deterministic", ctypes.c_int32), ("layout", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("cu_seqlens_q", ctypes.POINTER(ctypes.c_int32)),
        ("cu_seqlens_kv", ctypes.POINTER(ctypes.c_int32)),
        ("s1_max", ctypes.c_int32), ("s2_max", ctypes.c_int32), ("d_rope", ctypes.c_int32),
        ("reserved_", ctypes.c_int32),
    ]


class SagIo(ctypes.Structure):
    """Mirror of ``sag_io`` in include/selattn.h (device pointers as ints)."""
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "query", "key", "value", "attention_out", "attention_out_grad", "softmax_max", "softmax_sum",
        "topk_indices", "query_rope", "key_rope", "dq", "dk", "dv", "dq_rope", "dk_rope")]


class SagPlanInfo(ctypes.Structure):
    """Mirror of ``sag_plan_info`` in include/selattn.h."""
    _fields_ = [("workspace_bytes", ctypes.c_uint64), ("launches", ctypes.c_int32),
                ("token_chunks", ctypes.c_int32), ("items", ctypes.c_int64),
                ("main_kernel", ctypes.c_int32), ("dq_path", ctypes.c_int32)]


class SagError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({status_string(status)})")
        self.status = status


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libselattn.so (built by ``build.py``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} not found: build it with "
                           "`python -m sparse_attention_backward_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    D = ctypes.POINTER(SagDesc)
    lib.sel_attn_grad_workspace_size.argtypes = [D, ctypes.POINTER(sz)]
    lib.sel_attn_grad_workspace_size.restype = ctypes.c_int
    lib.sel_attn_grad.argtypes = [D] + [vp] * 11 + [vp, sz, vp]
    lib.sel_attn_grad.restype = ctypes.c_int
    lib.sel_attn_grad_timed.argtypes = [D] + [vp] * 11 + [vp, sz, vp, vp, vp]
    lib.sel_attn_grad_timed.restype = ctypes.c_int
    IO = ctypes.POINTER(SagIo)
    lib.sel_attn_grad_ex.argtypes = [D, IO, vp, sz, vp, vp, vp]
    lib.sel_attn_grad_ex.restype = ctypes.c_int
    lib.sel_attn_fwd_ex.argtypes = [D, IO, vp, sz, vp, vp, vp]
    lib.sel_attn_fwd_ex.restype = ctypes.c_int
    lib.sel_attn_grad_plan_info.argtypes = [D, ctypes.POINTER(SagPlanInfo)]
    lib.sel_attn_grad_plan_info.restype = ctypes.c_int
    lib.sel_attn_grad_query_error.argtypes = [vp, vp]
    lib.sel_attn_grad_query_error.restype = ctypes.c_int
    lib.sel_attn_fwd_workspace_size.argtypes = [D, ctypes.POINTER(sz)]
    lib.sel_attn_fwd_workspace_size.restype = ctypes.c_int
    lib.sel_attn_fwd.argtypes = [D] + [vp] * 7 + [vp, sz, vp]
    lib.sel_attn_fwd.restype = ctypes.c_int
    lib.sel_attn_fwd_timed.argtypes = [D] + [vp] * 7 + [vp, sz, vp, vp, vp]
    lib.sel_attn_fwd_timed.restype = ctypes.c_int
    lib.sel_attn_grad_status_string.argtypes = [ctypes.c_int]
    lib.sel_attn_grad_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().sel_attn_grad_status_string(int(status)).decode()


def make_desc(cu_seqlens_q, cu_seqlens_kv, n1, n2, d_qk, d_v, block_size, block_count, scale,
              dtype=SAG_BF16, deterministic=False, layout=SAG_LAYOUT_TND, s1_max=0, s2_max=0, d_rope=0):
    """Build a descriptor; keeps the host cu_seqlens arrays alive on the object.

    ``d_qk`` is the head dim of the query / key tensors (without the rope
    part when ``d_rope`` is set); BSND takes the padded lengths s1_max, s2_max.
    """
    cq = (ctypes.c_int32 * len(cu_seqlens_q))(*[int(x) for x in cu_seqlens_q])
    ck = (ctypes.c_int32 * len(cu_seqlens_kv))(*[int(x) for x in cu_seqlens_kv])
    d = SagDesc(batch=len(cu_seqlens_q) - 1, n1=n1, n2=n2, d_qk=d_qk, d_v=d_v,
                block_size=block_size, block_count=block_count, dtype=dtype,
                deterministic=1 if deterministic else 0, layout=int(layout), scale=float(scale),
                cu_seqlens_q=ctypes.cast(cq, ctypes.POINTER(ctypes.c_int32)),
                cu_seqlens_kv=ctypes.cast(ck, ctypes.POINTER(ctypes.c_int32)),
                s1_max=int(s1_max), s2_max=int(s2_max), d_rope=int(d_rope), reserved_=0)
    d._keep = (cq, ck)
    return d


def make_io(**ptrs) -> SagIo:
    """sag_io from device pointers (ints); names as in the C struct, others NULL."""
    io = SagIo()
    for k, v in ptrs.items():
        setattr(io, k, v)
    return io


def sel_attn_grad_ex(desc: SagDesc, io: SagIo, workspace, workspace_bytes: int, stream, main_start=None,
                     main_stop=None) -> None:
    """Phase 2 with every tensor in one sag_io; raises on a non-OK status."""
    st = load().sel_attn_grad_ex(ctypes.byref(desc), ctypes.byref(io), workspace, workspace_bytes, stream,
                                 main_start, main_stop)
    if st != SAG_OK:
        raise SagError(st, "sel_attn_grad_ex")


def sel_attn_fwd_ex(desc: SagDesc, io: SagIo, workspace, workspace_bytes: int, stream, passes_start=None,
                    passes_stop=None) -> None:
    """Forward phase 2 with every tensor in one sag_io; raises on a non-OK status."""
    st = load().sel_attn_fwd_ex(ctypes.byref(desc), ctypes.byref(io), workspace, workspace_bytes, stream,
                                passes_start, passes_stop)
    if st != SAG_OK:
        raise SagError(st, "sel_attn_fwd_ex")


def _layout_of(q, k, q_rope):
    """(layout, s1_max, s2_max, n1, d_qk, n2, d_rope) from the tensors' shapes."""
    if q.dim() == 4:
        if k.dim() != 4:
            raise ValueError("BSND needs 4-D query and key tensors")
        layout, s1_max, s2_max = SAG_LAYOUT_BSND, q.shape[1], k.shape[1]
    else:
        layout, s1_max, s2_max = SAG_LAYOUT_TND, 0, 0
    return layout, s1_max, s2_max, q.shape[-2], q.shape[-1], k.shape[-2], (q_rope.shape[-1] if q_rope is not None else 0)


def workspace_size(desc: SagDesc) -> int:
    """Phase 1: validate and return the workspace size in bytes."""
    n = ctypes.c_size_t(0)
    st = load().sel_attn_grad_workspace_size(ctypes.byref(desc), ctypes.byref(n))
    if st != SAG_OK:
        raise SagError(st, "sel_attn_grad_workspace_size")
    return n.value


def plan_info(desc: SagDesc) -> SagPlanInfo:
    """Launch plan of a problem (host only)."""
    info = SagPlanInfo()
    st = load().sel_attn_grad_plan_info(ctypes.byref(desc), ctypes.byref(info))
    if st != SAG_OK:
        raise SagError(st, "sel_attn_grad_plan_info")
    return info


def sel_attn_grad(desc: SagDesc, query, key, value, attention_out, attention_out_grad,
                  softmax_max, softmax_sum, topk_indices, dq, dk, dv, workspace,
                  workspace_bytes: int, stream, main_start=None, main_stop=None) -> None:
    """Phase 2 on raw device pointers (ints); raises on a non-OK status.

    ``main_start`` / ``main_stop`` are optional raw cudaEvent_t handles recorded
    around the main backward kernel (``sel_attn_grad_timed``).
    """
    lib = load()
    if main_start is None and main_stop is None:
        st = lib.sel_attn_grad(ctypes.byref(desc), query, key, value, attention_out,
                               attention_out_grad, softmax_max, softmax_sum, topk_indices,
                               dq, dk, dv, workspace, workspace_bytes, stream)
    else:
        st = lib.sel_attn_grad_timed(ctypes.byref(desc), query, key, value, attention_out,
                                     attention_out_grad, softmax_max, softmax_sum, topk_indices,
                                     dq, dk, dv, workspace, workspace_bytes, stream, main_start,
                                     main_stop)
    if st != SAG_OK:
        raise SagError(st, "sel_attn_grad")


def selftest_wait_timeout(workspace, limit_ns: int, stream) -> None:
    """Enqueue the bounded-wait self-test (see include/selattn.h); read its
    status with ``query_error``."""
    lib = load()
    f = lib.sel_attn_selftest_wait_timeout
    f.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p]
    f.restype = ctypes.c_int
    st = f(workspace, int(limit_ns), stream)
    if st != SAG_OK:
        raise SagError(st, "sel_attn_selftest_wait_timeout")


def query_error(workspace, stream) -> int:
    """Wait for the stream; return the status the device recorded."""
    return load().sel_attn_grad_query_error(workspace, stream)


def backward(q, k, v, o, dy, softmax_max, softmax_sum, topk, cu_seqlens_q, cu_seqlens_kv, scale,
             block_size, block_count, deterministic=False, out=None, workspace=None, stream=None,
             check=False, q_rope=None, k_rope=None):
    """torch-tensor convenience over the C ABI (allocation and marshalling only).

    All tensors must be contiguous CUDA tensors, TND ([T, N, D]) or BSND
    ([B, S, N, D], 4-D); returns (dq, dk, dv), or (dq, dk, dv, dq_rope,
    dk_rope) with the rope split.  With ``check`` the device status is read
    back (this synchronizes the stream).
    """
    import torch
    if not q.is_cuda:
        raise ValueError("inputs must be CUDA tensors (there is no CPU path)")
    dtype = SAG_FP16 if q.dtype == torch.float16 else SAG_BF16
    layout, s1_max, s2_max, n1, d_qk, n2, d_rope = _layout_of(q, k, q_rope)
    d_v = v.shape[-1]
    desc = make_desc(cu_seqlens_q, cu_seqlens_kv, n1, n2, d_qk, d_v, block_size, block_count, scale,
                     dtype, deterministic, layout, s1_max, s2_max, d_rope)
    need = workspace_size(desc)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
        if d_rope:
            out = out + (torch.empty_like(q_rope), torch.empty_like(k_rope))
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    named = dict(query=q, key=k, value=v, attention_out=o, attention_out_grad=dy, softmax_max=softmax_max,
                 softmax_sum=softmax_sum, topk_indices=topk, dq=out[0], dk=out[1], dv=out[2])
    if d_rope:
        named.update(query_rope=q_rope, key_rope=k_rope, dq_rope=out[3], dk_rope=out[4])
    for t in named.values():
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    io = make_io(**{k_: t.data_ptr() for k_, t in named.items()})
    sel_attn_grad_ex(desc, io, workspace.data_ptr(), need, stream.cuda_stream)
    if check:
        st = query_error(workspace.data_ptr(), stream.cuda_stream)
        if st != SAG_OK:
            raise SagError(st, "device")
    return out


def fwd_workspace_size(desc: SagDesc) -> int:
    """Forward phase 1: validate and return the forward's workspace size."""
    n = ctypes.c_size_t(0)
    st = load().sel_attn_fwd_workspace_size(ctypes.byref(desc), ctypes.byref(n))
    if st != SAG_OK:
        raise SagError(st, "sel_attn_fwd_workspace_size")
    return n.value


def sel_attn_fwd(desc: SagDesc, query, key, value, topk_indices, attention_out, softmax_max,
                 softmax_sum, workspace, workspace_bytes: int, stream, passes_start=None,
                 passes_stop=None) -> None:
    """Forward phase 2 on raw device pointers (ints); raises on a non-OK status."""
    lib = load()
    if passes_start is None and passes_stop is None:
        st = lib.sel_attn_fwd(ctypes.byref(desc), query, key, value, topk_indices, attention_out,
                              softmax_max, softmax_sum, workspace, workspace_bytes, stream)
    else:
        st = lib.sel_attn_fwd_timed(ctypes.byref(desc), query, key, value, topk_indices,
                                    attention_out, softmax_max, softmax_sum, workspace,
                                    workspace_bytes, stream, passes_start, passes_stop)
    if st != SAG_OK:
        raise SagError(st, "sel_attn_fwd")


def forward(q, k, v, topk, cu_seqlens_q, cu_seqlens_kv, scale, block_size, block_count,
            out=None, workspace=None, stream=None, check=False, q_rope=None, k_rope=None):
    """torch-tensor convenience over the forward's C ABI: returns
    (attention_out [.., n1, d_v], softmax_max [.., n1, 8], softmax_sum [.., n1, 8])
    in the layout of q (TND or 4-D BSND)."""
    import torch
    if not q.is_cuda:
        raise ValueError("inputs must be CUDA tensors (there is no CPU path)")
    dtype = SAG_FP16 if q.dtype == torch.float16 else SAG_BF16
    layout, s1_max, s2_max, n1, d_qk, n2, d_rope = _layout_of(q, k, q_rope)
    d_v = v.shape[-1]
    desc = make_desc(cu_seqlens_q, cu_seqlens_kv, n1, n2, d_qk, d_v, block_size, block_count, scale,
                     dtype, False, layout, s1_max, s2_max, d_rope)
    need = fwd_workspace_size(desc)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    lead = tuple(q.shape[:-1])
    if out is None:
        out = (torch.empty(lead + (d_v,), dtype=q.dtype, device=q.device),
               torch.empty(lead + (8,), dtype=torch.float32, device=q.device),
               torch.empty(lead + (8,), dtype=torch.float32, device=q.device))
    o, smax, ssum = out
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    named = dict(query=q, key=k, value=v, topk_indices=topk, attention_out=o, softmax_max=smax, softmax_sum=ssum)
    if d_rope:
        named.update(query_rope=q_rope, key_rope=k_rope)
    for t in named.values():
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    io = make_io(**{k_: t.data_ptr() for k_, t in named.items()})
    sel_attn_fwd_ex(desc, io, workspace.data_ptr(), need, stream.cuda_stream)
    if check:
        st = query_error(workspace.data_ptr(), stream.cuda_stream)
        if st != SAG_OK:
            raise SagError(st, "device")
    return o, smax, ssum


# ------------------------------------------------------------ lightning indexer
class SliDesc(ctypes.Structure):
    """Mirror of ``sli_desc`` in include/selattn.h."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("n1", ctypes.c_int32), ("n2", ctypes.c_int32), ("d", ctypes.c_int32),
        ("topk", ctypes.c_int32), ("dtype", ctypes.c_int32), ("deterministic", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("cu_seqlens_q", ctypes.POINTER(ctypes.c_int32)), ("cu_seqlens_kv", ctypes.POINTER(ctypes.c_int32)),
        ("s1_max", ctypes.c_int32), ("s2_max", ctypes.c_int32),
    ]


class SliIo(ctypes.Structure):
    """Mirror of ``sli_io`` in include/selattn.h (device pointers as ints)."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("query", "key", "weights", "dy", "indices", "dq", "dk", "dweights")]


def _lib_indexer():
    lib = load()
    if not getattr(lib, "_sli_ready", False):
        D, IO, vp, sz = ctypes.POINTER(SliDesc), ctypes.POINTER(SliIo), ctypes.c_void_p, ctypes.c_size_t
        lib.lightning_indexer_grad_workspace_size.argtypes = [D, ctypes.POINTER(sz)]
        lib.lightning_indexer_grad_workspace_size.restype = ctypes.c_int
        lib.lightning_indexer_grad.argtypes = [D, IO, vp, sz, vp]
        lib.lightning_indexer_grad.restype = ctypes.c_int
        lib._sli_ready = True
    return lib


def make_indexer_desc(cu_seqlens_q, cu_seqlens_kv, n1, n2, d, topk, dtype=SAG_BF16, deterministic=False,
                      layout=SAG_LAYOUT_TND, s1_max=0, s2_max=0) -> SliDesc:
    cq = (ctypes.c_int32 * len(cu_seqlens_q))(*[int(x) for x in cu_seqlens_q])
    ck = (ctypes.c_int32 * len(cu_seqlens_kv))(*[int(x) for x in cu_seqlens_kv])
    desc = SliDesc(batch=len(cu_seqlens_q) - 1, n1=n1, n2=n2, d=d, topk=topk, dtype=dtype,
                   deterministic=1 if deterministic else 0, layout=int(layout),
                   cu_seqlens_q=ctypes.cast(cq, ctypes.POINTER(ctypes.c_int32)),
                   cu_seqlens_kv=ctypes.cast(ck, ctypes.POINTER(ctypes.c_int32)), s1_max=int(s1_max),
                   s2_max=int(s2_max))
    desc._keep = (cq, ck)
    return desc


def indexer_workspace_size(desc: SliDesc) -> int:
    n = ctypes.c_size_t(0)
    st = _lib_indexer().lightning_indexer_grad_workspace_size(ctypes.byref(desc), ctypes.byref(n))
    if st != SAG_OK:
        raise SagError(st, "lightning_indexer_grad_workspace_size")
    return n.value


def lightning_indexer_grad(desc: SliDesc, io: SliIo, workspace, workspace_bytes: int, stream) -> None:
    """Phase 2 on raw device pointers (ints); raises on a non-OK status."""
    st = _lib_indexer().lightning_indexer_grad(ctypes.byref(desc), ctypes.byref(io), workspace, workspace_bytes,
                                               stream)
    if st != SAG_OK:
        raise SagError(st, "lightning_indexer_grad")


def indexer_backward(q, k, weights, dy, indices, cu_seqlens_q, cu_seqlens_kv, deterministic=False, out=None,
                     workspace=None, stream=None, check=False):
    """torch-tensor convenience for the lightning-indexer backward: returns
    (dq, dk, dweights).  TND tensors ([T, N, D]) or BSND (4-D, padded)."""
    import torch
    if not q.is_cuda:
        raise ValueError("inputs must be CUDA tensors (there is no CPU path)")
    dtype = SAG_FP16 if q.dtype == torch.float16 else SAG_BF16
    bsnd = q.dim() == 4
    layout = SAG_LAYOUT_BSND if bsnd else SAG_LAYOUT_TND
    desc = make_indexer_desc(cu_seqlens_q, cu_seqlens_kv, q.shape[-2], k.shape[-2], q.shape[-1], indices.shape[-1],
                             dtype, deterministic, layout, q.shape[1] if bsnd else 0, k.shape[1] if bsnd else 0)
    need = indexer_workspace_size(desc)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(weights))
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    named = dict(query=q, key=k, weights=weights, dy=dy, indices=indices, dq=out[0], dk=out[1], dweights=out[2])
    for t in named.values():
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    io = SliIo(**{k_: t.data_ptr() for k_, t in named.items()})
    lightning_indexer_grad(desc, io, workspace.data_ptr(), need, stream.cuda_stream)
    if check:
        st = query_error(workspace.data_ptr(), stream.cuda_stream)
        if st != SAG_OK:
            raise SagError(st, "device")
    return out
