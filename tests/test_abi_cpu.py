"""C ABI checks that need no GPU: the library loads, exports every entry point
declared in include/selattn.h, and phase 1 (parameter validation + workspace
size, host only) follows the operator's documented constraints."""
import json
import os
import re

import pytest

import sparse_attention_backward_gb300 as sab
from sparse_attention_backward_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLD = json.load(open(os.path.join(ROOT, "tests", "golden", "constraints.json")))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return sab.load()


def _declared():
    hdrs = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
            if f.endswith(".h")]
    names = set()
    for h in hdrs:
        txt = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b((?:sel_attn|lightning_indexer)_\w*)\s*\(", txt))
    return names


def test_exports_every_declared_entry_point(lib):
    names = _declared()
    assert set(sab.EXPORTED) <= names
    for n in names:
        assert hasattr(lib, n), n


def _desc(**kw):
    a = dict(cu_seqlens_q=[0, 256], cu_seqlens_kv=[0, 256], n1=4, n2=1, d_qk=192, d_v=128,
             block_size=16, block_count=4, scale=192 ** -0.5, dtype=sab.SAG_BF16, deterministic=False)
    a.update(kw)
    return sab.make_desc(**a)


def _status(d):
    import ctypes
    n = ctypes.c_size_t(0)
    return sab.load().sel_attn_grad_workspace_size(ctypes.byref(d), ctypes.byref(n)), n.value


def test_valid_descriptor_gives_workspace(lib):
    st, n = _status(_desc())
    assert st == sab.SAG_OK and n > 0
    st2, n2 = _status(_desc(deterministic=True))
    assert st2 == sab.SAG_OK and n2 > 0


G = sab.SAG_ERR_SHAPE


@pytest.mark.parametrize("kw,want", [
    (dict(block_size=8), G),                                   # below 16 / not a multiple of 16
    (dict(block_size=24), G),                                  # not a multiple of 16
    (dict(block_size=GOLD["block_size_max"] + 16, cu_seqlens_kv=[0, 1024]), G),
    (dict(block_count=0), G),
    (dict(block_count=GOLD["block_count"][1] + 1), G),
    (dict(block_size=64, block_count=128, cu_seqlens_kv=[0, 8192]), G),   # 64*128 = 8192 not < 8192
    (dict(block_size=64, block_count=127, cu_seqlens_kv=[0, 8128]), sab.SAG_OK),
    (dict(n1=33, n2=1), G),                                    # G = 33 > 32
    (dict(n1=32, n2=1), sab.SAG_OK),                           # G = 32
    (dict(n1=129, n2=1), G),
    (dict(n1=6, n2=4), G),                                     # N1 not a multiple of N2
    (dict(n1=256, n2=128), G),                                 # N1 > 128
    (dict(n1=128, n2=128), sab.SAG_OK),
    (dict(d_qk=64), G),
    (dict(d_v=96), G),
    (dict(d_qk=128, d_v=192), sab.SAG_OK),                     # K and V head dims may differ
    (dict(cu_seqlens_kv=[0, 250]), G),                         # S2 not a multiple of the block size
    (dict(cu_seqlens_kv=[0, 48]), G),                          # S2 < size * count
    (dict(cu_seqlens_kv=[0, 64]), sab.SAG_OK),                 # S2 == size * count (reading: >=)
    (dict(cu_seqlens_q=[0, 0, 10], cu_seqlens_kv=[0, 64, 128]), sab.SAG_OK),   # empty query batch
    (dict(cu_seqlens_q=[0, GOLD["S"][1] + 1], cu_seqlens_kv=[0, 256]), G),     # S1 > 128K
    (dict(cu_seqlens_kv=[0, GOLD["S"][1] + 16]), G),           # S2 > 128K
    (dict(cu_seqlens_q=[1, 256]), G),                          # prefix sums start at 0
    (dict(cu_seqlens_q=[0, 0]), G),                            # T1 >= 1
    (dict(dtype=2), sab.SAG_ERR_DTYPE),
    (dict(deterministic=2), G),
    (dict(scale=float("nan")), G),
])
def test_phase1_follows_documented_constraints(lib, kw, want):
    d = _desc(**{k: v for k, v in kw.items() if k != "deterministic"})
    if "deterministic" in kw:
        d.deterministic = kw["deterministic"]
    st, _ = _status(d)
    assert st == want, (kw, st, sab.status_string(st))


def test_null_arguments(lib):
    import ctypes
    n = ctypes.c_size_t(0)
    assert lib.sel_attn_grad_workspace_size(None, ctypes.byref(n)) == sab.SAG_ERR_NULL
    assert lib.sel_attn_grad_workspace_size(ctypes.byref(_desc()), None) == sab.SAG_ERR_NULL
    d = _desc()
    d.cu_seqlens_q = None
    assert _status(d)[0] == sab.SAG_ERR_NULL


def test_status_strings(lib):
    for st in range(10):
        assert sab.status_string(st) and sab.status_string(st) != "unknown status"
    assert sab.status_string(99) == "unknown status"


def test_golden_totals_match_limits():
    # the selection limit and stat lane count the validation encodes
    assert GOLD["selected_keys_below"] == 128 * 64 and GOLD["stat_lanes"] == 8


def _fwd_status(d):
    import ctypes
    n = ctypes.c_size_t(0)
    return sab.load().sel_attn_fwd_workspace_size(ctypes.byref(d), ctypes.byref(n)), n.value


def test_forward_phase1(lib):
    st, n = _fwd_status(_desc())
    assert st == sab.SAG_OK and n > 0
    # the forward's sums are order-dependent: no deterministic mode
    assert _fwd_status(_desc(deterministic=True))[0] == sab.SAG_ERR_UNSUPPORTED
    # tensor-core shapes only (d_v == 128)
    assert _fwd_status(_desc(d_v=192))[0] == sab.SAG_ERR_UNSUPPORTED
    # the backward's shape checks apply unchanged
    assert _fwd_status(_desc(block_size=24))[0] == sab.SAG_ERR_SHAPE


# ------------------------------------------------ launch plans (host only)
def test_plan_default_and_deterministic(lib):
    d = _desc()
    info = sab.plan_info(d)
    # preprocess, histogram, 3 scan passes, fill, main kernel, dQ cast (the
    # default mode takes the buckets unsorted)
    assert info.launches == 8 and info.token_chunks == 1 and info.main_kernel == 1
    assert info.workspace_bytes == sab.workspace_size(d)
    det = sab.plan_info(_desc(deterministic=True))
    # the bucket sort, then one chunk: main kernel (stores dS) and the fixed-order dQ pass
    assert det.token_chunks == 1 and det.launches == 7 + 2
    # items: key blocks (batch, KV head, block id)
    assert info.items == 256 // 16


def test_plan_items_follow_batches_and_heads(lib):
    d = _desc(cu_seqlens_q=[0, 100, 300], cu_seqlens_kv=[0, 256, 768], n1=8, n2=2, block_size=64,
              block_count=4)
    assert sab.plan_info(d).items == 2 * (256 // 64) + 2 * (512 // 64)


def test_plan_kernel_choice(lib, monkeypatch):
    assert sab.plan_info(_desc()).main_kernel == 1                    # tensor cores
    assert sab.plan_info(_desc(d_qk=128, d_v=192)).main_kernel == 0   # Dv = 192: CUDA cores
    monkeypatch.setenv("SELATTN_FORCE_CUDA_CORE", "1")
    assert sab.plan_info(_desc()).main_kernel == 0


def test_plan_token_windows(lib, monkeypatch):
    monkeypatch.setenv("SELATTN_WINDOW_TOKENS", "64")
    w = sab.plan_info(_desc())
    # windowed: buckets sorted (window starts are found by token), dK / dV
    # reduced as partials, so their cast runs too
    assert w.launches == 10
    monkeypatch.delenv("SELATTN_WINDOW_TOKENS")
    assert sab.plan_info(_desc()).launches == 8


def test_deterministic_workspace_holds_ds_not_dq(lib):
    # default: fp32 dQ accumulator [T1 * n1 * d_qk]; deterministic: dS in the
    # dtype for the token chunk [T1, n2, count, G, bs] -- here 2 B * 256 * 1 * 4 *
    # 4 * 16 = 131072 B against 4 B * 256 * 4 * 192 = 786432 B
    dflt = sab.workspace_size(_desc())
    det = sab.workspace_size(_desc(deterministic=True))
    assert dflt - det == pytest.approx(786432 - 131072, abs=4 * 256)


def test_forward_workspace_matches_default_backward(lib):
    # the forward carves the same regions (O accumulator in the dQ slot)
    assert _fwd_status(_desc())[1] == sab.workspace_size(_desc())
    assert _fwd_status(_desc(d_qk=128))[1] == sab.workspace_size(_desc(d_qk=128))


def test_selections_beyond_the_32_bit_index_are_unsupported(lib):
    """16 batches of 128K tokens (T1 = 2M, the documented maximum), N2 = 16
    and 128 blocks of 16 are within the constraints, but make 2^32 selections:
    more than the inverted index's 32-bit offsets hold."""
    cu = [i * 128 * 1024 for i in range(17)]
    big = dict(cu_seqlens_q=cu, cu_seqlens_kv=cu, n1=16, n2=16, d_qk=128, d_v=128, block_size=16,
               block_count=128, scale=0.1)
    assert _status(_desc(**big))[0] == sab.SAG_ERR_UNSUPPORTED
    # half the heads: 2^31 selections, still one too many
    assert _status(_desc(**dict(big, n1=8, n2=8)))[0] == sab.SAG_ERR_UNSUPPORTED
    # a quarter: 2^30 selections fit
    assert _status(_desc(**dict(big, n1=4, n2=4)))[0] == sab.SAG_OK


def test_bsnd_and_rope_descriptors(lib):
    """Layout and rope fields of the descriptor: BSND takes padded lengths that
    bound every batch's valid length; TND takes none; the rope part is 64 wide
    on a 128-wide query / key (192 in all) with d_v = 128."""
    bsnd = dict(cu_seqlens_q=[0, 100, 150], cu_seqlens_kv=[0, 256, 384], layout=sab.SAG_LAYOUT_BSND,
                s1_max=128, s2_max=256)
    assert _status(_desc(**bsnd))[0] == sab.SAG_OK
    assert _status(_desc(**dict(bsnd, s1_max=99)))[0] == G          # a batch longer than its padding
    assert _status(_desc(**dict(bsnd, s2_max=250)))[0] == G         # not a multiple of the block size
    assert _status(_desc(**dict(bsnd, s1_max=0)))[0] == G
    assert _status(_desc(s1_max=128))[0] == G                        # TND takes no padded lengths
    assert _status(_desc(layout=2))[0] == G
    rope = dict(d_qk=128, d_v=128, d_rope=64)
    assert _status(_desc(**rope))[0] == sab.SAG_OK
    assert _status(_desc(**dict(rope, d_rope=32)))[0] == G
    assert _status(_desc(**dict(rope, d_v=192)))[0] == sab.SAG_ERR_UNSUPPORTED
    assert _status(_desc(**dict(rope, d_qk=192)))[0] == G            # 256 in all
    # the rope split: same workspace as the unsplit 192-wide problem
    assert _status(_desc(**rope))[1] == _status(_desc(d_qk=192, d_v=128))[1]


def test_dq_path_of_the_plan(lib, monkeypatch):
    """The deterministic mode always forms dQ by a fixed-order pass: from the
    stored dS, or (small blocks and groups: the small-group workload) from
    per-slot fp32 partials.  The default mode takes the pass from the stored
    dS on long context, max selection and the varlen case (under 3x the
    reductions' bytes per selected block) and reduces dQ in the main kernel
    on the others; SELATTN_DQ_PASS forces either."""
    import synth
    for w in synth.WORKLOADS:
        for det in (False, True):
            d = sab.make_desc(w.cu_q, w.cu_kv, w.n1, w.n2, w.d_qk, w.d_v, w.block_size, w.block_count, w.scale,
                              sab.SAG_FP16 if w.dtype == "f16" else sab.SAG_BF16, det)
            if det:
                want = 2 if w.name == "small_group" else 1
            else:
                want = 1 if w.name in ("varlen", "long_context", "max_selection") else 0
            assert sab.plan_info(d).dq_path == want, (w.name, det)
            if not det:
                monkeypatch.setenv("SELATTN_DQ_PASS", "0")
                assert sab.plan_info(d).dq_path == 0
                monkeypatch.delenv("SELATTN_DQ_PASS")
    # the per-slot partials take count * halves * d_qk fp32 per query row
    w = synth.WORKLOADS[4]
    d = sab.make_desc(w.cu_q, w.cu_kv, w.n1, w.n2, w.d_qk, w.d_v, w.block_size, w.block_count, w.scale,
                      sab.SAG_FP16, True)
    monkeypatch.setenv("SELATTN_DQ_SLOTS", "0")
    small = sab.plan_info(d).workspace_bytes
    monkeypatch.setenv("SELATTN_DQ_SLOTS", "1")
    big = sab.plan_info(d).workspace_bytes
    t1 = w.cu_q[-1]
    parts = t1 * w.n1 * w.block_count * w.d_qk * 4
    dss = t1 * w.n2 * w.block_count * (w.n1 // w.n2) * w.block_size * 2
    assert big - small == parts - dss
    monkeypatch.delenv("SELATTN_DQ_SLOTS")
    monkeypatch.setenv("SELATTN_DQ_PASS", "1")
    w = synth.WORKLOADS[2]
    d = sab.make_desc(w.cu_q, w.cu_kv, w.n1, w.n2, w.d_qk, w.d_v, w.block_size, w.block_count, w.scale)
    info = sab.plan_info(d)
    # one token chunk: the default mode leaves the buckets unsorted
    assert info.dq_path == 1 and info.token_chunks == 1 and info.launches == 8



def _li_status(**kw):
    import ctypes
    a = dict(cu_seqlens_q=[0, 300, 1000], cu_seqlens_kv=[0, 300, 1000], n1=32, n2=1, d=128, topk=128)
    a.update(kw)
    d = sab.make_indexer_desc(**a)
    n = ctypes.c_size_t(0)
    return sab._lib_indexer().lightning_indexer_grad_workspace_size(ctypes.byref(d), ctypes.byref(n)), n.value


def test_indexer_descriptor_validation(lib):
    st, n = _li_status()
    # header + row starts / ends + fp32 dK [1000, 1, 128] + fp32 dW [1000, 32], 256-byte aligned
    assert st == sab.SAG_OK and n >= 1000 * 128 * 4 + 1000 * 32 * 4
    assert _li_status(topk=301)[0] == G                                # a batch shorter than topk
    assert _li_status(n1=30, n2=4)[0] == G                             # n1 not a multiple of n2
    assert _li_status(n1=128)[0] == sab.SAG_ERR_UNSUPPORTED            # G = 128 > 64
    assert _li_status(d=64)[0] == sab.SAG_ERR_UNSUPPORTED
    assert _li_status(deterministic=True)[0] == sab.SAG_ERR_UNSUPPORTED
    assert _li_status(layout=sab.SAG_LAYOUT_BSND, s1_max=700, s2_max=700)[0] == sab.SAG_OK
    assert _li_status(layout=sab.SAG_LAYOUT_BSND, s1_max=699, s2_max=700)[0] == G
    assert _li_status(s1_max=700)[0] == G


def test_default_dq_path_rule_by_kernel(lib):
    """The default mode's dQ path by bytes per query row.  For the main
    tensor-core kernel (G >= 8) the pass is taken under 3x the reductions'
    bytes counted once per selected block; the split schedule (G <= 4) and the
    CUDA-core kernel keep the stricter rule (under half the reductions' bytes,
    counted per 64-key tile)."""
    kv = dict(cu_seqlens_q=[0, 512], cu_seqlens_kv=[0, 2048])

    def path(**kw):
        return sab.plan_info(_desc(**dict(kv, **kw))).dq_path

    # pass / reductions per row: 16 blocks of 64, Dqk 192
    assert path(n1=16, n2=1, block_size=64, block_count=16) == 1     # G = 16: 28672 / 12288 = 2.33
    assert path(n1=32, n2=1, block_size=64, block_count=16) == 1     # G = 32: 16384 / 12288 = 1.33
    assert path(n1=8, n2=1, block_size=64, block_count=16) == 0      # G = 8: 53248 / 12288 = 4.33
    assert path(n1=16, n2=1, block_size=128, block_count=8) == 0     # 128-key blocks, G = 16: 28672 / 6144 = 4.67
    assert path(n1=32, n2=1, block_size=128, block_count=8) == 1     # G = 32: 16384 / 6144 = 2.67
    # the split schedule: G = 4, 16-key blocks (ratio 2.08, which the main kernel's rule would take)
    assert path(n1=4, n2=1, block_size=16, block_count=4) == 0
    # the CUDA-core kernel (Dv = 192), G = 16, 64-key blocks
    assert path(n1=16, n2=1, d_qk=128, d_v=192, block_size=64, block_count=16) == 0


def test_default_and_deterministic_share_the_pass_workspace(lib):
    """On a problem whose default mode takes the fixed-order pass in one token
    chunk, both modes carve the same workspace (dS buffer, no fp32 dQ
    accumulator); the default mode launches one kernel fewer (no bucket sort)."""
    kw = dict(cu_seqlens_q=[0, 512], cu_seqlens_kv=[0, 2048], n1=16, n2=1, block_size=64, block_count=16)
    d = sab.plan_info(_desc(**kw))
    t = sab.plan_info(_desc(deterministic=True, **kw))
    assert d.dq_path == t.dq_path == 1 and d.token_chunks == t.token_chunks == 1
    assert d.workspace_bytes == t.workspace_bytes
    assert d.launches + 1 == t.launches


def test_default_dq_path_rule_off_the_tensor_core_pass(lib):
    """Block sizes the tensor-core dQ pass does not take (here 48 keys, G = 16:
    the main kernel's rule would pick the pass) keep the stricter rule."""
    kw = dict(cu_seqlens_q=[0, 512], cu_seqlens_kv=[0, 1536], n1=16, n2=1, block_size=48, block_count=16)
    assert sab.plan_info(_desc(**kw)).dq_path == 0
