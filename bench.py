#!/usr/bin/env python
"""Benchmark of the GB300 selected-attention backward (one JSON line on rank 0).

A step is one full backward call (preprocess, index inversion, main kernel,
dQ finish) on one synthetic batch of the chosen workload, inputs resident in
HBM.  The default workload is the long-context one (B=1, S=32768, N1=64,
N2=4, Dqk=192, Dv=128, bf16, 16 blocks of 64).  Its inputs (Q alone is
805 MB) are larger than the 129 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config I]
                    [--deterministic] [--impl ours|reference]

Under torchrun each rank runs its own independent problem (weak scaling, no
collective on the data path); the time is the max over ranks.
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "selected-attn backward TFLOP/s and % of GB300 bf16 roofline; ms per call"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=2, help="workload index (0..4)")
    ap.add_argument("--deterministic", action="store_true")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU-baseline sample budget")
    ap.add_argument("--forward", action="store_true",
                    help="time the selected-attention forward (O and the softmax stats) instead")
    ap.add_argument("--seq", type=int, default=0,
                    help="override every batch's query and key length (smaller profiling captures)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload timings added to the line (long context, max selection, small group)")
    ap.add_argument("--op", choices=["backward", "indexer"], default="backward",
                    help="indexer: the lightning-indexer backward on its long workload instead")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


def host_cpu() -> str:
    """Host CPU model as /proc/cpuinfo names it (Arm parts by implementer / part id)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return "unknown CPU"
    for key in ("model name", "Model"):
        for line in info.splitlines():
            if line.split(":")[0].strip() == key:
                return line.split(":", 1)[1].strip()
    impl = part = None
    for line in info.splitlines():
        k = line.split(":")[0].strip()
        if k == "CPU implementer" and impl is None:
            impl = line.split(":", 1)[1].strip()
        elif k == "CPU part" and part is None:
            part = line.split(":", 1)[1].strip()
    return f"Arm CPU implementer {impl} part {part}" if impl else "unknown CPU"


# The sources the profiled kernels are built from: their translation units,
# the shared device headers and the C ABI header.  "main" is the main kernel
# with in-kernel dQ reductions, "main_dq_pass" the main kernel storing dS and
# the fixed-order dQ pass after it.
KERNEL_SOURCES = {"main": ["bwd_tc.cu"], "main_dq_pass": ["bwd_tc.cu", "dq_tc.cu"], "forward": ["fwd_tc.cu"]}


def kernel_source_hash(kernel: str = "main") -> str:
    csrc = os.path.join(ROOT, "sparse_attention_backward_gb300", "csrc")
    files = [os.path.join(csrc, f) for f in KERNEL_SOURCES[kernel]] + sorted(glob.glob(os.path.join(csrc, "*.cuh")))
    files.append(os.path.join(ROOT, "include", "selattn.h"))
    h = hashlib.sha256()
    for p in files:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, det: bool, mode: str = "", dq_path: int = 0):
    """DRAM bytes per call of the timed kernels from a committed ncu summary:
    the main kernel, plus the fixed-order dQ pass when the plan takes it
    (dq_path 1), or both forward passes with mode "forward".  Used only while
    those kernels' sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    key = f"{workload}:{mode or ('deterministic' if det else 'default')}"
    e = d.get(key)
    kernel = "forward" if mode == "forward" else ("main_dq_pass" if dq_path == 1 else "main")
    if not e or e.get("kernels") != kernel or e.get("kernel_source_hash") != kernel_source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                c = [x.strip() for x in line.split(",")]
                if len(c) < 9:
                    continue
                try:
                    sm.append(float(c[1]))
                    mx.append(float(c[2]))
                except ValueError:
                    continue
                for n, v in zip(names, c[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- CPU oracle
def _np16(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def oracle_sample(w, x, n_tokens, rng):
    """A bounded sample of the workload: n_tokens query tokens of batch 0 with
    the G heads of KV head 0 against their batch's keys (a full backward of
    those rows: dQ, and their dK / dV scatter).  When x carries no forward
    outputs (the reference arm) they come from the oracle forward of the
    sample, outside the timed call."""
    import oracle
    b, j, G = 0, 0, w.group
    q0, q1 = w.cu_q[b], w.cu_q[b + 1]
    toks = np.sort(rng.choice(np.arange(q0, q1), size=min(n_tokens, q1 - q0), replace=False))
    t = torch.as_tensor(toks, device=x["q"].device)
    k0, k1 = w.cu_kv[b], w.cu_kv[b + 1]
    hs = slice(j * G, (j + 1) * G)
    p = oracle.Problem(
        cu_q=np.array([0, len(toks)], np.int32), cu_kv=np.array([0, k1 - k0], np.int32), n1=G, n2=1,
        d_qk=w.d_qk, d_v=w.d_v, block_size=w.block_size, block_count=w.block_count, scale=w.scale,
        topk=x["topk"][t][:, j:j + 1].cpu().numpy(), q=_np16(x["q"][t][:, hs]),
        k=_np16(x["k"][k0:k1, j:j + 1]), v=_np16(x["v"][k0:k1, j:j + 1]), dy=_np16(x["dy"][t][:, hs]),
        stat_stride=8, kind=w.dtype)
    if "o" in x:
        p.o = _np16(x["o"][t][:, hs])
        p.smax = x["softmax_max"][t][:, hs].cpu().numpy()
        p.ssum = x["softmax_sum"][t][:, hs].cpu().numpy()
    else:
        o, m, l = oracle.forward(p)
        p.o = _np16(torch.from_numpy(o).to(w.torch_dtype))
        p.smax = np.repeat(m[..., None], 8, axis=-1).astype(np.float32)
        p.ssum = np.repeat(l[..., None], 8, axis=-1).astype(np.float32)
    flops = 2.0 * w.selected_keys * (3 * w.d_qk + 2 * w.d_v) * len(toks) * G
    return p, flops, len(toks)


def fwd_flops(w, n_rows) -> float:
    """Forward: 2 * L * (d_qk + d_v) per query head per token (S and P V)."""
    return 2.0 * w.selected_keys * (w.d_qk + w.d_v) * n_rows


def time_oracle(w, x, budget_s, seed=0, forward=False):
    """TFLOP/s of the oracle on a sample sized to about budget_s seconds."""
    import oracle
    run = oracle.forward if forward else oracle.backward
    rng = np.random.default_rng(seed)
    p, f, n = oracle_sample(w, x, 1, rng)
    t0 = time.perf_counter()
    run(p)
    per_token = max(1e-4, time.perf_counter() - t0)
    n = max(1, int(budget_s / per_token))
    p, f, n = oracle_sample(w, x, n, rng)
    if forward:
        f = fwd_flops(w, n * w.group)
    t0 = time.perf_counter()
    run(p)
    dt = time.perf_counter() - t0
    return f / dt / 1e12, dt, n


def run_reference(args, w, rank, world):
    x = synth.make_inputs(w, device="cpu" if w.t1 * w.n1 * w.d_qk < (1 << 27) else "cuda")
    per_step = min(5.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        time_oracle(w, x, per_step)
    vals, times = [], []
    for s in range(args.steps):
        v, dt, n = time_oracle(w, x, per_step, seed=s + 1)
        vals.append(v)
        times.append(dt)
    value = statistics.median(vals)
    sample = (f"{n} query tokens x {w.group} heads of KV head 0, batch 0 (full backward of those rows) "
              f"per step, ~{per_step:.1f} s each, one core of {host_cpu()} ({os.cpu_count()} cores)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w, args.deterministic),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(w, det):
    return {"workload": w.name, "batch": w.batch, "seq_len_q": [int(v) for v in np.diff(w.cu_q)[:4]] if w.batch <= 4 else "varlen",
            "n1": w.n1, "n2": w.n2, "d_qk": w.d_qk, "d_v": w.d_v, "block_size": w.block_size,
            "block_count": w.block_count, "dtype": w.dtype, "mode": "deterministic" if det else "default",
            "l2": "inputs larger than L2 (129 MB): no flush between steps" if w.algorithmic_bytes() > 4 * 129e6
            else "L2 flushed between steps (256 MB write)"}


# ------------------------------------------------------------ ranks (weak scaling)
def rank_seed(w, rank: int) -> int:
    """Each rank draws its own independent problem of the full workload size."""
    return w.seed + rank


def max_over_ranks(v: float, device) -> float:
    """The slowest rank's time (identity without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank: float, world: int, ms: float) -> float:
    """Whole-job TFLOP/s: every rank's work over the slowest rank's time."""
    return flops_per_rank * world / (ms * 1e-3) / 1e12


def runs_reference(rank: int) -> bool:
    """The reference arm (the oracle on host cores) runs on rank 0 only."""
    return rank == 0


# --------------------------------------------------------------------- ours
def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.op == "indexer":
        run_indexer(args, world, rank, local)
        return
    w = synth.WORKLOADS[args.config]
    if args.seq:
        cu = tuple(args.seq * i for i in range(w.batch + 1))
        w = w.with_(name=f"{w.name}_seq{args.seq}", cu_q=cu, cu_kv=cu)
    if args.impl == "reference":
        if runs_reference(rank):
            run_reference(args, w, rank, world)
        return

    import sparse_attention_backward_gb300 as sab
    sab.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    x = synth.make_inputs(w, device=dev, seed=rank_seed(w, rank))
    stream = torch.cuda.current_stream(dev)
    if args.forward:
        run_forward(args, w, x, dev, stream, world, rank, local)
        return
    # attentionOut and the [T1, N1, 8] stats: the library's forward (untimed)
    o, smax, ssum = sab.forward(x["q"], x["k"], x["v"], x["topk"], w.cu_q, w.cu_kv, w.scale, w.block_size,
                                w.block_count, check=True)
    x.update(o=o, softmax_max=smax, softmax_sum=ssum)
    desc = sab.make_desc(w.cu_q, w.cu_kv, w.n1, w.n2, w.d_qk, w.d_v, w.block_size, w.block_count,
                         w.scale, sab.SAG_FP16 if w.dtype == "f16" else sab.SAG_BF16, args.deterministic)
    info = sab.plan_info(desc)
    ws = torch.empty(int(info.workspace_bytes), dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"])
    ins = [x[k] for k in ("q", "k", "v", "o", "dy", "softmax_max", "softmax_sum", "topk")]
    flush = None
    if w.algorithmic_bytes() <= 4 * 129e6:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def call(ev0=None, ev1=None):
        sab.sel_attn_grad(desc, *[t.data_ptr() for t in ins], dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                          ws.data_ptr(), ws.numel(), stream.cuda_stream,
                          ev0.cuda_event if ev0 is not None else None,
                          ev1.cuda_event if ev1 is not None else None)

    for _ in range(args.warmup):
        call()
    st = sab.query_error(ws.data_ptr(), stream.cuda_stream)
    if st != sab.SAG_OK:
        raise sab.SagError(st, "device")

    K = args.steps
    mk0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    mk1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for e in mk0 + mk1:
        e.record(stream)   # creates the event so its handle can be passed down
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = Clocks(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    t0.record(stream)
    for i in range(K):
        if flush is not None:
            flush.zero_()
        call(mk0[i], mk1[i])
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    ms = t0.elapsed_time(t1) / K
    main_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(mk0, mk1))
    ms = max_over_ranks(ms, dev)

    flops = w.flops()
    value = job_throughput(flops, world, ms)
    pk, pk_src = peaks()
    peak = float(pk["bf16_tflops"])
    roofline_ms = max(flops / (peak * 1e12), w.algorithmic_bytes() / (float(pk["hbm_gbs"]) * 1e9)) * 1e3
    achieved = flops / (main_ms * 1e-3) / 1e12

    # end to end through the C ABI with host buffers (pinned), copies timed
    e2e = None
    if not args.no_e2e:
        host_in = [t.cpu().pin_memory() for t in ins]
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dq, dk, dv)]
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out)

        def e2e_step():
            for d, h in zip(ins, host_in):
                d.copy_(h, non_blocking=True)
            call()
            for h, d in zip(host_out, (dq, dk, dv)):
                h.copy_(d, non_blocking=True)
        for _ in range(max(1, min(args.warmup, 3))):
            e2e_step()
        torch.cuda.synchronize()
        ke = max(3, min(K, 10))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(ke):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        ems = a.elapsed_time(b) / ke
        ems = max_over_ranks(ems, dev)
        e2e = {"value": job_throughput(flops, world, ems), "unit": "TFLOP/s", "ms_per_step": ems,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, n = time_oracle(w, x, args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} query tokens x {w.group} heads (KV head 0, batch 0), full backward of those "
                         f"rows, {dt:.1f} s on one core of {host_cpu()} ({os.cpu_count()} cores)"}

    # the other large workloads, both modes, after this run's tensors are freed
    workloads = None
    if rank == 0 and world == 1 and not args.no_workloads and not args.seq and args.config == 2:
        del x, ins, dq, dk, dv, ws
        torch.cuda.empty_cache()
        workloads = time_workloads(dev, stream, peak)

    if rank == 0:
        traffic = profiled_traffic(w.name, args.deterministic, dq_path=int(info.dq_path))
        timed_kernels = ("main backward (stores dS) + fixed-order dQ pass" if info.dq_path == 1 else
                         "main backward (dQ slot partials) + slot sum" if info.dq_path == 2 else "main backward")
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": workload_config(w, args.deterministic),
            "pct_of_roofline": 100.0 * roofline_ms / ms,
            "roofline_ms": roofline_ms,
            "roofline": {"bound": "tensor", "kernel": timed_kernels, "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": f"{pk_src} bf16 burst",
                         "peak_sustained": float(pk.get("bf16_tflops_sustained", peak)),
                         "frac_sustained": achieved / float(pk.get("bf16_tflops_sustained", peak)),
                         "kernel_ms": main_ms, "traffic": traffic},
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": int(info.launches) * K,
            "clocks": clk,
            "workloads": workloads,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def time_workloads(dev, stream, peak):
    """ms per call (CUDA events, after warm-up; inputs beyond L2) of the
    long-context, max-selection and small-group workloads in both modes, with
    TFLOP/s and the fraction of the bf16 burst peak; the main kernel alone in
    parentheses (`main_ms`, which spans the dQ pass too when the plan's
    `dq_path` is 1 or 2).  Attention outputs and stats from the library's
    forward."""
    import sparse_attention_backward_gb300 as sab
    out = {}
    for idx, reps in ((2, 10), (3, 2), (4, 10)):
        w = synth.WORKLOADS[idx]
        x = synth.make_inputs(w, device=dev)
        o, m, l = sab.forward(x["q"], x["k"], x["v"], x["topk"], w.cu_q, w.cu_kv, w.scale, w.block_size,
                              w.block_count, check=True)
        ins = [x["q"], x["k"], x["v"], o, x["dy"], m, l, x["topk"]]
        outs = [torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"])]
        for det in (False, True):
            desc = sab.make_desc(w.cu_q, w.cu_kv, w.n1, w.n2, w.d_qk, w.d_v, w.block_size, w.block_count, w.scale,
                                 sab.SAG_FP16 if w.dtype == "f16" else sab.SAG_BF16, det)
            need = sab.workspace_size(desc)
            ws = torch.empty(need, dtype=torch.uint8, device=dev)
            e0 = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
            e1 = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
            for e in e0 + e1:
                e.record(stream)

            def call(a=None, b=None):
                sab.sel_attn_grad(desc, *[t.data_ptr() for t in ins], *[t.data_ptr() for t in outs], ws.data_ptr(),
                                  need, stream.cuda_stream, a.cuda_event if a is not None else None,
                                  b.cuda_event if b is not None else None)
            call()
            call()
            st = sab.query_error(ws.data_ptr(), stream.cuda_stream)
            if st != sab.SAG_OK:
                raise sab.SagError(st, "device")
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            t0.record(stream)
            for i in range(reps):
                call(e0[i], e1[i])
            t1.record(stream)
            torch.cuda.synchronize()
            ms = t0.elapsed_time(t1) / reps
            main_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(e0, e1))
            tf = w.flops() / (ms * 1e-3) / 1e12
            out[f"{w.name}:{'deterministic' if det else 'default'}"] = {
                "ms": ms, "main_ms": main_ms, "tflops": tf, "frac": tf / peak,
                "main_frac": w.flops() / (main_ms * 1e-3) / 1e12 / peak, "calls": reps,
                "dq_path": int(sab.plan_info(desc).dq_path)}
            del ws
        del x, o, m, l, ins, outs
        torch.cuda.empty_cache()
    return out


def run_forward(args, w, x, dev, stream, world, rank, local):
    """The forward: both tensor-core passes timed with events, the whole call
    (init, inversion, passes, finalize) timed per step."""
    import sparse_attention_backward_gb300 as sab
    desc = sab.make_desc(w.cu_q, w.cu_kv, w.n1, w.n2, w.d_qk, w.d_v, w.block_size, w.block_count,
                         w.scale, sab.SAG_FP16 if w.dtype == "f16" else sab.SAG_BF16, False)
    need = sab.fwd_workspace_size(desc)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    o = torch.empty((w.t1, w.n1, w.d_v), dtype=x["q"].dtype, device=dev)
    smax = torch.empty((w.t1, w.n1, 8), dtype=torch.float32, device=dev)
    ssum = torch.empty_like(smax)
    ins = [x[k] for k in ("q", "k", "v", "topk")]
    outs = [o, smax, ssum]

    def call(ev0=None, ev1=None):
        sab.sel_attn_fwd(desc, *[t.data_ptr() for t in ins], *[t.data_ptr() for t in outs], ws.data_ptr(), need,
                         stream.cuda_stream, ev0.cuda_event if ev0 is not None else None,
                         ev1.cuda_event if ev1 is not None else None)

    for _ in range(args.warmup):
        call()
    st = sab.query_error(ws.data_ptr(), stream.cuda_stream)
    if st != sab.SAG_OK:
        raise sab.SagError(st, "device")
    K = args.steps
    mk0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    mk1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for e in mk0 + mk1:
        e.record(stream)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = Clocks(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    t0.record(stream)
    for i in range(K):
        call(mk0[i], mk1[i])
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1) / K, dev)
    pass_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(mk0, mk1))
    flops = fwd_flops(w, w.t1 * w.n1)
    pk, pk_src = peaks()
    peak = float(pk["bf16_tflops"])
    achieved = flops / (pass_ms * 1e-3) / 1e12
    e2e = None
    if not args.no_e2e:
        host_in = [t.cpu().pin_memory() for t in ins]
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out)

        def e2e_step():
            for d, h in zip(ins, host_in):
                d.copy_(h, non_blocking=True)
            call()
            for h, d in zip(host_out, outs):
                h.copy_(d, non_blocking=True)
        for _ in range(max(1, min(args.warmup, 3))):
            e2e_step()
        torch.cuda.synchronize()
        ke = max(3, min(K, 10))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(ke):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(a.elapsed_time(b) / ke, dev)
        e2e = {"value": job_throughput(flops, world, ems), "unit": "TFLOP/s", "ms_per_step": ems,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, n = time_oracle(w, x, args.cpu_seconds, forward=True)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} query tokens x {w.group} heads (KV head 0, batch 0), forward of those rows, "
                         f"{dt:.1f} s on one core of {host_cpu()} ({os.cpu_count()} cores)"}
    if rank == 0:
        line = {
            "metric": "selected-attn forward TFLOP/s and % of GB300 bf16 roofline; ms per call",
            "value": job_throughput(flops, world, ms), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": dict(workload_config(w, False), mode="forward"),
            "roofline": {"bound": "tensor", "kernel": "forward passes (max, sum + P V)", "achieved": achieved,
                         "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                         "peak_source": f"{pk_src} bf16 burst", "kernel_ms": pass_ms,
                         "traffic": profiled_traffic(w.name, False, "forward")},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 10 * K, "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_indexer(args, world, rank, local):
    """The lightning-indexer backward on its long workload (8192 tokens, 64
    query heads on one key head, head dim 128, 2048 selections per token):
    one call per step (row starts staged, accumulators zeroed, the tensor-core
    kernel, two casts); flops = 3 contractions x 2 * d per (query head,
    selection)."""
    import oracle.indexer as li
    import sparse_attention_backward_gb300 as sab
    w = synth.INDEXER_WORKLOADS[2 if args.config == 2 else args.config]
    if args.seq:
        cu = tuple(args.seq * i for i in range(w.batch + 1))
        w = w.with_(name=f"{w.name}_seq{args.seq}", cu_q=cu, cu_kv=cu)
    if args.impl == "reference":
        if rank != 0:
            return
        x = synth.make_indexer_inputs(w, device="cpu")
    else:
        sab.load()
        torch.cuda.set_device(local)
        dev = torch.device("cuda", local)
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("nccl", device_id=dev)
        x = synth.make_indexer_inputs(w, device=dev, seed=w.seed + rank)
    flops = w.flops()

    def oracle_rate(budget_s, seed=0):
        rng = np.random.default_rng(seed)
        xs = {k: v.cpu() for k, v in x.items()}
        p = li.Problem(cu_q=np.asarray(w.cu_q, np.int32), cu_kv=np.asarray(w.cu_kv, np.int32), n1=w.n1, n2=w.n2,
                       d=w.d, topk=w.topk, idx=xs["idx"].numpy(), q=_np16(xs["q"]), k=_np16(xs["k"]),
                       w=_np16(xs["w"]), dy=xs["dy"].numpy(), kind=w.dtype)
        t0 = time.perf_counter()
        li.q_rows(p, [0])
        per = max(1e-4, time.perf_counter() - t0)
        n = max(1, int(budget_s / (2 * per)))    # dK of the same rows costs about as much again
        toks = np.sort(rng.choice(w.t1, min(n, w.t1), replace=False))
        t0 = time.perf_counter()
        li.backward_range(p, int(toks[0]), int(toks[0]) + len(toks))
        dt = time.perf_counter() - t0
        return 3 * 2.0 * w.d * w.topk * len(toks) * w.n1 / dt / 1e12, dt, len(toks)

    cfg = {"workload": w.name, "batch": w.batch, "seq_len_q": [int(v) for v in np.diff(w.cu_q)], "n1": w.n1,
           "n2": w.n2, "d": w.d, "topk": w.topk, "dtype": w.dtype, "mode": "default",
           "l2": "inputs larger than L2 (129 MB): no flush between steps"}
    metric = "lightning-indexer backward TFLOP/s and % of GB300 bf16 roofline; ms per call"
    if args.impl == "reference":
        per_step = min(5.0, 150.0 / max(1, args.steps + args.warmup))
        vals, times = [], []
        for s_ in range(args.warmup + args.steps):
            v, dt, n = oracle_rate(per_step, s_)
            if s_ >= args.warmup:
                vals.append(v)
                times.append(dt)
        value = statistics.median(vals)
        print(json.dumps({"impl": "reference", "metric": metric, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(times),
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": cfg,
                          "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                                           "sample": f"{n} consecutive query tokens (all heads) per step, one core "
                                                     f"of {host_cpu()}"},
                          "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return
    dev = x["q"].device
    stream = torch.cuda.current_stream(dev)
    desc = sab.make_indexer_desc(w.cu_q, w.cu_kv, w.n1, w.n2, w.d, w.topk,
                                 sab.SAG_FP16 if w.dtype == "f16" else sab.SAG_BF16)
    need = sab.indexer_workspace_size(desc)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    outs = (torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["w"]))
    io = sab.SliIo(query=x["q"].data_ptr(), key=x["k"].data_ptr(), weights=x["w"].data_ptr(), dy=x["dy"].data_ptr(),
                   indices=x["idx"].data_ptr(), dq=outs[0].data_ptr(), dk=outs[1].data_ptr(),
                   dweights=outs[2].data_ptr())

    def call():
        sab.lightning_indexer_grad(desc, io, ws.data_ptr(), need, stream.cuda_stream)

    for _ in range(args.warmup):
        call()
    st = sab.query_error(ws.data_ptr(), stream.cuda_stream)
    if st != sab.SAG_OK:
        raise sab.SagError(st, "device")
    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = Clocks(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    t0.record(stream)
    for _ in range(K):
        call()
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1) / K, dev)
    pk, pk_src = peaks()
    peak = float(pk["bf16_tflops"])
    achieved = flops / (ms * 1e-3) / 1e12
    e2e = None
    if not args.no_e2e:
        names = ("q", "k", "w", "dy", "idx")
        host_in = [x[k].cpu().pin_memory() for k in names]
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out)

        def e2e_step():
            for k_, h in zip(names, host_in):
                x[k_].copy_(h, non_blocking=True)
            call()
            for h, d in zip(host_out, outs):
                h.copy_(d, non_blocking=True)
        e2e_step()
        torch.cuda.synchronize()
        ke = max(3, min(K, 10))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(ke):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(a.elapsed_time(b) / ke, dev)
        e2e = {"value": job_throughput(flops, world, ems), "unit": "TFLOP/s", "ms_per_step": ems,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, n = oracle_rate(args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} consecutive query tokens (all heads), full backward of those rows, {dt:.1f} s on "
                         f"one core of {host_cpu()} ({os.cpu_count()} cores)"}
    if rank == 0:
        print(json.dumps({
            "metric": metric, "value": job_throughput(flops, world, ms), "unit": "TFLOP/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic", "config": cfg,
            "roofline": {"bound": "tensor", "kernel": "indexer backward (whole call)", "achieved": achieved,
                         "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                         "peak_source": f"{pk_src} bf16 burst", "kernel_ms": ms, "traffic": None},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 3 * K, "clocks": clk}), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
