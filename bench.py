"""Benchmark of one absorbed-MLA decode step on GB300.

A step is one pass of the whole path on one batch: split schedule, W_UK
absorption (with the q assembly: RoPE of q_pe at each new token's position),
paged absorbed decode, LSE combine and W_UV
un-absorption, on the DeepSeek-V3-shaped workload (B=64, H=128, s_q=1, every
context 4096 tokens, 576/512 dims, page 64, synthetic bf16 data).  The metric
is algorithmic TFLOP/s of the step; HBM GB/s and the fraction of the roofline
max(FLOPs / 2.25 PFLOP/s, bytes / 8 TB/s) ride along, and the `roofline` object
rates the dominant kernel (the mla_decode call) against the measured HBM peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

--workload picks another shape (mla_absorbed_decode_gb300/workloads.py): the
ragged, MTP (s_q = 2, causal) and long-context ones, the V3 shape over an FP8
(E4M3) cache (fp8_deepseek_v3_b64_h128_l4096: mla_decode_fp8, the FP8 tensor rate
in the roofline), and the V3.2-shaped top-2048 sparse decode over a bf16 or an
FP8 cache (sparse_b64_h128_l16384_top2048, sparse_fp8_b64_h128_l16384_top2048), the V3
step with FP8 projections (fp8proj_deepseek_v3_b64_h128_l4096: bmm_fp8), and the chunked
extend on the expanded path (extend_t512_l32768_h128_chunk4096: mla_extend_chunked).
Each timed step replays --inner passes (default 256) back to back from one CUDA graph,
cycling over enough copies of the inputs, weights and buffers that more than 512 MiB
is touched between two uses of a copy (L2 holds 126 MB), so that the timed region
lasts long enough for the clock samples; ms_per_step is per pass.  The decode call and
(with projections) each projection call are timed the same way on their own
(roofline.ms_per_launch, projections_back_to_back_us); components_us is an eager
per-call breakdown (events between the calls, host work included).
--impl reference times the CPU oracle (numpy float64) on a bounded sample of
the same workload per step.  With N > 1 (torchrun) every rank runs its own
replica of the workload (requests shard across GPUs with no exchange).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode TFLOP/s and HBM GB/s, % of GB300 roofline (1 GPU)"
SPEC_FLOPS = 2.25e15
SPEC_FLOPS_FP8 = 4.5e15   # nominal dense FP8 tensor rate (twice bf16)
SPEC_BW = 8.0e12
# the decode kernel and the host code that encodes its tensor maps (their L2 fill units set part
# of the traffic)
DECODE_KERNEL_SOURCES = ("mla_absorbed_decode_gb300/csrc/mla_decode.cu", "mla_absorbed_decode_gb300/csrc/mla_ptx.cuh",
                         "mla_absorbed_decode_gb300/csrc/mla_host.cu")


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def _source_digest():
    import hashlib
    h = hashlib.sha256()
    for rel in DECODE_KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic_per_launch(workload_name):
    """DRAM bytes per decode launch from a committed ncu summary, if it was taken on
    the current kernel source; otherwise None."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload_name)
    if not e or e.get("source_digest") != _source_digest():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return len(os.sched_getaffinity(0))


def oracle_sample_step(inp, kv_np, sel, with_proj):
    """One CPU oracle pass over the sampled requests; returns its algorithmic FLOPs."""
    import numpy as np
    import oracle
    from mla_absorbed_decode_gb300 import accounting as acc
    B, s_q, H, _ = inp["q"].shape
    flops = 0
    if with_proj:
        qn = inp["q_nope"].float().numpy().reshape(B, s_q, H, 128)[sel].reshape(-1, H, 128)
        qp = inp["q_pe"].float().numpy().reshape(B, s_q, H, 64)[sel].reshape(-1, H, 64)
        sl = inp["seqlens"][sel].numpy()
        pos = (np.repeat(sl, s_q) - s_q + np.tile(np.arange(s_q), len(sel))).clip(min=0)
        if "w_uk_t_fp8" in inp:   # FP8 projections (bmm_fp8 with per-tensor input quantization)
            q = oracle.assemble_q_fp8(qn, qp, inp["w_uk_t_fp8"].numpy(), inp["w_scale"], positions=pos)
        else:
            q = oracle.assemble_q(qn, qp, inp["_w_uk_np"], positions=pos)
        q = q.reshape(len(sel), s_q, H, 576)
        flops += acc.bmm_work(len(sel) * s_q, H, True)[0]
    else:
        q = inp["q"][sel].double().numpy()
    if "indices" in inp:   # sparse (top-k) decode over each request's list
        idx = inp["indices"][sel].numpy()
        kl = inp["topk_lens"][sel].numpy()
        out, _ = oracle.decode_sparse(q, kv_np, inp["block_table"][sel].numpy(), inp["seqlens"][sel].numpy(), idx,
                                      kl, inp["softmax_scale"], causal=inp["causal"], kv_scale=inp.get("kv_scale"))
        flops += acc.sparse_decode_work(inp["seqlens"][sel].tolist(), kl.tolist(), s_q, H, inp["causal"],
                                        indices=idx.tolist())[0]
    elif "kv_scale" in inp:   # FP8 cache: kv_np holds its E4M3 codes
        out, _ = oracle.decode_fp8(q, kv_np, inp["kv_scale"], inp["block_table"][sel].numpy(),
                                   inp["seqlens"][sel].numpy(), inp["softmax_scale"], causal=inp["causal"])
        flops += acc.decode_work(inp["seqlens"][sel].tolist(), s_q, H, inp["causal"])[0]
    else:
        out, _ = oracle.decode_absorbed(q, kv_np, inp["block_table"][sel].numpy(), inp["seqlens"][sel].numpy(),
                                        inp["softmax_scale"], causal=inp["causal"])
        flops += acc.decode_work(inp["seqlens"][sel].tolist(), s_q, H, inp["causal"])[0]
    if with_proj:
        if "w_uv_t_fp8" in inp:
            oracle.unabsorb_o_fp8(out.reshape(-1, H, 512), inp["w_uv_t_fp8"].numpy(), inp["w_scale"])
        else:
            oracle.unabsorb_o(out.reshape(-1, H, 512), inp["_w_uv_np"])
        flops += acc.bmm_work(len(sel) * s_q, H, False)[0]
    return flops


def _kv_for_oracle(inp):
    """The cache as the oracle takes it: float values, or an FP8 cache's codes."""
    if "kv_scale" in inp:
        return inp["kv_cache"].numpy()
    return inp["kv_cache"].float().numpy()


def cpu_sample(inp, w, target_s=10.0, max_reqs=None):
    """Time the oracle on a bounded sample of the workload (about target_s seconds)."""
    import numpy as np
    if "_kv_np" not in inp:
        inp["_kv_np"] = _kv_for_oracle(inp)
    if w.with_projections and "_w_uk_np" not in inp:
        inp["_w_uk_np"] = inp["w_uk"].double().numpy()
        inp["_w_uv_np"] = inp["w_uv"].double().numpy()
    B = inp["q"].shape[0]
    t0 = time.perf_counter()
    flops = oracle_sample_step(inp, inp["_kv_np"], [0], w.with_projections)
    dt = time.perf_counter() - t0
    n = max(1, min(B if max_reqs is None else max_reqs, int(target_s / max(dt, 1e-3))))
    sel = list(range(n))
    t0 = time.perf_counter()
    flops = oracle_sample_step(inp, inp["_kv_np"], sel, w.with_projections)
    dt = time.perf_counter() - t0
    return flops, dt, sel


def run_reference(args, w):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    from mla_absorbed_decode_gb300 import workloads as W
    inp = W.make_inputs(w)
    if w.chunk_tokens:   # chunked extend: the oracle on one head and the last 8 new tokens per step
        import numpy as np
        import oracle
        from mla_absorbed_decode_gb300 import accounting as acc
        T, L = w.s_q, w.seqlen
        sel_t = np.arange(T - 8, T)
        args_o = (inp["q_nope"][sel_t][:, :1].float().numpy(), inp["q_pe"][sel_t][:, :1].float().numpy(),
                  inp["w_uk"][:1].float().numpy(), inp["w_uv"][:1].float().numpy(), inp["kv_cache"].float().numpy(),
                  inp["block_table"][0].numpy(), L - (T - 8), inp["softmax_scale"], w.chunk_tokens)
        for _ in range(args.warmup):
            oracle.extend_chunked_expanded(*args_o)
        times = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            oracle.extend_chunked_expanded(*args_o)
            times.append(time.perf_counter() - t0)
        t = statistics.mean(times)
        value = acc.extend_work(L - (T - 8), 8, 1)[0] / t / 1e12
        sample = f"one head, the last 8 new tokens (context {L - (T - 8)}) per step"
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "T_new": T, "H": w.H, "seqlen": L, "chunk_tokens": w.chunk_tokens,
                       "sample": sample},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return 0
    inp["_kv_np"] = _kv_for_oracle(inp)
    if w.with_projections:
        inp["_w_uk_np"] = inp["w_uk"].double().numpy()
        inp["_w_uv_np"] = inp["w_uv"].double().numpy()
    sel = [0]
    for _ in range(args.warmup):
        oracle_sample_step(inp, inp["_kv_np"], sel, w.with_projections)
    times, flops = [], 0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        flops = oracle_sample_step(inp, inp["_kv_np"], sel, w.with_projections)
        times.append(time.perf_counter() - t0)
    t = statistics.mean(times)
    value = flops / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "s_q": w.s_q, "H": w.H,
                   "sample": f"request 0 of {w.B} per step ("
                             + ("absorb, decode, un-absorb" if w.with_projections else
                                "sparse decode" if w.topk else "decode") + " on the CPU oracle)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                         "sample": f"request 0 of {w.B} per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def max_over_ranks(values, dist, device):
    """Each value's maximum over all ranks (every rank gets the result); the values
    unchanged without a process group.  Timings are reduced this way: the job's step
    time is that of its slowest replica."""
    if dist is None:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def _graphed(torch, fn, dev):
    """Record fn's stream work once in a CUDA graph (after one uncaptured run on a side
    stream); returns a callable that replays it on the current stream."""
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream(dev).wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g.replay


def run_extend(args, w):
    """The chunked extend on the expanded path (mla_extend_chunked): T = w.s_q new tokens after
    a (seqlen - T)-token prefix of one request, the cache expanded w.chunk_tokens at a time.
    A step is one extend call; value = algorithmic TFLOP/s; the roofline object rates the
    call against the measured bf16 tensor rate (the path is tensor-bound)."""
    import torch
    import mla_absorbed_decode_gb300 as mla
    from mla_absorbed_decode_gb300 import accounting as acc, build_lib, workloads as W

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build_lib.build()
    dev = torch.device("cuda", local)
    inp = W.make_inputs(w, seed=rank)
    T, H, L, chunk = w.s_q, w.H, w.seqlen, w.chunk_tokens
    qn, qp = inp["q_nope"].to(dev), inp["q_pe"].to(dev)
    wk, wv = inp["w_uk"].to(dev), inp["w_uv"].to(dev)
    kv, row = inp["kv_cache"].to(dev), inp["block_table"][0].contiguous().to(dev)
    work = torch.empty(mla.extend_workspace_size(T, H, chunk), dtype=torch.uint8, device=dev)
    out = torch.empty((T, H, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    flush_w = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=dev)

    def flush():
        flush_w.zero_()
        flush_r.sum()

    def call(q_nope=qn, q_pe=qp):
        mla.extend_chunked(q_nope, q_pe, wk, wv, kv, row, L, inp["softmax_scale"], chunk_tokens=chunk,
                           workspace=work, out=out, lse=lse)

    for _ in range(max(args.warmup, 3)):
        flush()
        call()
    torch.cuda.synchronize()
    if mla.get_device_status() != 0:
        raise RuntimeError("device status during warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush()
            starts[i].record()
            call()
            ends[i].record()
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    if mla.get_device_status() != 0:
        raise RuntimeError("device status in the timed region")
    t_step = statistics.mean(a.elapsed_time(b) for a, b in zip(starts, ends)) / 1e3
    t_step, = max_over_ranks([t_step], dist, dev)
    flops, nbytes = acc.extend_work(L, T, H)
    n = ws
    value = n * flops / t_step / 1e12
    # end to end: q_nope and q_pe from pinned host memory, out and lse back, every step
    e2e = None
    if not args.no_e2e:
        hq, hp = inp["q_nope"].pin_memory(), inp["q_pe"].pin_memory()
        dq, dp = torch.empty_like(qn), torch.empty_like(qp)
        ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        es = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ee = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps + 2):
            flush()
            if i >= 2:
                es[i - 2].record()
            dq.copy_(hq, non_blocking=True)
            dp.copy_(hp, non_blocking=True)
            call(dq, dp)
            ho.copy_(out, non_blocking=True)
            hl.copy_(lse, non_blocking=True)
            if i >= 2:
                ee[i - 2].record()
        torch.cuda.synchronize()
        t_e2e = statistics.mean(a.elapsed_time(b) for a, b in zip(es, ee)) / 1e3
        t_e2e, = max_over_ranks([t_e2e], dist, dev)
        e2e = {"value": n * flops / t_e2e / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": hq.numel() * 2 + hp.numel() * 2,
               "d2h_bytes_per_step": ho.numel() * 2 + hl.numel() * 4, "ms_per_step": t_e2e * 1e3}
    peaks = _peaks()
    ach = flops / t_step / 1e12
    roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": ach / peaks["bf16_tflops"], "peak_source": peaks["source"], "traffic": None,
            "kernel": "mla_extend_chunked (expansion GEMM + flash attention per chunk)",
            "algorithmic_per_launch": {"bytes": nbytes, "flops": flops}, "ms_per_launch": t_step * 1e3,
            "frac_of_spec_roofline": acc.roofline_time(flops, nbytes, SPEC_FLOPS, SPEC_BW) / t_step}
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:   # the oracle on one head and 8 new tokens
        import numpy as np
        import oracle
        sel_t = np.arange(T - 8, T)
        t0 = time.perf_counter()
        oracle.extend_chunked_expanded(inp["q_nope"][sel_t][:, :1].float().numpy(),
                                       inp["q_pe"][sel_t][:, :1].float().numpy(), inp["w_uk"][:1].float().numpy(),
                                       inp["w_uv"][:1].float().numpy(), inp["kv_cache"].float().numpy(),
                                       inp["block_table"][0].numpy(), L - (T - 8), inp["softmax_scale"], chunk)
        dt = time.perf_counter() - t0
        f1, _ = acc.extend_work(L - (T - 8), 8, 1)
        cpu = {"value": f1 / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": f"one head, the last 8 new tokens (context {L - (T - 8)}), {dt:.1f} s"}
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": n, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": t_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "T_new": T, "H": H, "seqlen": L, "chunk_tokens": chunk,
                       "path": "mla_extend_chunked", "parallelism": f"replicas x{n}",
                       "l2": "flushed between timed steps (256 MiB write, then 256 MiB read; outside the step events)"},
            "pct_of_roofline": 100.0 * acc.roofline_time(flops, nbytes, SPEC_FLOPS, SPEC_BW) / t_step,
            "roofline_spec": {"peak_tflops": SPEC_FLOPS / 1e12, "peak_gbs": SPEC_BW / 1e9},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": 2 * ((L + chunk - 1) // chunk) * args.steps, "clocks": clocks.summary()}))
    if dist:
        dist.destroy_process_group()
    return 0


def run_ours(args, w):
    import torch
    import mla_absorbed_decode_gb300 as mla
    from mla_absorbed_decode_gb300 import accounting as acc, build_lib, workloads as W

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build_lib.build()
    dev = torch.device("cuda", local)
    inp = W.make_inputs(w, seed=rank)
    B, s_q, H = w.B, w.s_q, w.H
    # RoPE positions of the new tokens (row b * s_q + i sits at position seqlens[b] - s_q + i)
    pos_host = (inp["seqlens"].repeat_interleave(s_q) - s_q
                + torch.arange(s_q, dtype=torch.int32).repeat(B)).clamp_min(0).to(torch.int32)
    positions = pos_host.to(dev)
    q_nope = inp["q_nope"].to(dev) if w.with_projections else None
    q_pe = inp["q_pe"].to(dev) if w.with_projections else None
    w_uk = inp["w_uk"].to(dev) if w.with_projections else None
    w_uv = inp["w_uv"].to(dev) if w.with_projections else None
    proj_fp8 = w.with_projections and w.proj_fp8   # W_UK / W_UV as E4M3 codes: bmm_fp8
    w_uk_t = inp["w_uk_t_fp8"].to(dev) if proj_fp8 else None
    w_uv_t = inp["w_uv_t_fp8"].to(dev) if proj_fp8 else None
    fp8_ws = torch.empty(mla.bmm_fp8_workspace_size(), dtype=torch.uint8, device=dev) if proj_fp8 else None
    kv = inp["kv_cache"].to(dev)
    bt = inp["block_table"].to(dev)
    sl = inp["seqlens"].to(dev)
    sparse = w.topk > 0   # sparse (top-k) decode: each request attends to its listed tokens only
    fp8 = w.kv_fp8        # FP8 (E4M3) cache with a per-tensor scale
    kv_scale = inp.get("kv_scale")
    idx = inp["indices"].to(dev) if sparse else None
    kl = inp["topk_lens"].to(dev) if sparse else None
    parts = args.parts or mla.num_sm_parts(s_q, H)
    # the split schedule walks what the decode walks: the tokens, or the top-k lists
    step = mla.DecodeStep(B, s_q, H, kl if sparse else sl, w.causal, w.softmax_scale, parts=parts, device=dev,
                          kv_scale=kv_scale)
    q_direct = inp["q"].to(dev)
    stream = torch.cuda.current_stream()
    # Between timed steps L2 is flushed: a 256 MiB write (larger than the 126 MB L2),
    # then a 256 MiB read of another buffer that evicts those dirty lines, so that each
    # step starts with a cold and clean L2 (no write-back of the flush in the step).
    flush_w = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=dev)

    class _Flush:
        @staticmethod
        def zero_():
            flush_w.zero_()
            flush_r.sum()

    flush = _Flush()

    # Everything one pass reads or writes (the inputs, the weights and the step's buffers);
    # the timed steps cycle through several copies of it (see --inner)
    class InputSet:
        pass

    S0 = InputSet()
    S0.step, S0.kv, S0.bt, S0.sl, S0.idx, S0.kl = step, kv, bt, sl, idx, kl
    S0.q_nope, S0.q_pe, S0.positions, S0.q_direct = q_nope, q_pe, positions, q_direct
    S0.w_uk, S0.w_uv, S0.w_uk_t, S0.w_uv_t, S0.fp8_ws = w_uk, w_uv, w_uk_t, w_uv_t, fp8_ws

    def copy_of(S):
        C = InputSet()
        for name, val in vars(S).items():
            setattr(C, name, val.clone() if isinstance(val, torch.Tensor) else val)
        C.step = mla.DecodeStep(B, s_q, H, C.kl if sparse else C.sl, w.causal, w.softmax_scale, parts=parts,
                                device=dev, kv_scale=kv_scale)
        return C

    def decode_only(S=S0):
        st = S.step
        q_dec = st.q if w.with_projections else S.q_direct
        if sparse and fp8:
            mla.decode_sparse_fp8(q_dec, S.kv, kv_scale, S.bt, S.sl, S.idx, S.kl, w.softmax_scale, w.causal,
                                  st.metadata, parts, workspace=st.workspace, out=st.out, lse=st.lse)
        elif sparse:
            mla.decode_sparse(q_dec, S.kv, S.bt, S.sl, S.idx, S.kl, w.softmax_scale, w.causal, st.metadata, parts,
                              workspace=st.workspace, out=st.out, lse=st.lse)
        elif fp8:
            mla.decode_fp8(q_dec, S.kv, kv_scale, S.bt, S.sl, w.softmax_scale, w.causal, st.metadata, parts,
                           workspace=st.workspace, out=st.out, lse=st.lse)
        else:
            mla.decode(q_dec, S.kv, S.bt, S.sl, w.softmax_scale, w.causal, st.metadata, parts, workspace=st.workspace,
                       out=st.out, lse=st.lse)

    def absorb_call(qn, qp, pos_d, S=S0):
        if proj_fp8:
            mla.absorb_q_fp8(qn, S.w_uk_t, w.w_scale, S.step.q, q_pe=qp, positions=pos_d, workspace=S.fp8_ws)
        else:
            mla.absorb_q(qn, S.w_uk, S.step.q, q_pe=qp, positions=pos_d)

    def unabsorb_call(S=S0):
        out = S.step.out.view(B * s_q, H, 512)
        if proj_fp8:
            mla.unabsorb_o_fp8(out, S.w_uv_t, w.w_scale, o=S.step.o, workspace=S.fp8_ws)
        else:
            mla.unabsorb_o(out, S.w_uv, o=S.step.o)

    # with projections the split schedule runs in the absorption's launch (one more CTA: of the
    # bf16 bmm, or of the FP8 path's amax pass); otherwise on a side stream
    fused_plan = w.with_projections and B <= mla.absorb_plan_max_batch()

    def absorb_and_plan(qn, qp, pos_d, S=S0):
        if fused_plan and proj_fp8:
            st = S.step
            mla.absorb_q_fp8_plan(qn, S.w_uk_t, w.w_scale, st.q, st.seqlens, st.parts, st.metadata, q_pe=qp,
                                  positions=pos_d, workspace=S.fp8_ws)
        elif fused_plan:
            S.step.absorb_and_plan(qn, qp, S.w_uk, positions=pos_d)
        else:
            S.step.plan_beside(lambda: absorb_call(qn, qp, pos_d, S) if w.with_projections else None)

    def one_step(S=S0):
        absorb_and_plan(S.q_nope, S.q_pe, S.positions, S)
        decode_only(S)
        if w.with_projections:
            unabsorb_call(S)

    # schedule (alone or in the absorption's launch), decode + combine, the bmms
    launches_per_step = (0 if fused_plan else 1) + 2 + ((4 if proj_fp8 else 2) if w.with_projections else 0)
    # Each timed step runs `inner` passes back to back, so that the timed region lasts long
    # enough for the clock samples to see the load.  The passes cycle through `copies` input
    # sets, as many as it takes for the data touched between two uses of a set to exceed
    # 512 MiB (four times the L2): no pass finds its cache, weights or queries in L2, as
    # with the flush between steps.  ms_per_step is per pass.
    inner = args.inner if args.inner > 0 else (1 if args.eager else 256)
    set_bytes = sum(t.numel() * t.element_size() for t in vars(S0).values() if isinstance(t, torch.Tensor))
    copies = 1 if inner == 1 else min(inner, max(2, 1 + -(-(512 << 20) // set_bytes)))
    sets = [S0] + [copy_of(S0) for _ in range(copies - 1)]
    for _ in range(max(args.warmup, 3)):
        for S in sets:
            flush.zero_()
            one_step(S)
    torch.cuda.synchronize()
    status = mla.get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} during warm-up")

    def timed_step():
        for j in range(inner):
            one_step(sets[j % copies])

    def timed_decodes():
        for j in range(inner):
            decode_only(sets[j % copies])

    # the step's library calls recorded once in a CUDA graph and replayed (one host call
    # per timed step); --eager issues them one by one
    step_fn = timed_step if args.eager else _graphed(torch, timed_step, dev)
    dec_fn = timed_decodes if args.eager else _graphed(torch, timed_decodes, dev)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    d0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    d1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.zero_()
            starts[i].record()
            step_fn()
            ends[i].record()
        # the decode call (decode kernel + combine) on its own, with the step's metadata
        # and q: events between the kernels of a step would stop them from overlapping,
        # so it is timed apart from the steps, in the same way (L2 flushed before each
        # timed step, `inner` calls back to back over the input copies)
        for i in range(args.steps):
            flush.zero_()
            d0[i].record()
            dec_fn()
            d1[i].record()
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    status = mla.get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} in the timed region")

    # the projection calls on their own, timed like the decode call: `inner` calls back to back
    # from one CUDA graph, L2 flushed before each timed step (outside the timed region).  Each
    # call cycles through its own copies of what it reads and writes (activations, weights,
    # output), as many as it takes for more than 512 MiB to be touched between two uses of a
    # copy, so that no call finds its operands in L2.  Kernel time per call, launches
    # overlapping as in a step; the absorption is timed without the schedule's CTA.
    proj_b2b = None
    if w.with_projections:
        def cycled(tensors):
            nbytes = sum(t.numel() * t.element_size() for t in tensors)
            k = min(inner, max(2, 1 + -(-(512 << 20) // nbytes)))
            return [tensors] + [[t.clone() for t in tensors] for _ in range(k - 1)]

        w_uk_op = w_uk_t if proj_fp8 else w_uk
        w_uv_op = w_uv_t if proj_fp8 else w_uv
        a_sets = cycled([q_nope, q_pe, positions, w_uk_op, step.q])
        u_sets = cycled([step.out.view(B * s_q, H, 512), w_uv_op, step.o])

        def timed_absorbs():
            for j in range(inner):
                qn, qp, pos_d, wk, qo = a_sets[j % len(a_sets)]
                if proj_fp8:
                    mla.absorb_q_fp8(qn, wk, w.w_scale, qo, q_pe=qp, positions=pos_d, workspace=fp8_ws)
                else:
                    mla.absorb_q(qn, wk, qo, q_pe=qp, positions=pos_d)

        def timed_unabsorbs():
            for j in range(inner):
                ol, wv, oo = u_sets[j % len(u_sets)]
                if proj_fp8:
                    mla.unabsorb_o_fp8(ol, wv, w.w_scale, o=oo, workspace=fp8_ws)
                else:
                    mla.unabsorb_o(ol, wv, o=oo)

        proj_b2b = {}
        for name, fn in (("absorb", timed_absorbs), ("unabsorb", timed_unabsorbs)):
            fn()   # warm-up (and the graph's first capture sees every copy)
            torch.cuda.synchronize()
            g = fn if args.eager else _graphed(torch, fn, dev)
            t = []
            for i in range(args.steps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                g()
                e1.record()
                torch.cuda.synchronize()
                t.append(e0.elapsed_time(e1) * 1e3 / inner)
            proj_b2b[name] = round(statistics.mean(t), 2)
        proj_b2b["copies"] = {"absorb": len(a_sets), "unabsorb": len(u_sets)}
        del a_sets, u_sets
        status = mla.get_device_status()
        if status != 0:
            raise RuntimeError(f"device status {status} timing the projections")

    # per-call breakdown of a step, outside the timed region: eager calls with events
    # between them (so without launch overlap, and with each call's host work between its
    # events), L2 flushed before each step
    comp = {"schedule": [], "absorb": [], "decode_and_combine": [], "unabsorb": []}
    for i in range(args.steps):
        flush.zero_()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        ev[0].record()
        step.plan()
        ev[1].record()
        if w.with_projections:
            absorb_call(q_nope, q_pe, positions)
        ev[2].record()
        decode_only()
        ev[3].record()
        if w.with_projections:
            unabsorb_call()
        ev[4].record()
        torch.cuda.synchronize()
        for j, k in enumerate(comp):
            comp[k].append(ev[j].elapsed_time(ev[j + 1]) * 1e3)
    if fused_plan:   # the launch the step uses: absorption and schedule together
        comp["absorb_and_schedule"] = []
        for i in range(args.steps):
            flush.zero_()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            ev[0].record()
            absorb_and_plan(q_nope, q_pe, positions)
            ev[1].record()
            torch.cuda.synchronize()
            comp["absorb_and_schedule"].append(ev[0].elapsed_time(ev[1]) * 1e3)
    components = {k: round(statistics.mean(v), 2) for k, v in comp.items()
                  if w.with_projections or k not in ("absorb", "unabsorb")}
    step_ms = [s.elapsed_time(e) / inner for s, e in zip(starts, ends)]
    dec_ms = [a.elapsed_time(b) / inner for a, b in zip(d0, d1)]
    t_step = statistics.mean(step_ms) / 1e3
    t_dec = statistics.mean(dec_ms) / 1e3
    t_step, t_dec = max_over_ranks([t_step, t_dec], dist, dev)

    if sparse:
        dflops, dbytes = acc.sparse_decode_work(inp["seqlens"].tolist(), inp["topk_lens"].tolist(), s_q, H, w.causal,
                                                indices=inp["indices"].tolist(),
                                                kv_value_bytes=acc.FP8 if fp8 else acc.BF16)
    else:
        dflops, dbytes = acc.decode_work(inp["seqlens"].tolist(), s_q, H, w.causal,
                                         kv_value_bytes=acc.FP8 if fp8 else acc.BF16)
    spec_dec_flops = SPEC_FLOPS_FP8 if fp8 else SPEC_FLOPS   # the decode's MMAs run at the FP8 rate
    bflops = bbytes = 0
    if w.with_projections:
        for absorb in (True, False):
            f, b = acc.bmm_work(B * s_q, H, absorb, weight_bytes=acc.FP8 if proj_fp8 else acc.BF16)
            bflops += f
            bbytes += b
    step_flops, step_bytes = dflops + bflops, dbytes + bbytes
    n = ws
    value = n * step_flops / t_step / 1e12
    gbs = n * step_bytes / t_step / 1e9
    rl_time = max(dflops / spec_dec_flops + bflops / SPEC_FLOPS, step_bytes / SPEC_BW)

    # end to end through the public API with host buffers: H2D of the step's inputs,
    # the step, D2H of its result, every step
    e2e = None
    if not args.no_e2e:
        # The step's inputs are staged in two pinned host buffers: the lengths and the block
        # table (and the top-k lists) in a small one on a side stream (where a separate split
        # schedule runs on them at once), and the queries (with their RoPE positions) in a
        # large one on the main stream, where the W_UK absorption (with the schedule in its
        # launch, for bf16 projections) waits for them.  The lse goes back on a side stream
        # while the W_UV un-absorption runs, then o.  Device tensors are views of the two
        # buffers, each 256-byte aligned.
        big_specs = [("q_nope", inp["q_nope"]), ("q_pe", inp["q_pe"]), ("pos", pos_host)] if w.with_projections \
            else [("q", inp["q"])]
        small_specs = [("sl", inp["seqlens"]), ("bt", inp["block_table"])]
        if sparse:
            small_specs += [("idx", inp["indices"]), ("kl", inp["topk_lens"])]
        dv = {}

        def stage(specs):
            offs, total = {}, 0
            for name, t in specs:
                nb = t.numel() * t.element_size()
                offs[name] = (total, nb)
                total += (nb + 255) // 256 * 256
            host_pack = torch.zeros(total, dtype=torch.uint8).pin_memory()
            dev_pack = torch.empty(total, dtype=torch.uint8, device=dev)
            for name, t in specs:
                o, nb = offs[name]
                host_pack[o:o + nb].copy_(t.contiguous().view(-1).view(torch.uint8))
                dv[name] = dev_pack[o:o + nb].view(t.dtype).view(t.shape)
            return host_pack, dev_pack, total

        host_small, dev_small, n_small = stage(small_specs)
        host_big, dev_big, n_big = stage(big_specs)
        res_dev = step.o if w.with_projections else step.out
        host_out = torch.empty(res_dev.shape, dtype=res_dev.dtype).pin_memory()
        host_lse = torch.empty(step.lse.shape, dtype=torch.float32).pin_memory()
        h2d = n_small + n_big
        d2h = host_out.numel() * host_out.element_size() + host_lse.numel() * 4
        step.seqlens = dv["kl"] if sparse else dv["sl"]   # the schedule reads the staged lengths
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def e2e_step():
            cur = torch.cuda.current_stream(dev)
            s_in.wait_stream(cur)
            with torch.cuda.stream(s_in):   # lengths and table first; the schedule right behind them
                dev_small.copy_(host_small, non_blocking=True)
                if not fused_plan:
                    step.plan()
            dev_big.copy_(host_big, non_blocking=True)
            if fused_plan:   # the schedule in the absorption's launch, once both packs are in
                cur.wait_stream(s_in)
                absorb_and_plan(dv["q_nope"], dv["q_pe"], dv["pos"])
            elif w.with_projections:
                absorb_call(dv["q_nope"], dv["q_pe"], dv["pos"])
            cur.wait_stream(s_in)
            q_in = step.q if w.with_projections else dv["q"]
            if sparse and fp8:
                mla.decode_sparse_fp8(q_in, kv, kv_scale, dv["bt"], dv["sl"], dv["idx"], dv["kl"], w.softmax_scale,
                                      w.causal, step.metadata, parts, workspace=step.workspace, out=step.out,
                                      lse=step.lse)
            elif sparse:
                mla.decode_sparse(q_in, kv, dv["bt"], dv["sl"], dv["idx"], dv["kl"], w.softmax_scale, w.causal,
                                  step.metadata, parts, workspace=step.workspace, out=step.out, lse=step.lse)
            elif fp8:
                mla.decode_fp8(q_in, kv, kv_scale, dv["bt"], dv["sl"], w.softmax_scale, w.causal, step.metadata,
                               parts, workspace=step.workspace, out=step.out, lse=step.lse)
            else:
                mla.decode(q_in, kv, dv["bt"], dv["sl"], w.softmax_scale, w.causal, step.metadata, parts,
                           workspace=step.workspace, out=step.out, lse=step.lse)
            s_out.wait_stream(cur)
            with torch.cuda.stream(s_out):   # lse back while the un-absorption runs
                host_lse.copy_(step.lse, non_blocking=True)
            if w.with_projections:
                unabsorb_call()
            host_out.copy_(res_dev, non_blocking=True)
            cur.wait_stream(s_out)

        for _ in range(3):
            flush.zero_()
            e2e_step()
        torch.cuda.synchronize()
        e2e_fn = e2e_step if args.eager else _graphed(torch, e2e_step, dev)
        es = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ee = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            es[i].record()
            e2e_fn()
            ee[i].record()
        torch.cuda.synchronize()
        t_e2e = statistics.mean(a.elapsed_time(b) for a, b in zip(es, ee)) / 1e3
        t_e2e, = max_over_ranks([t_e2e], dist, dev)
        e2e = {"value": n * step_flops / t_e2e / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e * 1e3}

    peaks = _peaks()
    dec_achieved = dbytes / t_dec / 1e9
    roof_bound = "hbm" if dflops / spec_dec_flops < dbytes / SPEC_BW else "tensor"
    if roof_bound == "hbm":
        roof = {"bound": "hbm", "achieved": dec_achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": dec_achieved / peaks["hbm_gbs"]}
    else:   # FP8: the measured bf16 rate times the nominal FP8 / bf16 ratio (2)
        ach = dflops / t_dec / 1e12
        tpeak = peaks["bf16_tflops"] * (2.0 if fp8 else 1.0)
        roof = {"bound": "tensor", "achieved": ach, "peak": tpeak, "unit": "TFLOP/s", "frac": ach / tpeak}
    roof["peak_source"] = peaks["source"]
    roof["traffic"] = _traffic_per_launch(w.name)
    roof["kernel"] = ("mla_decode_sparse_fp8" if sparse and fp8 else "mla_decode_sparse" if sparse
                      else "mla_decode_fp8" if fp8 else "mla_decode") \
        + " (decode kernel + LSE combine)"
    roof["algorithmic_per_launch"] = {"bytes": dbytes, "flops": dflops}
    roof["ms_per_launch"] = t_dec * 1e3
    roof["frac_of_spec_roofline"] = acc.roofline_time(dflops, dbytes, spec_dec_flops, SPEC_BW) / t_dec

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        f, dt, sel = cpu_sample(inp, w, target_s=args.cpu_seconds)
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": f"requests {sel[0]}..{sel[-1]} of {B} ({len(sel)}), one pass of the oracle's "
                         f"absorb/decode/un-absorb, {dt:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": n, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": t_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if fp8 else "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": B, "s_q": s_q, "H": H,
                       "seqlens": (w.seqlen or f"ragged 1..{w.ragged_max}" if not w.fixed_seqlens
                                   else list(w.fixed_seqlens)),
                       "page": 64, "parts": parts, "parallelism": f"replicas x{n}",
                       **({"topk": w.topk, "path": "mla_decode_sparse"} if sparse else {}),
                       **({"projections": f"bmm_fp8: E4M3 weights (per-tensor scale {w.w_scale}), activations "
                                          "quantized per tensor on the fly (input_to_float8)"} if proj_fp8 else {}),
                       **({"kv_cache": f"e4m3 codes, per-tensor scale {kv_scale}",
                           "path": "mla_decode_sparse_fp8" if sparse else "mla_decode_fp8",
                           "mma": "kind::f8f6f4; q and P each as two E4M3 terms, fp32 accumulation"}
                          if fp8 else {}),
                       "l2": "flushed between timed steps (256 MiB write, then 256 MiB read; outside the step events)"
                             + (f"; each timed step runs {inner} passes cycling over {copies} copies of the inputs, "
                                f"weights and buffers ({(copies - 1) * set_bytes / 2**20:.0f} MiB touched between "
                                "two uses of a copy); ms_per_step is per pass" if inner > 1 else ""),
                       "decode_timing": "K further timed steps of decode calls alone inside the timed region, timed like the "
                                        "steps (ms_per_launch is per call)",
                       "launch": ("eager" if args.eager else "CUDA graph of the step's library calls")
                                 + (("; split schedule computed by one more CTA of the FP8 absorption's amax pass"
                                     if proj_fp8 else "; split schedule computed in the W_UK absorption's launch "
                                     "(one more CTA)") if fused_plan else
                                    "; split schedule on a side stream beside the W_UK absorption")},
            "hbm_gbs": gbs,
            "pct_of_roofline": 100.0 * rl_time / t_step,
            "roofline_spec": {"peak_tflops": SPEC_FLOPS / 1e12, "peak_gbs": SPEC_BW / 1e9},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "components_us": components,
            "projections_back_to_back_us": proj_b2b,
            "gpu_launches": (launches_per_step + 2) * args.steps * inner,
            "clocks": clocks.summary(),
        }
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="deepseek_v3_b64_h128_l4096")
    ap.add_argument("--parts", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0, help="override B (smaller cases for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true", help="launch the step's calls one by one instead of a CUDA graph")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--inner", type=int, default=0,
                    help="passes per timed step, cycling over input copies (default 256; 1 with --eager)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    from mla_absorbed_decode_gb300 import workloads as W
    w = W.BY_NAME[args.workload]
    if args.batch:
        import dataclasses
        w = dataclasses.replace(w, B=args.batch, name=f"{w.name}_b{args.batch}")
    if args.impl == "reference":
        return run_reference(args, w)
    if w.chunk_tokens:
        return run_extend(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
