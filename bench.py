#!/usr/bin/env python
"""Ragged paged attention benchmark (one JSON line on stdout).

A step is one full call of the library -- planner, decode attention, prefill
attention, split-KV combine -- over one batch of the workload, with inputs
resident in HBM.  The default workload is the Llama-3-8B-like decode batch:
256 sequences, q_len 1, kv_len ~ U[512, 8192], 32 q heads / 8 kv heads,
head_dim 128, page_size 16, bf16 (seeded synthetic data).  Its K/V cache
(about 4.6 GB) is far larger than L2, so no flush is needed between steps.
The default line also carries, under "workloads", the same measurements of
the mixed prefill/decode batch, the fp8 K/V windowed batch and the long
prefill (the metric's prefill TFLOP/s), each timed the same way.

  python bench.py [--steps K] [--warmup W] [--gpus N] [--workload NAME] [--impl reference]

--impl reference times the fp64 CPU oracle (the only reference this project
has) on the host cores, on a bounded sample of the same workload.
Under torchrun (N > 1) every rank runs its own replica of the batch (weak
scaling, no collective on the data path); rank 0 prints the line.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import rpa_inputs as ri  # noqa: E402

METRIC = "ragged paged attn tokens/s; decode HBM GB/s & prefill TFLOP/s vs roofline"
KERNEL_NAMES = ("planner", "decode_attention", "prefill_attention", "combine")
CSRC = "ragged_paged_attention_02_gb300/csrc/"


def kernel_sources(prob, kernel):
    """The source files of the kernel that runs `kernel` ("decode_attention" or
    "prefill_attention") on this problem: its own .cu file and the shared header."""
    eight = prob.kv_dtype in ("fp8_e4m3", "fp8_e5m2", "int8")
    if kernel == "decode_attention":
        f = "rpa_decode.cu"
    elif prob.kv_layout == "latent":
        f = "rpa_mla.cu"
    elif eight or prob.head_dim == 256:
        f = "rpa_prefill_tc8.cu"
    else:
        f = "rpa_prefill_tc.cu"
    return [CSRC + f, CSRC + "rpa_internal.cuh"]


DESCR = {
    "tiny": "3 seqs q_len {1,5,16} kv_len {17,40,64}, Hq 4 / Hkv 2, D 64, page 16, bf16",
    "decode": "256 seqs x q_len 1, kv_len~U[512,8192], Hq 32 / Hkv 8, D 128, page 16, bf16",
    "mixed": "8 prefill chunks x 512 + 56 decodes (4152 tokens), Hq 32 / Hkv 8, D 128, page 32, bf16",
    "fp8_window": "128 seqs q_len~U{1..64} kv_len~U[256,16384], Hq 16 / Hkv 8, D 256, page 16, "
                  "fp8 e4m3 K/V, softcap 50, window 4096",
    "long_prefill": "4 seqs x 8192 fresh prefill, Hq 64 / Hkv 8, D 128, page 64, bf16",
    "decode_quarter": "64 seqs x q_len 1, kv_len~U[512,8192], Hq 32 / Hkv 8, D 128, page 16, bf16",
    "fp8_window_quarter": "the first 32 seqs of fp8_window (q_len~U{1..64} kv_len~U[256,16384]), "
                          "Hq 16 / Hkv 8, D 256, page 16, fp8 e4m3 K/V, softcap 50, window 4096",
    "mla_decode": "latent attention decode: 128 seqs x q_len 1, kv_len~U[1024,8192], Hq 16 on one latent "
                  "kv head, rows 576 (V 512), page 64, bf16",
    "long_prefill_d256": "4 seqs x 8192 fresh prefill, Hq 16 / Hkv 8, D 256, page 64, bf16",
    "decode_g16": "256 seqs x q_len 1, kv_len~U[512,8192], Hq 32 / Hkv 2 (16 q heads a kv head), D 128, "
                  "page 16, bf16",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=list(ri.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--all", action="store_true",
                    help="one line per workload (tiny excluded), no CPU baseline or e2e")
    ap.add_argument("--no-side-workloads", action="store_true",
                    help="the decode line without the other workloads' measurements")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def sources_sha(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, sources):
    """dram bytes per launch from profiles/kernel_traffic.txt, if taken on the current source of
    the kernel (the hash of `sources`)."""
    path = os.path.join(ROOT, "profiles", "kernel_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = sources_sha(sources)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and \
                    parts[1] == workload and parts[2] == sha:
                return float(parts[3])
    return None


class Clocks:
    """nvidia-smi samples (200 ms) during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.proc = None
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "200"]
            if uuid:
                cmd += ["-i", uuid]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline(prob, budget_s=12.0, max_reps=8):
    """The oracle as it stands, on the host cores, over the whole batch or a sample."""
    import oracle

    T = int(prob.cu_q_lens[prob.num_seqs])
    rows_all = np.stack(np.meshgrid(np.arange(T), np.arange(prob.num_q_heads), indexing="ij"),
                        axis=-1).reshape(-1, 2).astype(np.int64)
    # size the sample from one small probe so the run stays within budget
    probe = rows_all[: max(1, min(len(rows_all), 64))]
    t0 = time.perf_counter()
    _, threads = oracle.rows(prob, probe, return_threads=True)
    per_row = (time.perf_counter() - t0) / len(probe)
    n = int(min(len(rows_all), max(prob.num_q_heads, budget_s / max(per_row, 1e-9))))
    n -= n % prob.num_q_heads or 0
    n = max(n, prob.num_q_heads)
    sample = rows_all[:n]
    done, t0 = 0, time.perf_counter()
    reps = 0
    while reps < max_reps:
        oracle.rows(prob, sample)
        done += len(sample)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    tokens = done / prob.num_q_heads
    # the same oracle on one thread, over a smaller sample (a few seconds)
    n1 = int(min(n, max(prob.num_q_heads, (budget_s / 4) / max(per_row * threads, 1e-9))))
    n1 -= n1 % prob.num_q_heads or 0
    n1 = max(n1, prob.num_q_heads)
    t1 = time.perf_counter()
    oracle.rows(prob, rows_all[:n1], nthreads=1)
    el1 = time.perf_counter() - t1
    return {"value": tokens / el, "unit": "tokens/s", "cores": int(threads), "kind": "oracle",
            "sample": f"first {n // prob.num_q_heads} of {T} query tokens (all {prob.num_q_heads} heads)"
                      f" x {reps} reps, {el:.1f} s",
            "value_1thread": n1 / prob.num_q_heads / el1,
            "sample_1thread": f"first {n1 // prob.num_q_heads} query tokens (all heads), {el1:.1f} s"}


def run_reference(args, rank):
    """--impl reference: the fp64 oracle on the host cores, same metric and workload."""
    if rank != 0:
        return
    import oracle

    prob = ri.workload(args.workload)
    T = int(prob.cu_q_lens[prob.num_seqs])
    rows_all = np.stack(np.meshgrid(np.arange(T), np.arange(prob.num_q_heads), indexing="ij"),
                        axis=-1).reshape(-1, 2).astype(np.int64)
    steps, warm = max(1, args.steps), max(0, args.warmup)
    t0 = time.perf_counter()
    _, threads = oracle.rows(prob, rows_all[: prob.num_q_heads], return_threads=True)
    per_tok = time.perf_counter() - t0
    budget = 90.0 / (steps + warm)  # whole run within ~1.5 minutes
    ntok = int(max(1, min(T, budget / max(per_tok, 1e-9))))
    sample = rows_all[: ntok * prob.num_q_heads]
    for _ in range(warm):
        oracle.rows(prob, sample)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.rows(prob, sample)
    el = time.perf_counter() - t0
    value = ntok * steps / el
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": steps,
            "warmup": warm, "ms_per_step": el / steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": f"{args.workload}: {DESCR[args.workload]}",
                       "sample_tokens_per_step": ntok},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": int(threads), "kind": "oracle",
                             "sample": f"first {ntok} of {T} query tokens (all heads) per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line, default=float), flush=True)


def rank_layout():
    """(world size, rank, local rank) as torch.distributed.run exports them; 1, 0, 0 alone."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_ranks(world):
    """Join the process group when launched as several ranks (NCCL on GPUs, gloo on the CPU).

    The ranks are independent replicas: the group carries only the barriers around the timed
    region and the max-reduction of its length, never attention data."""
    if world <= 1:
        return None
    import torch
    import torch.distributed as dist

    dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return dist


def max_over_ranks(ms, dist, device):
    """The job's elapsed time: the largest of the ranks' own (the job ends with its slowest)."""
    if dist is None:
        return float(ms)
    import torch

    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank, steps, world, ms_total):
    """Whole-job query tokens per second: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * steps * world / (ms_total / 1e3)


def upload(prob, dev):
    import torch

    q = torch.from_numpy(prob.q.view(np.int16)).view(torch.bfloat16).to(dev)
    if prob.kv_dtype == "bf16":
        kv = torch.from_numpy(prob.kv_pages.view(np.int16)).view(torch.bfloat16).to(dev)
    else:
        kv = torch.from_numpy(prob.kv_pages).to(dev)
    kvl = torch.from_numpy(prob.kv_lens).to(dev)
    pi = torch.from_numpy(prob.page_indices).to(dev)
    cu = torch.from_numpy(prob.cu_q_lens).to(dev)
    return q, kv, kvl, pi, cu


def out_for(prob, like):
    """An output tensor for prob, of like's dtype and device: [num_q_tokens, Hq, v_head_dim] (the
    width of V: head_dim, or the latent layout's value width)."""
    return like.new_empty((prob.num_q_tokens, prob.num_q_heads, prob.out_dim))


def gpu_uuid(dev):
    import torch

    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        return None


def measure(name, steps, warmup, dist, dev, world, e2e_steps=0):
    """Time `steps` calls of the library on workload `name` (after `warmup` untimed ones) with CUDA
    events on the launching stream, barrier and synchronise on both sides, max over ranks; per-kernel
    times from the library's own events; the roofline of each attention kernel and of the step."""
    import torch

    from ragged_paged_attention_02_gb300 import RPA_OPT_PLAN_EARLY, RaggedPagedAttention

    prob = ri.workload(name)
    work = ri.algorithmic_work(prob)
    q, kv, kvl, pi, cu = upload(prob, dev)
    out = out_for(prob, q)
    att = RaggedPagedAttention(**prob.cfg_dict())
    # the step's inputs are resident and written by no kernel (the end-to-end leg copies them from
    # the host): each call's planner may read them while the previous call's last kernel runs
    att.set_option(RPA_OPT_PLAN_EARLY, 1)
    stream = torch.cuda.current_stream()

    def step():
        att.forward(q, kv, kvl, pi, cu, prob.num_seqs, out=out, stream=stream)

    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize()
    if att.status() != 0:
        raise SystemExit(f"library status {att.status()} on warm-up ({name})")

    K = max(1, steps)
    clocks = Clocks(gpu_uuid(dev))
    time.sleep(0.3)

    def timed(profiled):
        # K steps between a barrier and a synchronise on both sides, CUDA events on the launching
        # stream, max over ranks; `profiled`: the library's per-kernel events on as well
        if profiled:
            att.profile_begin(K)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        return max_over_ranks(e0.elapsed_time(e1), dist, dev)

    # the step time is taken without the per-kernel events: a call's eight event records keep its
    # kernels' programmatic launches from overlapping (11-20 us a step on the short workloads); the
    # same K steps then run again with them for each kernel's own duration
    ms_total = timed(False)
    ms_total_prof = timed(True)
    clk = clocks.stop()
    kern = att.profile_read(K)  # [K, 4] ms
    ms_step = ms_total / K
    tokens = work["q_tokens"]
    value = job_throughput(tokens, K, world, ms_total)

    # per-kernel roofline: each attention kernel is charged with its own sequences' work,
    # bound by whichever of HBM bytes / tensor FLOPs takes longer at peak
    hbm, tf_burst, tf_sust, src = peaks()
    mean_k = kern.mean(axis=0)

    # the decode class is the library's (rpa_read_plan info[5]: rows of a decode tile); with fp8
    # K/V on tensor memory the prefill kernel also runs the decode-class units (info[15] bit 1):
    # charge it with both classes' work
    info = att.plan(max_items=1)[0]
    if int(info[5]) != 16:
        work = ri.algorithmic_work(prob, decode_rows=int(info[5]))
    if int(info[15]) & 2:
        d, pf = work["decode"], work["prefill"]
        work["prefill"] = {k: d[k] + pf[k] for k in pf}
        work["decode"] = {k: 0 for k in d}
    has_work = {"decode_attention": int(info[1]) > 0, "prefill_attention": int(info[2]) > 0}

    def kernel_roof(kname, ms):
        w = work["decode" if kname == "decode_attention" else "prefill"]
        t_hbm = w["bytes"] / (hbm * 1e9)
        t_tc = w["flops"] / (tf_burst * 1e12)
        if t_tc > t_hbm:
            bound, achieved, peak, unit, key = "tensor", w["flops"] / (ms * 1e-3) / 1e12, tf_burst, "TFLOP/s", "bf16_tflops"
        else:
            bound, achieved, peak, unit, key = "hbm", w["bytes"] / (ms * 1e-3) / 1e9, hbm, "GB/s", "hbm_gbs"
        r = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
             "traffic": recorded_traffic(kname, name, kernel_sources(prob, kname)), "kernel": kname,
             "peak_source": f"{src} ({key})", "kernel_ms": float(ms),
             "algorithmic": {"bytes": w["bytes"], "flops": w["flops"]}}
        if int(info[15]) & 1 and bound == "tensor" and all(has_work.values()):
            # decode and prefill ran at once on disjoint SMs: the kernel's share of the chip's tensor peak
            # (HBM bandwidth is shared, not split by SMs)
            per_sm = int(info[13] if kname == "decode_attention" else info[14])
            ctas = int(info[10] if kname == "decode_attention" else info[11])
            sms = min(int(info[12]), -(-ctas // max(per_sm, 1)))
            r["sms"] = sms
            r["frac_of_sm_share"] = achieved / (peak * sms / max(int(info[12]), 1)) if sms else None
        return r

    # the dominant kernel: the longer of the attention kernels that had work (an idle kernel's
    # span is only its launch)
    attn = [i for i, n in enumerate(KERNEL_NAMES) if n.endswith("_attention") and has_work[n]]
    kroofs = {KERNEL_NAMES[i]: kernel_roof(KERNEL_NAMES[i], mean_k[i]) for i in attn}
    dom = max(attn, key=lambda i: mean_k[i]) if attn else None
    roof = kroofs[KERNEL_NAMES[dom]] if dom is not None else None
    # the whole step against the combined roofline time max(bytes / BW, FLOPs / peak)
    t_star = max(work["bytes"] / (hbm * 1e9), work["flops"] / (tf_burst * 1e12))
    kv_gb = prob.kv_pages.nbytes / 1e9
    res = {
        "workload": f"{name}: {DESCR[name]}", "value": value, "unit": "tokens/s", "steps": K,
        "warmup": max(3, warmup), "ms_per_step": ms_step,
        "dtype": "bf16" if prob.kv_dtype == "bf16" else "f16 (8-bit K/V converted exactly)",
        "config": {"workload": f"{name}: {DESCR[name]}", "num_seqs": prob.num_seqs, "q_tokens": tokens,
                   "kv_tokens": int(prob.kv_lens[: prob.num_seqs].sum()),
                   "l2": f"no flush: inputs larger than L2 (K/V cache {kv_gb:.2f} GB)"
                   if kv_gb > 0.129 else f"K/V cache {kv_gb:.3f} GB, about L2-sized (no flush)",
                   "ranks": world, "plan_early": "inputs complete at launch (RPA_OPT_PLAN_EARLY)"},
        "step_hbm_gbs": work["bytes"] / (ms_step * 1e-3) / 1e9,
        "step_tflops": work["flops"] / (ms_step * 1e-3) / 1e12,
        "step_roofline_frac": t_star / (ms_step * 1e-3),
        "step_roofline_bound": "hbm" if work["bytes"] / (hbm * 1e9) >= work["flops"] / (tf_burst * 1e12) else "tensor",
        "kernel_rooflines": kroofs,
        "kernel_timing": "per-kernel CUDA events over a second timed pass of the same steps "
                         f"({ms_total_prof / K:.4f} ms a step with the events on)",
        # an attention kernel with no work is launched all the same; its event span is its wait for
        # SMs (the other kernel may hold them all), not work, so it is listed as idle instead
        "kernels_ms": {n: float(v) for n, v in zip(KERNEL_NAMES, mean_k) if has_work.get(n, True)},
        "idle_kernels": [n for n in KERNEL_NAMES if not has_work.get(n, True)],
        # a call launches the planner, the prefill-side kernel, the combine and (unless the
        # prefill-side kernel takes the decode units too) the decode kernel
        "roofline": roof, "gpu_launches": (3 if int(info[15]) & 2 else 4) * K, "clocks": clk,
    }

    # end to end through the public host-buffer entry point
    if e2e_steps > 0:
        hq = q.cpu().pin_memory()
        hkvl = kvl.cpu().pin_memory()
        hpi = pi.cpu().pin_memory()
        hcu = cu.cpu().pin_memory()
        hout = out_for(prob, hq).pin_memory()
        for _ in range(3):
            att.forward_host(hq, kv, hkvl, hpi, hcu, prob.num_seqs, hout, stream=stream)
        torch.cuda.synchronize()
        Ke = e2e_steps
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(Ke):
            att.forward_host(hq, kv, hkvl, hpi, hcu, prob.num_seqs, hout, stream=stream)
        a1.record(stream)
        torch.cuda.synchronize()
        ms_e = max_over_ranks(a0.elapsed_time(a1), dist, dev)
        h2d = sum(x.numel() * x.element_size() for x in (hq, hkvl, hpi, hcu))
        res["e2e"] = {"value": job_throughput(tokens, Ke, world, ms_e), "unit": "tokens/s",
                      "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(hout.numel() * hout.element_size()),
                      "ms_per_step": ms_e / Ke, "steps": Ke}
    att.close()
    del q, kv, kvl, pi, cu, out
    torch.cuda.empty_cache()
    return res, prob


# the other workloads of the default line: (name, timed steps); each K/V cache is far above L2
# except long_prefill's (134 MB, about L2-sized)
SIDE_WORKLOADS = (("mixed", 300), ("fp8_window", 300), ("long_prefill", 100), ("mla_decode", 300),
                  ("long_prefill_d256", 100), ("decode_g16", 300))


def main():
    args = parse()
    world, rank, local_rank = rank_layout()
    if args.impl == "reference":
        run_reference(args, rank)
        return
    import torch

    import __graft_entry__

    torch.cuda.set_device(local_rank)  # before the process group, so NCCL binds this rank's GPU
    dist = init_ranks(world)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if dist is not None:
        dist.barrier()

    res, prob = measure(args.workload, args.steps, args.warmup, dist, dev, world, e2e_steps=args.e2e_steps)
    # the default line also carries the other workloads of the metric (prefill TFLOP/s, the mixed
    # batch, fp8 K/V), each measured the same way; the headline value stays the decode batch's
    side = {}
    if not args.no_side_workloads and args.workload == "decode":
        for name, k in SIDE_WORKLOADS:
            r, _ = measure(name, min(k, max(1, args.steps)), args.warmup, dist, dev, world)
            side[name] = {key: r[key] for key in ("value", "unit", "ms_per_step", "steps", "dtype", "config",
                                                  "step_roofline_frac", "step_roofline_bound", "step_hbm_gbs",
                                                  "step_tflops", "kernel_rooflines", "kernels_ms", "kernel_timing",
                                                  "idle_kernels", "roofline", "clocks")}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(prob)

    if rank == 0:
        line = {
            "metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": world, "steps": res["steps"],
            "warmup": res["warmup"], "ms_per_step": res["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": res["dtype"], "data": "synthetic (seeded)",
            "config": res["config"],
            "step_hbm_gbs": res["step_hbm_gbs"], "step_tflops": res["step_tflops"],
            "step_roofline_frac": res["step_roofline_frac"],
            "kernel_rooflines": res["kernel_rooflines"], "kernels_ms": res["kernels_ms"],
            "kernel_timing": res["kernel_timing"], "idle_kernels": res["idle_kernels"],
            "roofline": res["roofline"], "cpu_baseline": cpu, "e2e": res.get("e2e"),
            "gpu_launches": res["gpu_launches"], "clocks": res["clocks"],
        }
        if side:
            line["workloads"] = side
        print(json.dumps(line, default=float), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    a0 = parse()
    if a0.all and a0.impl == "ours":
        for w in ("decode", "mixed", "fp8_window", "long_prefill", "mla_decode", "long_prefill_d256", "decode_g16"):
            sys.argv = [sys.argv[0], "--workload", w, "--steps", str(a0.steps), "--warmup",
                        str(a0.warmup), "--no-cpu-baseline", "--e2e-steps", "0", "--no-side-workloads"]
            main()
    else:
        main()
