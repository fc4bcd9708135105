"""Benchmark: the Qwen2.5-1.5B-shaped BF16 decode weight chain on GB300.

One step = one replay of the whole chain as one CUDA graph: 28 decoder blocks
(merged QKV + RMSNorm, Wo + residual, gate/up + RMSNorm + SwiGLU, Wd +
residual), the final RMSNorm, the LM head 151936 x 1536 and the argmax, batch
1, with the tuned L2-prefetch plans.  Weights are seeded synthetic bf16
(N(0, 0.02)); 3.09 GB per step is far larger than L2, so no flush is needed
between steps.

Prints one JSON line.  `value` is achieved HBM GB/s = algorithmic bytes per
step / device time per step (higher is better); `us_per_step` is the time.

  python bench.py [--steps K] [--warmup W] [--batch B] [--impl ours|reference]
Under torchrun (N > 1) every rank runs an independent replica (the chain has
no exchange step); `value` sums all ranks' bytes over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-chain µs/step and achieved HBM GB/s (fraction of GB300 roofline), 1 GPU"
WORKLOAD = ("Qwen2.5-1.5B-shaped decode weight chain: 28 blocks (H 1536, KV 256, MLP 8960, "
            "SwiGLU) + final RMSNorm + LM head 151936x1536 + argmax, one CUDA graph")
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["ws_gemv_kernel.cuh", "ws_gemv_host.cu", "ws_common.cuh", "ws_device.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--prefetch", choices=["tuned", "off"], default="tuned")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--mode", choices=["chain", "kernel", "sweep", "configs", "attention", "q4",
                                       "step-attention", "prefetch", "train", "crossover"],
                    default="chain",
                    help="chain: the decode step (the metric); kernel: gate/up alone (profiler "
                         "captures); sweep: the batch GEMV sweep, fp16 RMSNorm and the "
                         "LayerNorm block chain; configs: the fused 256x256 op beside the launch "
                         "floor, one block warm and cold, the LayerNorm chain with and without "
                         "prefetch (one JSON line each); attention: decode attention over "
                         "a key-value cache at batch 1/4/16 and 1k-32k cached slots; q4: "
                         "4-bit group-128 weights, each GEMV shape and the decode step "
                         "beside bf16; step-attention: the decode step with decode "
                         "attention over a key-value cache in every block; prefetch: gate/up "
                         "after the L2 prefetch of its own weights, of none and of a decoy; "
                         "train: forward + backward of the 72-block LayerNorm chain at batch "
                         "4 and 16 with the backward's W_(i-1) prefetch off, tuned, decoy; "
                         "crossover: the decode step at batch 1..128 on CUDA cores and tensor "
                         "cores, against its HBM and FMA floors")
    ap.add_argument("--q4-gemv", default=None,
                    help="q4 mode: one 'M,K,B' GEMV only (no decode step)")
    ap.add_argument("--attn-config", default=None,
                    help="attention mode: one 'batch,slots' configuration instead of all nine")
    ap.add_argument("--chain-mode", choices=["graph", "persistent"], default="graph",
                    help="graph: one launch per op, PDL edges, one CUDA graph; persistent: "
                         "the whole step as one cooperative kernel")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "weight_streaming_gemv_bf16_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            d = json.load(f)
        e = d.get(kernel_key)
        if e and e.get("kernel_source_hash") == kernel_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# --------------------------------------------------------------------------- inputs

def replicas_value(dt, steps, step_bytes, world, dist=None, device="cuda"):
    """Whole-job throughput of N independent replicas: the timed region of
    every rank reduced to the slowest (max over ranks), then all ranks' bytes
    over it.  Returns (slowest seconds, seconds per step, GB/s)."""
    if world > 1:
        import torch
        t = torch.tensor([dt], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dt = float(t.item())
    per_step = dt / max(steps, 1)
    return dt, per_step, world * step_bytes / per_step / 1e9


def make_host_inputs(B, seed):
    from weight_streaming_gemv_bf16_gb300 import synth
    sh = synth.QWEN2_5_1_5B
    blocks = [synth.qwen_block_weights(sh, seed, l) for l in range(sh.layers)]
    head = synth.qwen_head_weights(sh, seed)
    attn = np.stack([synth.qwen_attn(sh, B, seed, l) for l in range(sh.layers)])
    h0 = synth.qwen_hidden(sh, B, seed)
    return sh, blocks, head, attn, h0


def to_dev(bits, torch):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


# --------------------------------------------------------------------------- oracle arm

def oracle_sample(sh, blocks, head, attn, h0, budget_s, threads=None):
    """Time the oracle on the chain: whole steps (28 blocks, then the LM head
    and argmax) while they fit in the time budget, at least one block.
    Returns (GB/s, seconds, sample, threads)."""
    import oracle
    threads = threads or len(os.sched_getaffinity(0))
    att = [oracle.bf16_to_f64(a) for a in attn]
    bytes_block = sh.block_weight_bytes()
    done_bytes = 0
    t0 = time.perf_counter()
    h = h0.astype(np.float64)
    nblk = 0
    while True:
        for l in range(sh.layers):
            h = oracle.qwen_block(h, blocks[l], att[l], sh.eps, threads)["h"]
            done_bytes += bytes_block
            nblk += 1
            if time.perf_counter() - t0 > budget_s:
                break
        if time.perf_counter() - t0 > budget_s:
            break
        oracle.argmax_rows(oracle.lmhead_logits(h, oracle.bf16_to_f64(head["gamma_f"]),
                                                head["Wlm"], sh.eps, threads))
        done_bytes += sh.lm_head_bytes()
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    sample = f"{nblk} decoder blocks (+ LM heads of completed steps), batch {h0.shape[0]}, {threads} threads"
    return done_bytes / dt / 1e9, dt, sample, threads


def cpu_baseline(sh, blocks, head, attn, h0, all_s=4.0, single_s=2.0, reps=3):
    """The oracle as it stands on the host cores: the median of `reps`
    bounded samples on all cores (OpenMP over output rows) and the median of
    `reps` on one thread."""
    runs = [oracle_sample(sh, blocks, head, attn, h0, all_s) for _ in range(reps)]
    one = [oracle_sample(sh, blocks, head, attn, h0, single_s, threads=1) for _ in range(reps)]
    med = sorted(runs, key=lambda r: r[0])[reps // 2]
    med1 = sorted(one, key=lambda r: r[0])[reps // 2]
    return {"value": round(med[0], 3), "unit": "GB/s", "cores": med[3], "kind": "oracle",
            "sample": f"median of {reps} samples of about {all_s:g} s each: " + med[2],
            "seconds": round(sum(r[1] for r in runs) + sum(r[1] for r in one), 1),
            "all_cores_runs_gbs": [round(r[0], 3) for r in runs],
            "single_thread": {"value": round(med1[0], 4), "unit": "GB/s", "cores": 1,
                              "sample": f"median of {reps} samples of about {single_s:g} s each: "
                                        + med1[2],
                              "runs_gbs": [round(r[0], 4) for r in one]}}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    sh, blocks, head, attn, h0 = make_host_inputs(args.batch, args.seed)
    import oracle
    oracle.build()
    threads = len(os.sched_getaffinity(0))
    att = [oracle.bf16_to_f64(a) for a in attn]
    # one reference "step" = one decoder block of the chain (a bounded sample)
    h = h0.astype(np.float64)
    for w in range(args.warmup):
        h = oracle.qwen_block(h, blocks[w % sh.layers], att[w % sh.layers], sh.eps, threads)["h"]
    t0 = time.perf_counter()
    for k in range(args.steps):
        h = oracle.qwen_block(h, blocks[k % sh.layers], att[k % sh.layers], sh.eps, threads)["h"]
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    gbs = sh.block_weight_bytes() / dt / 1e9
    us_chain = sh.chain_weight_bytes() / (gbs * 1e9) * 1e6
    sample = f"one decoder block per step (93.6 MB of bf16 weights), batch {args.batch}"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(us_chain / 1e3, 3), "us_per_step": round(us_chain, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "batch": args.batch,
                                       "reference": "CPU oracle (plain C, double accumulation)",
                                       "sample": "each step is one decoder block of the chain "
                                                 "(93.6 MB of weights), blocks taken in turn; "
                                                 "us_per_step extrapolates the block rate to the "
                                                 "whole chain's bytes"},
        "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- our arm

def read_roofline(torch, wb, nbytes=4 << 30, reps=5):
    buf = torch.empty(nbytes // 4, dtype=torch.int32, device="cuda")
    buf.fill_(1)
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    sink = torch.zeros(nsm * 4, dtype=torch.int32, device="cuda")
    best = 0.0
    for blocks in (nsm * 2, nsm * 4):
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            wb.read_probe(buf, nbytes, blocks, sink)
            e1.record()
            e1.synchronize()
            best = max(best, nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del buf
    return best


def time_dominant_kernel(torch, wb, dblocks, sh, B, reps=20):
    """The gate/up GEMV (RMSNorm prologue + SwiGLU epilogue, 2 x 8960 x 1536)
    over every block's weights in turn (inputs larger than L2), launched back
    to back with programmatic dependent launch as the chain launches its ops
    (one CUDA graph of L launches), timed with CUDA events around the graph
    on the launching stream: the average launch duration is the graph's time
    over L.  Also returned: the average of launches timed one by one (each
    with its own launch latency, ramp-up and tail, nothing overlapped)."""
    x = torch.randn((B, sh.hidden), device="cuda")
    s = torch.empty((B, sh.inter), dtype=torch.bfloat16, device="cuda")
    nbytes = 2 * sh.inter * sh.hidden * 2 + sh.hidden * 2  # Wg + Wu + gamma2
    base = wb.get_tuning()
    t = wb.Tuning()
    for f, _ in wb.Tuning._fields_:
        setattr(t, f, getattr(base, f))
    t.launch_pdl = 1
    wb.set_tuning(t)
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for w in dblocks:  # plans, workspaces and kernel attributes before capture
                wb.swiglu_gemv(x, w["gamma2"], w["Wg"], w["Wu"], s, sh.eps, stream=side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            st = torch.cuda.current_stream()
            for w in dblocks:
                wb.swiglu_gemv(x, w["gamma2"], w["Wg"], w["Wu"], s, sh.eps, stream=st)
    finally:
        wb.set_tuning(base)
    st = torch.cuda.current_stream()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        g.replay()
    e1.record(st)
    torch.cuda.synchronize()
    dur = e0.elapsed_time(e1) * 1e-3 / (reps * len(dblocks))
    # one by one, for reference
    ts = []
    for r in range(2):
        for w in dblocks:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            wb.swiglu_gemv(x, w["gamma2"], w["Wg"], w["Wu"], s, sh.eps, stream=st)
            b.record(st)
            if r > 0:
                ts.append((a, b))
    torch.cuda.synchronize()
    alone = float(np.mean([a.elapsed_time(b) for a, b in ts])) * 1e-3
    return nbytes, dur, reps * len(dblocks), alone


def in_chain_op_us(torch, wc, dblocks, dhead, dattn, dh0, sh, reps=3):
    """Per-op time inside the chain from globaltimer stamps every CTA writes
    (entry, dependency released, activations staged, done): an op's time runs
    from the previous op's last CTA end to its own last CTA end, averaged
    over the blocks and over `reps` replays.  Returns {kind: us}."""
    ch = wc.qwen_chain(dblocks, dhead, dattn, dh0, eps=sh.eps, use_pdl=True, prefetch=0)
    g, nops = ch.chain.grid(), ch.chain.n_ops
    buf = torch.zeros((g, nops, 44), dtype=torch.int64, device="cuda")
    ch.chain.debug_stamps(buf)
    ch.chain.capture()
    kinds = ["qkv", "wo", "gate_up", "wd"] * sh.layers + ["lm_head"]
    tot = {k: 0.0 for k in set(kinds)}
    cnt = {k: 0 for k in set(kinds)}
    for _ in range(2):
        ch.run()
    for _ in range(reps):
        buf.zero_()
        ch.run()
        torch.cuda.synchronize()
        raw = buf.cpu().numpy()[:, :, :4].astype(np.float64)
        valid = raw[:, :, 0] > 0
        prev_end = raw[:, 0, 0][valid[:, 0]].min()
        for f in range(nops):
            end = raw[valid[:, f], f, 3].max()
            tot[kinds[f]] += (end - prev_end) / 1e3
            cnt[kinds[f]] += 1
            prev_end = end
    ch.chain.close()
    return {k: tot[k] / cnt[k] for k in tot}


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)

    import __graft_entry__
    __graft_entry__.build()
    from weight_streaming_gemv_bf16_gb300 import binding as wb
    from weight_streaming_gemv_bf16_gb300 import chain as wc

    B = args.batch
    sh, blocks, head, attn, h0 = make_host_inputs(B, args.seed + rank)
    dblocks = [{k: to_dev(v, torch) for k, v in b.items()} for b in blocks]
    dhead = {k: to_dev(v, torch) for k, v in head.items()}
    dattn = to_dev(attn, torch)
    dh0 = torch.from_numpy(h0).cuda()
    step_bytes = sh.chain_weight_bytes() + sh.chain_gamma_bytes()

    read_gbs = read_roofline(torch, wb)

    persistent = args.chain_mode == "persistent"

    def make_chain(prefetch, decoy=False):
        return wc.qwen_chain(dblocks, dhead, dattn, dh0, eps=sh.eps, use_pdl=True,
                             prefetch=prefetch, decoy=decoy, tune_pairs=30, min_gain=0.01,
                             persistent=persistent)

    t_tune = time.perf_counter()
    main = make_chain(1 if args.prefetch == "tuned" else 0)
    main.chain.tune()
    t_tune = time.perf_counter() - t_tune
    main.chain.capture()
    plans = main.chain.plans()
    n_prefetch_launches = 0
    op_reads = [3, 1, 2, 1] * sh.layers + [1]
    for i, (pl, lo, mean) in enumerate(plans):
        if pl[0] != 0 and i >= 1:
            n_prefetch_launches += op_reads[i]

    def timed(ch, steps, warmup):
        st = torch.cuda.current_stream()
        for _ in range(warmup):
            ch.run(st)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.nvtx.range_push("timed")
        e0.record(st)
        for _ in range(steps):
            ch.run(st)
        e1.record(st)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        return e0.elapsed_time(e1) * 1e-3

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    dt = timed(main, args.steps, args.warmup)
    clk = clocks.stop()
    dt, per_step, value = replicas_value(dt, args.steps, step_bytes, world, dist)

    # controls: no prefetch, and a decoy of the same traffic (when a plan was kept)
    variants = {}
    ksteps = max(10, min(args.steps, 500))
    if rank == 0 and not main.chain.persistent:
        off = make_chain(0)
        off.chain.capture()
        variants["no_prefetch_us"] = round(timed(off, ksteps, 5) / ksteps * 1e6, 2)
        if any(p[0][0] != 0 for p in plans):
            dec = make_chain(1, decoy=True)
            dec.chain.tune()
            dec.chain.capture()
            variants["decoy_us"] = round(timed(dec, ksteps, 5) / ksteps * 1e6, 2)
        variants["tuned_us"] = round(per_step * 1e6, 2)

    hbm, hbm_kind = peaks()
    nbytes, kdur, nlaunch, kalone = time_dominant_kernel(torch, wb, dblocks, sh, B)
    op_us = in_chain_op_us(torch, wc, dblocks, dhead, dattn, dh0, sh)
    achieved = nbytes / kdur / 1e9
    dom_key = "k_stream_gemv<1,2,2,F_RMS_SWIGLU> gate/up+SwiGLU 8960x1536 B=1"
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": ncu_traffic(dom_key),
                "kernel": dom_key, "algorithmic_bytes_per_launch": nbytes,
                "avg_launch_us": round(kdur * 1e6, 3), "launches_timed": nlaunch,
                "launches": "back to back with programmatic dependent launch, one CUDA graph",
                "alone_launch_us": round(kalone * 1e6, 3),
                "in_chain_launch_us": round(op_us["gate_up"], 3),
                "in_chain_frac": round(nbytes / (op_us["gate_up"] * 1e-6) / 1e9 / hbm, 4),
                "in_chain_op_us": {k: round(v, 3) for k, v in sorted(op_us.items())},
                "in_chain_note": "per-op globaltimer stamps of the chain itself (previous "
                                 "op's last CTA end to this op's), averaged over blocks",
                "peak_kind": f"{hbm_kind} (copy, MEASURED_PEAKS hbm_gbs)" if hbm_kind == "measured"
                else "fallback"}

    e2e = None
    if not args.no_e2e:
        import torch as _t
        h_host = _t.from_numpy(h0).pin_memory()
        a_host = _t.from_numpy(np.ascontiguousarray(attn).view(np.int16)).pin_memory()
        out = _t.empty((B,), dtype=_t.int32).pin_memory()
        n_e2e = max(5, min(args.steps, 300))
        for _ in range(3):
            main.chain.step_host(h_host, a_host, out)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            main.chain.step_host(h_host, a_host, out)
        e_dt = (time.perf_counter() - t0) / n_e2e
        e2e = {"value": round(world * step_bytes / e_dt / 1e9, 1), "unit": "GB/s",
               "us_per_step": round(e_dt * 1e6, 2),
               "h2d_bytes_per_step": int(h0.nbytes + attn.nbytes), "d2h_bytes_per_step": 4 * B,
               "steps": n_e2e}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        cpu = cpu_baseline(sh, blocks, head, attn, h0)

    if rank != 0:
        return 0
    n_ops = main.chain.n_ops
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 4),
        "us_per_step": round(per_step * 1e6, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,0.02) bf16 weights)",
        "config": {"workload": WORKLOAD, "batch": B, "layers": sh.layers,
                   "bytes_per_step": step_bytes, "prefetch": args.prefetch, "pdl": True,
                   "chain_mode": "persistent" if main.chain.persistent else "graph",
                   "l2": "inputs larger than L2 (3.09 GB of weights per step, no flush)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "frac_of_copy_peak": round(value / world / hbm, 4),
        "read_roofline_gbs": round(read_gbs, 1),
        "frac_of_read_roofline": round(value / world / read_gbs, 4),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(args.steps * (1 if main.chain.persistent else n_ops + n_prefetch_launches)),
        "clocks": clk,
        "prefetch_plans": {"kept": sum(1 for p in plans if p[0][0] != 0), "ops": len(plans),
                           "tune_seconds": round(t_tune, 2),
                           "best_lower_ci": round(max([p[1] for p in plans] or [0.0]), 4)},
        "variants": variants,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_kernel_only(args):
    """The dominant kernel alone (gate/up GEMV + RMSNorm + SwiGLU, 2 x 8960 x
    1536, batch B) over 4 rotating weight copies (220 MB, larger than L2): the
    small case for profiler captures."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from weight_streaming_gemv_bf16_gb300 import binding as wb
    from weight_streaming_gemv_bf16_gb300 import synth
    sh = synth.QWEN2_5_1_5B
    B = args.batch
    copies = [{k: to_dev(synth.normal_bf16((sh.inter, sh.hidden), 0.02, args.seed, f"k{i}/{k}"), torch)
               for k in ("Wg", "Wu")} for i in range(4)]
    g = to_dev(synth.uniform_bf16((sh.hidden,), 0.5, 1.5, args.seed, "k/g"), torch)
    x = torch.from_numpy(synth.normal_f32((B, sh.hidden), 1.0, args.seed, "k/x")).cuda()
    s = torch.empty((B, sh.inter), dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.current_stream()
    for i in range(args.warmup):
        c = copies[i % 4]
        wb.swiglu_gemv(x, g, c["Wg"], c["Wu"], s, sh.eps, stream=st)
    torch.cuda.synchronize()
    ev = []
    for i in range(args.steps):
        c = copies[i % 4]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        wb.swiglu_gemv(x, g, c["Wg"], c["Wu"], s, sh.eps, stream=st)
        e1.record(st)
        ev.append((e0, e1))
    torch.cuda.synchronize()
    dur = float(np.mean([a.elapsed_time(b) for a, b in ev])) * 1e-3
    nbytes = 2 * sh.inter * sh.hidden * 2 + sh.hidden * 2
    print(json.dumps({"mode": "kernel", "kernel": "gate/up GEMV + RMSNorm + SwiGLU 8960x1536",
                      "batch": B, "launches": args.steps, "avg_us": round(dur * 1e6, 3),
                      "gbs": round(nbytes / dur / 1e9, 1)}), flush=True)
    return 0


def run_prefetch_probe(args):
    """The L2-prefetch path on one op: the gate/up GEMV (2 x 8960 x 1536,
    batch B) over 4 rotating weight copies (220 MB, larger than L2, so every
    launch starts cold), each launch preceded on the same stream by one of:
    nothing; the pages' prefetch kernel over exactly the weights the launch
    reads (per-line `prefetch.global.L2` every 128 bytes, or bulk 16 KiB
    chunks); or a decoy that prefetches the same number of bytes of buffers
    no launch reads ("Making small PyTorch ops faster on a laptop GPU", "Prefetching the
    next layer while this one runs" and its control).  Prints the gate/up
    launch time per variant; an ncu capture of the same command reads the L2
    hit rate and DRAM bytes of each gate/up launch."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from weight_streaming_gemv_bf16_gb300 import binding as wb
    from weight_streaming_gemv_bf16_gb300 import synth
    sh = synth.QWEN2_5_1_5B
    B = args.batch
    copies = [{k: to_dev(synth.normal_bf16((sh.inter, sh.hidden), 0.02, args.seed, f"k{i}/{k}"), torch)
               for k in ("Wg", "Wu")} for i in range(4)]
    # the decoy's target: the same bytes in buffers no GEMV ever reads
    decoy = {k: torch.empty((sh.inter, sh.hidden), dtype=torch.bfloat16, device="cuda")
             for k in ("Wg", "Wu")}
    g = to_dev(synth.uniform_bf16((sh.hidden,), 0.5, 1.5, args.seed, "k/g"), torch)
    x = torch.from_numpy(synth.normal_f32((B, sh.hidden), 1.0, args.seed, "k/x")).cuda()
    s = torch.empty((B, sh.inter), dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.current_stream()
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    plans = {"none": None,
             "line": wb.PrefetchPlan(2 * nsm, 256, 128, 1),
             "bulk": wb.PrefetchPlan(nsm, 256, 16384, 3),
             "decoy": wb.PrefetchPlan(2 * nsm, 256, 128, 1)}
    mat_bytes = sh.inter * sh.hidden * 2
    out = {}
    ref = None
    for name, plan in plans.items():
        ev = []
        for i in range(args.warmup + args.steps):
            c = copies[i % 4]
            if plan is not None:
                tgt = decoy if name == "decoy" else c
                for k in ("Wg", "Wu"):
                    wb.l2_prefetch(tgt[k], mat_bytes, plan, stream=st)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            wb.swiglu_gemv(x, g, c["Wg"], c["Wu"], s, sh.eps, stream=st)
            e1.record(st)
            if i >= args.warmup:
                ev.append((e0, e1))
        torch.cuda.synchronize()
        if ref is None:
            ref = s.clone()
        assert torch.equal(s, ref), "a prefetch changed the output"
        out[name] = round(float(np.mean([a.elapsed_time(b) for a, b in ev])) * 1e3, 3)
    nbytes = 2 * mat_bytes + sh.hidden * 2
    print(json.dumps({"mode": "prefetch", "kernel": "gate/up GEMV + RMSNorm + SwiGLU 8960x1536",
                      "batch": B, "launches_per_variant": args.steps, "gate_up_us": out,
                      "bytes_per_launch": nbytes,
                      "prefetch_plans": {k: (None if v is None else [v.blocks, v.threads,
                                                                     v.stride_bytes, v.mode])
                                         for k, v in plans.items()},
                      "note": "prefetch kernel and GEMV serialised on one stream; the time is "
                              "the GEMV launch alone"}), flush=True)
    return 0


def run_train(args):
    """Small-batch training of the 72-block LayerNorm(768) -> Linear(768, 768)
    -> GELU chain ("Making small PyTorch ops faster on a laptop GPU", "It works
    in training too"): one step = the training forward (one CUDA graph) and
    the backward with the mean-square loss of the output (one CUDA graph),
    at batch 4 and 16, with the backward's L2 prefetch of W_(i-1) off, tuned
    (measured plan, kept only if its 95% CI clears +1%) and as a decoy aimed
    at the wrong block.  Gradients are checked bit-identical across the
    variants.  Prints one JSON line per batch size."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from weight_streaming_gemv_bf16_gb300 import binding as wb
    from weight_streaming_gemv_bf16_gb300 import chain as wc
    from weight_streaming_gemv_bf16_gb300 import synth
    sh = synth.MlpShape()
    w, L = sh.width, sh.blocks
    st = torch.cuda.current_stream()
    for B in ([args.batch] if args.batch != 1 else [4, 16]):
        blocks = [{k: to_dev(v, torch) for k, v in synth.mlp_block_weights(sh, args.seed, i).items()}
                  for i in range(L)]
        x = to_dev(synth.mlp_input(sh, B, args.seed), torch)
        fwd = wc.mlp_chain(blocks, x, eps=sh.eps, training=True)
        fwd.chain.capture()
        fwd.run()
        runs = {"none": wc.mlp_backward(blocks, fwd)}
        if args.prefetch != "off":  # --prefetch off: the no-prefetch backward alone
            runs["tuned"] = wc.mlp_backward(blocks, fwd, prefetch=1, tune_pairs=30)
            runs["decoy"] = wc.mlp_backward(blocks, fwd, prefetch=2, decoy=True,
                                            fixed_plan=wb.PrefetchPlan(16, 256, 16384, 3))
        t0 = time.perf_counter()
        if "tuned" in runs:
            runs["tuned"].bwd.tune()
        t_tune = time.perf_counter() - t0
        (mode, nb, nt, stride), lo, mean = (runs["tuned"].bwd.plan() if "tuned" in runs
                                            else ((0, 0, 0, 0), float("nan"), float("nan")))
        for r in runs.values():
            r.bwd.capture()

        def timed(fn, n):
            for _ in range(5):
                fn()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            for _ in range(n):
                fn()
            b.record(st)
            b.synchronize()
            return a.elapsed_time(b) / n * 1e3

        n = max(20, min(args.steps, 400))
        res = {"fwd_us": [], **{k: [] for k in runs}}
        ref = None
        for rnd in range(5):  # interleaved rounds
            res["fwd_us"].append(timed(lambda: fwd.run(st), n))
            for k, r in runs.items():
                res[k].append(timed(lambda r=r: (fwd.run(st), r.run(st)), n))
                g = [r.dx.cpu()] + [t.cpu() for gg in r.grads for t in gg.values()]
                if ref is None:
                    ref = g
                assert all(torch.equal(a_, b_) for a_, b_ in zip(g, ref)), f"{k}: gradients differ"
        med = {k: float(np.median(v)) for k, v in res.items()}
        wbytes = L * (w * w + 3 * w) * 2
        step_bytes = 2 * wbytes + L * w * w * 2  # W read forward and backward, dW written
        print(json.dumps({
            "mode": "train", "workload": f"72 x [LayerNorm({w}) -> Linear({w},{w}) -> GELU], "
                                         "mean-square loss, bf16",
            "batch": B, "steps_per_round": n, "rounds": 5,
            "forward_us": round(med["fwd_us"], 2),
            "step_us": {k: round(med[k], 2) for k in runs},
            "backward_us": {k: round(med[k] - med["fwd_us"], 2) for k in runs},
            "prefetch_gain_tuned": (round(1 - med["tuned"] / med["none"], 4) if "tuned" in med
                                    else None),
            "prefetch_gain_decoy": (round(1 - med["decoy"] / med["none"], 4) if "decoy" in med
                                    else None),
            "tuned_plan": {"mode": mode, "blocks": nb, "threads": nt, "stride": stride,
                           "gain_lower_95": round(lo, 4), "gain_mean": round(mean, 4),
                           "tune_seconds": round(t_tune, 2)},
            "bytes_per_step": step_bytes,
            "gbs_none": round(step_bytes / (med["none"] * 1e-6) / 1e9, 1),
            "launches_per_step": L + (L + 2),
            "gradients_bit_identical": True}), flush=True)
    return 0


def run_crossover(args):
    """Batching: when does the decode step stop being memory-bound ("One
    Token, Kernel by Kernel", "Batching: when does decode stop being
    memory-bound?").  The full Qwen2.5-1.5B-shaped chain (seeded N(0, 0.02)
    weights drawn on the device) at B = 1 .. 128, on CUDA cores (the default
    kernels) and with the optional warp-level tensor-core kernel; batches
    above 16 run every op once per 16-row tile.  Per batch: us per step, the
    weight bytes read once per step over that time (GB/s), the FLOP rate
    (2 x weights x B per step), and the step's floors: HBM (weights once at
    the measured copy peak) and, for CUDA cores, the FP32 FMA issue rate."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from weight_streaming_gemv_bf16_gb300 import binding as wb
    from weight_streaming_gemv_bf16_gb300 import chain as wc
    from weight_streaming_gemv_bf16_gb300 import synth
    sh = synth.QWEN2_5_1_5B
    H, KV, I, V, L = sh.hidden, sh.kv_dim, sh.inter, sh.vocab, sh.layers
    g = torch.Generator(device="cuda")
    g.manual_seed(args.seed)

    def rw(*shape):
        return (torch.randn(shape, device="cuda", generator=g) * 0.02).to(torch.bfloat16)

    def gam():
        return (torch.rand(H, device="cuda", generator=g) + 0.5).to(torch.bfloat16)
    blocks = [dict(gamma1=gam(), Wq=rw(H, H), Wk=rw(KV, H), Wv=rw(KV, H), Wo=rw(H, H),
                   gamma2=gam(), Wg=rw(I, H), Wu=rw(I, H), Wd=rw(H, I)) for _ in range(L)]
    head = dict(gamma_f=gam(), Wlm=rw(V, H))
    wbytes = sh.chain_weight_bytes()
    weights = wbytes / 2
    hbm, _ = peaks()
    fma_rate = 36.3e12  # measured mixed bf16 FMA rate of this part (see the design notes)
    st = torch.cuda.current_stream()
    base = wb.get_tuning()
    rows = []
    for B in [1, 2, 4, 8, 16, 32, 64, 128]:
        attn = (torch.randn((L, B, H), device="cuda", generator=g)).to(torch.bfloat16)
        h0 = torch.randn((B, H), device="cuda", generator=g)
        for mma in (0, 1):
            t = wb.Tuning()
            for f, _ in wb.Tuning._fields_:
                setattr(t, f, getattr(base, f))
            t.mma = mma
            wb.set_tuning(t)
            try:
                ch = wc.qwen_chain(blocks, head, attn, h0, eps=sh.eps)
                ch.chain.capture()
            finally:
                wb.set_tuning(base)
            n = max(5, min(args.steps, int(0.5e6 / (650 * max(1, B / 4)))))
            times = []
            for _ in range(3):
                for _ in range(3):
                    ch.run(st)
                torch.cuda.synchronize()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(st)
                for _ in range(n):
                    ch.run(st)
                b.record(st)
                b.synchronize()
                times.append(a.elapsed_time(b) / n * 1e3)
            us = float(np.median(times))
            row = {"B": B, "kernel": "tensor-core (mma.sync)" if mma else "CUDA cores",
                   "us_per_step": round(us, 1), "weight_gbs": round(wbytes / (us * 1e-6) / 1e9, 1),
                   "tflops": round(2 * weights * B / (us * 1e-6) / 1e12, 2),
                   "hbm_floor_us": round(wbytes / (hbm * 1e9) * 1e6, 1),
                   "launches_per_step": ch.chain.n_ops}
            if not mma:
                row["fma_floor_us"] = round(weights * B / fma_rate * 1e6, 1)
            rows.append(row)
            print(json.dumps(dict(mode="crossover", **row)), flush=True)
            ch.chain.close()
    return 0


def run_sweep(args):
    """The standalone workloads of the batch sweep and of the LayerNorm block
    chain, one JSON line: each GEMV shape of the decode step at batch 1..16
    (launched back to back with programmatic dependent launch over rotating
    weight copies larger than L2, one CUDA graph, CUDA events around it), the
    fp16 RMSNorm on [R, 896] rows, and the 72-block LayerNorm + GEMV + bias +
    GELU chain (768 x 768) at batch 4 and 16."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from weight_streaming_gemv_bf16_gb300 import binding as wb
    from weight_streaming_gemv_bf16_gb300 import chain as wc
    from weight_streaming_gemv_bf16_gb300 import synth
    torch.cuda.set_device(0)
    gen = torch.Generator(device="cuda").manual_seed(args.seed)
    st = torch.cuda.current_stream()

    def graph_time(fn, n_inner, reps=10):
        side = torch.cuda.Stream()
        side.wait_stream(st)
        with torch.cuda.stream(side):
            fn(side)  # plans, workspaces and kernel attributes before capture
        st.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn(torch.cuda.current_stream())
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(reps):
            g.replay()
        e1.record(st)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e-3 / (reps * n_inner)

    base = wb.get_tuning()
    t = wb.Tuning()
    for f, _ in wb.Tuning._fields_:
        setattr(t, f, getattr(base, f))
    t.launch_pdl = 1
    wb.set_tuning(t)
    gemv = []
    try:
        for M, K in [(8960, 1536), (1536, 8960), (256, 1536), (151936, 1536)]:
            ncopy = max(2, -(-(256 << 20) // (M * K * 2)))
            Ws = [(torch.randn((M, K), device="cuda", generator=gen) * 0.02).to(torch.bfloat16)
                  for _ in range(ncopy)]
            for B in (1, 2, 4, 8, 16):
                x = torch.randn((B, K), device="cuda", generator=gen).to(torch.bfloat16)
                y = torch.empty((B, M), device="cuda")
                nws = wb.workspace_bytes(wb.OP_GEMV, M, K, B)
                ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")

                def fn(s, Ws=Ws, x=x, y=y, ws=ws):
                    for W in Ws:
                        wb.gemv_bf16(W, x, y, workspace=ws, stream=s)
                dur = graph_time(fn, len(Ws))
                nbytes = M * K * 2 + B * K * 2 + B * M * 4
                gemv.append({"M": M, "K": K, "B": B, "us": round(dur * 1e6, 2),
                             "gbs": round(nbytes / dur / 1e9, 1)})
            del Ws
    finally:
        wb.set_tuning(base)
    rms = []
    N = 896
    for R in (1, 128, 4096):
        xs = [torch.randn((R, N), device="cuda", generator=gen).to(torch.float16) for _ in range(8)]
        gmm = (torch.rand((N,), device="cuda", generator=gen) + 0.5).to(torch.float16)
        ys = [torch.empty_like(v) for v in xs]

        def fn(s, xs=xs, ys=ys, gmm=gmm):
            for v, o in zip(xs, ys):
                wb.rmsnorm(v, gmm, o, 1e-6, stream=s)
        dur = graph_time(fn, len(xs))
        rms.append({"R": R, "N": N, "us": round(dur * 1e6, 2),
                    "gbs": round(2 * R * N * 2 / dur / 1e9, 1)})
    mlp = []
    sh = synth.MlpShape()
    hb = [synth.mlp_block_weights(sh, args.seed, l) for l in range(sh.blocks)]
    db = [{k: to_dev(v, torch) for k, v in b.items()} for b in hb]
    for B in (4, 16):
        x_in = to_dev(synth.mlp_input(sh, B, args.seed), torch)
        ch = wc.mlp_chain(db, x_in, eps=sh.eps)
        ch.chain.capture()
        for _ in range(5):
            ch.run(st)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 200
        e0.record(st)
        for _ in range(reps):
            ch.run(st)
        e1.record(st)
        torch.cuda.synchronize()
        dur = e0.elapsed_time(e1) * 1e-3 / reps
        nbytes = sh.blocks * sh.block_bytes()
        mlp.append({"B": B, "blocks": sh.blocks, "us_per_step": round(dur * 1e6, 2),
                    "gbs": round(nbytes / dur / 1e9, 1)})
        ch.chain.close()
    print(json.dumps({"mode": "sweep", "gemv_back_to_back": gemv, "rmsnorm_fp16": rms,
                      "mlp_chain": mlp}), flush=True)
    return 0


def run_configs(args):
    """The small configurations, one JSON line:
    - the fused RMSNorm + GEMV 256 x 256 at batch 1 (latency-bound) beside the
      on-box launch floor (an empty kernel, and one with a DRAM round trip),
      each as back-to-back launches in one CUDA graph;
    - one Qwen2.5-1.5B-shaped block at batch 1 (93.6 MB): L2-warm (the same
      block replayed) and cold (six blocks with their own weights, 562 MB,
      replayed in turn);
    - the 72-block LayerNorm chain at batch 4 and 16: the measured prefetch
      plans against none (with the tuner's kept plans and best lower CI),
      warm (one chain, 85 MB) and cold (six chains in turn)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from weight_streaming_gemv_bf16_gb300 import binding as wb
    from weight_streaming_gemv_bf16_gb300 import chain as wc
    from weight_streaming_gemv_bf16_gb300 import synth
    torch.cuda.set_device(0)
    st = torch.cuda.current_stream()

    def events(fn, reps):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(reps):
            fn()
        e1.record(st)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e-3 / reps

    def graph_of(fn, n):
        side = torch.cuda.Stream()
        side.wait_stream(st)
        with torch.cuda.stream(side):
            fn(side)
        st.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(n):
                fn(torch.cuda.current_stream())
        return g

    out = {"mode": "configs"}
    # config 1 and the launch floor
    n = 100
    x = to_dev(synth.normal_bf16((1, 256), 1.0, args.seed, "c1/x"), torch)
    gm = to_dev(synth.uniform_bf16((256,), 0.5, 1.5, args.seed, "c1/g"), torch)
    W = to_dev(synth.normal_bf16((256, 256), 0.02, args.seed, "c1/W"), torch)
    y = torch.empty((1, 256), device="cuda")
    ws = torch.empty(max(wb.workspace_bytes(wb.OP_GEMV, 256, 256, 1), 16), dtype=torch.uint8,
                     device="cuda")
    g1 = graph_of(lambda s: wb.rmsnorm_gemv(x, gm, W, y, 1e-6, workspace=ws, stream=s), n)
    sink = torch.zeros(16, dtype=torch.int32, device="cuda")
    probe = torch.zeros(1 << 20, dtype=torch.int32, device="cuda")
    ge = graph_of(lambda s: wb.empty_probe(0, probe, sink, stream=s), n)
    gt = graph_of(lambda s: wb.empty_probe(1, probe, sink, stream=s), n)
    out["config1_rmsnorm_gemv_256"] = {
        "us_per_launch": round(events(g1.replay, 20) / n * 1e6, 3),
        "empty_kernel_us": round(events(ge.replay, 20) / n * 1e6, 3),
        "one_dram_round_trip_us": round(events(gt.replay, 20) / n * 1e6, 3)}
    # config 2: one block, warm and cold
    sh = synth.QwenShape(layers=1)
    chains = []
    for c in range(6):
        blk = synth.qwen_block_weights(sh, args.seed + c, 0)
        dblk = {k: to_dev(v, torch) for k, v in blk.items()}
        dattn = to_dev(synth.qwen_attn(sh, 1, args.seed + c, 0), torch)[None]
        dh = torch.from_numpy(synth.qwen_hidden(sh, 1, args.seed + c)).cuda()
        ch = wc.qwen_chain([dblk], None, dattn, dh, eps=sh.eps, prefetch=0)
        ch.chain.capture()
        chains.append(ch)
    warm = events(lambda: chains[0].run(st), 200)

    def cold_round():
        for ch in chains:
            ch.run(st)
    cold = events(cold_round, 50) / len(chains)
    bb = sh.block_weight_bytes()
    out["config2_one_block_b1"] = {"warm_us": round(warm * 1e6, 2),
                                   "warm_gbs": round(bb / warm / 1e9, 1),
                                   "cold_us": round(cold * 1e6, 2),
                                   "cold_gbs": round(bb / cold / 1e9, 1), "bytes": bb}
    for ch in chains:
        ch.chain.close()
    del chains
    # config 4: prefetch plans vs none, warm and cold
    msh = synth.MlpShape()
    mout = []
    sets = []
    for c in range(6):
        hb = [synth.mlp_block_weights(msh, args.seed + c, l) for l in range(msh.blocks)]
        sets.append([{k: to_dev(v, torch) for k, v in b.items()} for b in hb])
    for B in (4, 16):
        x_in = to_dev(synth.mlp_input(msh, B, args.seed), torch)
        res = {"B": B}
        for pf in (0, 1):
            chs = []
            for c in range(6):
                ch = wc.mlp_chain(sets[c], x_in, eps=msh.eps, prefetch=pf)
                if pf:
                    ch.chain.tune()
                ch.chain.capture()
                chs.append(ch)
            key = "tuned" if pf else "none"
            res[key + "_warm_us"] = round(events(lambda: chs[0].run(st), 200) * 1e6, 2)

            def rnd(chs=chs):
                for ch in chs:
                    ch.run(st)
            res[key + "_cold_us"] = round(events(rnd, 30) / len(chs) * 1e6, 2)
            if pf:
                pl = chs[0].chain.plans()
                res["plans_kept"] = sum(1 for p in pl if p[0][0] != 0)
                res["best_lower_ci"] = round(max(p[1] for p in pl), 4)
            for ch in chs:
                ch.chain.close()
        mout.append(res)
    out["config4_mlp_chain"] = mout
    print(json.dumps(out), flush=True)
    return 0


def _graph_time(torch, fn, n_inner, reps=10):
    """Seconds per inner launch of fn(stream) captured in one CUDA graph and
    replayed `reps` times between CUDA events (after a warm call and three
    warm replays)."""
    st = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(st)
    with torch.cuda.stream(side):
        fn(side)
    st.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn(torch.cuda.current_stream())
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        g.replay()
    e1.record(st)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e-3 / (reps * n_inner)


def run_q4(args):
    """4-bit group-128 weights, one JSON line:
    - each GEMV shape of the Qwen2.5-1.5B decode step at batch 1, 2 and 4
      (packed rows quantised on the GPU from random bf16 weights, rotating
      copies of at least 256 MB, launched back to back with programmatic
      dependent launch in one CUDA graph): time per launch and the packed
      bytes over it against the measured copy peak;
    - the whole decode step (28 blocks and the LM head) on 4-bit weights
      quantised from the same bf16 weights as the bf16 chain, both timed as
      graph replays between CUDA events, at batch 1 and 4."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from weight_streaming_gemv_bf16_gb300 import binding as wb
    from weight_streaming_gemv_bf16_gb300 import chain as wc
    torch.cuda.set_device(0)
    st = torch.cuda.current_stream()
    gen = torch.Generator(device="cuda").manual_seed(args.seed)
    hbm = peaks()[0]
    base = wb.get_tuning()
    t = wb.Tuning()
    for f, _ in wb.Tuning._fields_:
        setattr(t, f, getattr(base, f))
    t.launch_pdl = 1
    wb.set_tuning(t)
    gemv = []
    shapes = [(2048, 1536), (1536, 1536), (8960, 1536), (1536, 8960), (151936, 1536)]
    batches = (1, 2, 4)
    if args.q4_gemv:
        M1, K1, B1 = (int(v) for v in args.q4_gemv.split(","))
        shapes, batches = [(M1, K1)], (B1,)
    try:
        for M, K in shapes:
            rb = wb.q4_row_bytes(K)
            nbytes = M * rb
            ncopy = max(2, -(-(256 << 20) // nbytes))
            W = (torch.randn((M, K), device="cuda", generator=gen) * 0.02).to(torch.bfloat16)
            Wqs = []
            for _ in range(ncopy):
                Wq = torch.empty((M, rb), dtype=torch.uint8, device="cuda")
                wb.quantize_q4(W, Wq)
                Wqs.append(Wq)
            del W
            for B in batches:
                x = torch.randn((B, K), device="cuda", generator=gen).to(torch.bfloat16)
                y = torch.empty((B, M), device="cuda")

                def fn(s, Wqs=Wqs, x=x, y=y, K=K):
                    for Wq in Wqs:
                        wb.gemv_q4(Wq, x, y, K, stream=s)
                dt = _graph_time(torch, fn, ncopy)
                gemv.append({"M": M, "K": K, "batch": B, "us_per_launch": round(dt * 1e6, 2),
                             "packed_bytes": nbytes, "GB_s": round(nbytes / dt / 1e9, 1),
                             "frac_of_measured_hbm": round(nbytes / dt / 1e9 / hbm, 3)})
            del Wqs
            torch.cuda.empty_cache()
    finally:
        wb.set_tuning(base)
    if args.q4_gemv:
        print(json.dumps({"mode": "q4", "hbm_peak_gbs": hbm, "gemv": gemv}))
        return 0

    sh, blocks, head, attn, h0 = make_host_inputs(4, args.seed)
    dblocks = [{k: to_dev(v, torch) for k, v in b.items()} for b in blocks]
    dhead = {k: to_dev(v, torch) for k, v in head.items()}
    mats = ("Wq", "Wk", "Wv", "Wo", "Wg", "Wu", "Wd")

    def packed(Wbf):
        Wq = torch.empty((Wbf.shape[0], wb.q4_row_bytes(Wbf.shape[1])), dtype=torch.uint8,
                         device="cuda")
        wb.quantize_q4(Wbf, Wq)
        return Wq
    qblocks = [{k: (packed(v) if k in mats else v) for k, v in b.items()} for b in dblocks]
    qhead = {"gamma_f": dhead["gamma_f"], "Wlm": packed(dhead["Wlm"])}
    torch.cuda.synchronize()
    q4_bytes = sum(v.numel() for b in qblocks for k, v in b.items() if k in mats)
    q4_bytes += qhead["Wlm"].numel()
    bf16_bytes = sh.chain_weight_bytes()
    chain = {"weights_bf16_bytes": bf16_bytes, "weights_q4_bytes": q4_bytes,
             "bytes_ratio": round(bf16_bytes / q4_bytes, 3)}
    for B in (1, 4):
        dattn = to_dev(attn[:, :B], torch)
        dh0 = torch.from_numpy(np.ascontiguousarray(h0[:B])).cuda()
        res = {}
        for name, blks, hd, q4 in (("bf16", dblocks, dhead, False), ("q4", qblocks, qhead, True)):
            ch = wc.qwen_chain(blks, hd, dattn, dh0, eps=sh.eps, use_pdl=True, q4=q4)
            ch.chain.capture()
            for _ in range(5):
                ch.run(st)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n = 200
            e0.record(st)
            for _ in range(n):
                ch.run(st)
            e1.record(st)
            torch.cuda.synchronize()
            res[name] = e0.elapsed_time(e1) * 1e3 / n
            del ch
        chain[f"batch{B}"] = {
            "bf16_us_per_step": round(res["bf16"], 1), "q4_us_per_step": round(res["q4"], 1),
            "speedup": round(res["bf16"] / res["q4"], 2),
            "q4_GB_s": round(q4_bytes / res["q4"] / 1e3, 1),
            "q4_frac_of_measured_hbm": round(q4_bytes / res["q4"] / 1e3 / hbm, 3)}
    assert wb.device_error() == 0
    print(json.dumps({"mode": "q4", "hbm_peak_gbs": hbm, "gemv": gemv, "chain": chain}))
    return 0


def run_step_attention(args):
    """The Qwen2.5-1.5B decode step with decode attention in every block (the
    configs' seeded stand-in replaced), one JSON line: per batch (1, 4) and
    cached slots (1024, 4096, 32768 at batch 1) the time per step as graph
    replays between CUDA events, beside the same step with the stand-in."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from weight_streaming_gemv_bf16_gb300 import binding as wb
    from weight_streaming_gemv_bf16_gb300 import chain as wc
    from weight_streaming_gemv_bf16_gb300 import synth
    torch.cuda.set_device(0)
    st = torch.cuda.current_stream()
    gen = torch.Generator(device="cuda").manual_seed(args.seed)
    sh = synth.QWEN2_5_1_5B
    H, KV, I, V, L = sh.hidden, sh.kv_dim, sh.inter, sh.vocab, sh.layers

    def rnd(*s, scale=0.02):
        return (torch.randn(s, device="cuda", generator=gen) * scale).to(torch.bfloat16)
    blocks = [{"gamma1": rnd(H, scale=0.1) + 1, "gamma2": rnd(H, scale=0.1) + 1,
               "Wq": rnd(H, H), "Wk": rnd(KV, H), "Wv": rnd(KV, H), "Wo": rnd(H, H),
               "Wg": rnd(I, H), "Wu": rnd(I, H), "Wd": rnd(H, I)} for _ in range(L)]
    head = {"gamma_f": rnd(H, scale=0.1) + 1, "Wlm": rnd(V, H)}

    def step_us(ch, n=100):
        ch.chain.capture()
        for _ in range(5):
            ch.run(st)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(n):
            ch.run(st)
        e1.record(st)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / n
    rows = []
    for B, n in ((1, 1024), (1, 4096), (1, 32768), (4, 1024), (4, 4096)):
        h0 = torch.randn((B, H), device="cuda", generator=gen)
        attn = rnd(L, B, H, scale=1.0)
        base = wc.qwen_chain(blocks, head, attn, h0, eps=sh.eps)
        t_base = step_us(base)
        del base
        caches = [(rnd(B, KV // 128, n, 128, scale=1.0), rnd(B, KV // 128, n, 128, scale=1.0))
                  for _ in range(L)]
        pos = torch.full((B,), n - 1, dtype=torch.int32, device="cuda")
        ch = wc.qwen_chain(blocks, head, None, h0, eps=sh.eps, caches=caches, pos=pos)
        t_att = step_us(ch)
        del ch, caches
        torch.cuda.empty_cache()
        cache_bytes = L * B * (KV // 128) * n * 128 * 2 * 2
        rows.append({"batch": B, "cached_slots": n, "step_us": round(t_att, 1),
                     "step_us_with_stand_in": round(t_base, 1),
                     "attention_us_per_step": round(t_att - t_base, 1),
                     "kv_cache_bytes_read": cache_bytes})
    assert wb.device_error() == 0
    print(json.dumps({"mode": "step-attention", "rows": rows}))
    return 0


def run_attention(args):
    """Decode attention with the key-value append, Qwen2.5-1.5B heads (12 query
    heads over 2 key-value heads of 128), one JSON line: per (batch, cached
    slots) the time per launch over rotating caches larger than L2 (launched
    back to back in one CUDA graph, CUDA events around it), and the
    algorithmic bytes per launch (the key and value rows of slots 0..pos read,
    the new rows written, q read and the fp32 output written) over that time
    against the measured copy peak."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from weight_streaming_gemv_bf16_gb300 import binding as wb
    torch.cuda.set_device(0)
    st = torch.cuda.current_stream()
    gen = torch.Generator(device="cuda").manual_seed(args.seed)
    hbm = peaks()[0]
    nh, nkv, d = 12, 2, 128
    rows = []
    configs = [(B, n) for B in (1, 4, 16) for n in (1024, 4096, 32768)]
    if args.attn_config:
        configs = [tuple(int(v) for v in args.attn_config.split(","))]
    for B, n in configs:
        if True:
            S = n
            cache_b = B * nkv * S * d * 2
            ncopy = max(2, -(-(256 << 20) // (2 * cache_b)))
            ks = [torch.randn((B, nkv, S, d), device="cuda", generator=gen).to(torch.bfloat16)
                  for _ in range(ncopy)]
            vs = [torch.randn((B, nkv, S, d), device="cuda", generator=gen).to(torch.bfloat16)
                  for _ in range(ncopy)]
            q = torch.randn((B, nh * d), device="cuda", generator=gen)
            kn = torch.randn((B, nkv * d), device="cuda", generator=gen)
            vn = torch.randn((B, nkv * d), device="cuda", generator=gen)
            pos = torch.full((B,), n - 1, dtype=torch.int32, device="cuda")
            ws = torch.zeros(wb.attention_workspace_bytes(B, nh, nkv, S), dtype=torch.uint8,
                             device="cuda")
            out = torch.empty((B, nh * d), device="cuda")

            def fn(s):
                for c in range(ncopy):
                    wb.decode_attention(q, kn, vn, ks[c], vs[c], pos, ws, out, None, stream=s)
            side = torch.cuda.Stream()
            side.wait_stream(st)
            with torch.cuda.stream(side):
                fn(side)
            st.wait_stream(side)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn(torch.cuda.current_stream())
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            reps = max(3, min(50, (400 << 20) // (ncopy * 2 * cache_b)))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _ in range(reps):
                g.replay()
            e1.record(st)
            torch.cuda.synchronize()
            dt = e0.elapsed_time(e1) * 1e-3 / (reps * ncopy)
            nbytes = B * nkv * (2 * n * d * 2 + 2 * d * 2) + B * nh * d * 4 * 2
            rows.append({"batch": B, "cached_slots": n, "us_per_launch": round(dt * 1e6, 2),
                         "algorithmic_bytes": nbytes, "GB_s": round(nbytes / dt / 1e9, 1),
                         "frac_of_measured_hbm": round(nbytes / dt / 1e9 / hbm, 3)})
            del ks, vs
            torch.cuda.empty_cache()
    assert wb.device_error() == 0
    print(json.dumps({"mode": "attention", "heads": [nh, nkv, d], "hbm_peak_gbs": hbm,
                      "l2": "rotating caches, at least 256 MB per graph replay", "rows": rows}))
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.mode == "kernel":
        return run_kernel_only(args)
    if args.mode == "sweep":
        return run_sweep(args)
    if args.mode == "configs":
        return run_configs(args)
    if args.mode == "attention":
        return run_attention(args)
    if args.mode == "q4":
        return run_q4(args)
    if args.mode == "step-attention":
        return run_step_attention(args)
    if args.mode == "prefetch":
        return run_prefetch_probe(args)
    if args.mode == "train":
        return run_train(args)
    if args.mode == "crossover":
        return run_crossover(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
