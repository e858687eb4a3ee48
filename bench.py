"""Benchmark of the linear-attention hot path on GB300.

One JSON line on rank 0.  The headline ``value`` is gated-linear-attention
prefill throughput (tokens/s) on B=4, H=16, T=4096, d_k=d_v=128, chunk 64,
bf16 activations, fp32 state; a step is one prefill call over the whole batch.
Sub-objects report Gated DeltaNet decode at batch 256 (16 heads, 512-slot
fp32 state pool, conv cache), Gated DeltaNet prefill (B=2, H=16, T=8192, conv
+ L2 norm) and the long-context run (B=1, H=32, T=32768 in three segments,
then 64 requests x 4-token speculative decode), each with its roofline.

Timing: W untimed warm-up steps, then K steps between a barrier and
torch.cuda.synchronize() on both sides, CUDA events on the launching stream,
max over ranks.  No step finds the previous step's data in L2 (129 MB): the
working set of a step is larger than L2, or, where it is smaller (the SSD-form
prefill, the selective scan, the replay round), consecutive steps cycle over
disjoint copies of their buffers whose combined footprint is about three times
L2, so no flush is needed.  Multi-GPU runs are replicas: each rank runs the same per-GPU workload
("scaling": "weak"); there is no data-path collective.

``--impl reference`` times the plain fp64 CPU oracle on the host cores on a
bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill tokens/s (%tensor peak); decode tokens/s at batch 256 (%HBM BW)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------

def dist_setup(backend="nccl"):
    """One process per GPU from the launcher's environment.  The replicas
    exchange nothing on the data path: the process group only carries the
    barriers around the timed region and the max over ranks of its time."""
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return dist, rank, ws, local
    return None, 0, 1, 0


def aggregate(units_per_rank, world_size, ms_max):
    """Whole-job throughput of weak-scaled replicas: every rank processes the
    same number of units; the job takes as long as its slowest rank."""
    return units_per_rank * world_size / (ms_max / 1e3)


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float, device):
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def timed_steps(fn, steps, warmup, dist, device):
    """Returns (ms per step over the timed region, [per-step event ms])."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    barrier(dist)
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(steps):
        fn()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    total = ev[0].elapsed_time(ev[steps])
    return max_over_ranks(dist, total / steps, device), per


L2_BYTES = 129 * 10**6


def rotation(step_bytes, most=8):
    """Number of disjoint buffer copies for a step touching ``step_bytes``, so
    that the memory touched between two uses of one copy is about 3x L2."""
    return max(1, min(most, -(-3 * L2_BYTES // max(1, step_bytes))))


def cycling(fns):
    """A step that runs the next of several equivalent steps (each on its own
    buffers) on every call."""
    state = {"i": 0}

    def step():
        fns[state["i"] % len(fns)]()
        state["i"] += 1
    return step


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "gated_deltanet_02_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, src_files, units_scale=1.0):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(kernel)
    if not ent or ent.get("source_hash") != source_hash(*src_files):
        return None
    return ent["dram_bytes_per_launch"] * units_scale


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------

GLA_CFG = dict(B=4, H=16, T=4096, d=128)
GDN_CFG = dict(B=2, H=16, T=8192, d=128)
DEC_CFG = dict(N=256, H=16, d=128, P=512)


def gla_bytes_flops(B, H, T, d):
    bt = B * T * H
    bytes_ = bt * d * 2 * 3 + bt * 4 + bt * d * 2 + B * H * d * d * 4  # q k v, alpha, o (bf16), S_T
    flops = bt * (4 * 64 * d + 4 * d * d)  # QK^T, PV, QS, K^T V per head-token
    return bytes_, flops


def gdn_bytes_flops(B, H, T, d):
    bt = B * T * H
    bytes_ = bt * d * 2 * 3 + bt * 8 + bt * d * 2 + 2 * B * H * d * d * 4 + 3 * H * d * 16
    flops = bt * (10 * 64 * d + 6 * d * d + 64 * 64 // 3)
    return bytes_, flops


def decode_state_bytes(N, H, d):
    return N * H * d * d * 4 * 2  # read + write of every touched fp32 state


def run_ours(args):
    import torch

    from gated_deltanet_02_gb300 import GDN, GLA, glinattn_decode, glinattn_prefill, inputs
    dist, rank, ws, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk, pk_kind = peaks()
    hbm, tc = pk["hbm_gbs"], pk["bf16_tflops"]

    # ---- GLA prefill (headline) ------------------------------------------------
    c = GLA_CFG
    ex = inputs.gla_prefill(c["B"], c["H"], c["T"], c["d"], seed=rank, device=dev)
    o = torch.empty(c["B"], c["T"], c["H"], c["d"], dtype=torch.bfloat16, device=dev)
    S = torch.empty(c["B"], c["H"], c["d"], c["d"], dtype=torch.float32, device=dev)

    def step_gla():
        glinattn_prefill(ex["q"], ex["k"], ex["v"], ex["alpha"], None, None, variant=GLA, o=o, S_T=S)

    with ClockSampler(local) as clk:
        ms, per = timed_steps(step_gla, args.steps, args.warmup, dist, dev)
    tokens = c["B"] * c["T"]
    gbytes, gflops = gla_bytes_flops(**c)
    kern_ms = statistics.mean(per)
    value = aggregate(tokens, ws, ms)

    # ---- end to end through the C ABI with host buffers -------------------------
    # Every step copies its inputs in from pinned host memory, runs the prefill
    # and copies o and S_T back; steps are pipelined over two buffer sets with
    # the copies in and out on their own streams (both directions of the host
    # link and the kernel run side by side), so the figure is the whole job's
    # rate.  The copy in (202 MB a step) sets it: spreading it over three copy
    # streams measured no faster.  The step's inputs sit in one pinned buffer
    # (q, k, v, alpha back to back, each at a 16-byte boundary), so the copy
    # in is one transfer; the prefill gets views into the device copy.
    names = ("q", "k", "v", "alpha")
    sizes = [ex[k].numel() * ex[k].element_size() for k in names]
    offs = [sum((n + 255) // 256 * 256 for n in sizes[:i]) for i in range(len(sizes))]
    total = offs[-1] + sizes[-1]

    def views(buf):
        return {k: buf[off:off + n].view(ex[k].dtype).view(ex[k].shape) for k, off, n in zip(names, offs, sizes)}

    hraw = torch.empty(total, dtype=torch.uint8).pin_memory()
    host = views(hraw)
    for k in names:
        host[k].copy_(ex[k].cpu())
    o_h = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    S_h = [torch.empty(S.shape, dtype=S.dtype).pin_memory() for _ in range(2)]
    draw = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    dbuf = [views(d) for d in draw]
    o2 = [o, torch.empty_like(o)]
    S2 = [S, torch.empty_like(S)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    comp = torch.cuda.current_stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for j in range(2):  # every event recorded once, so the first waits are satisfied
        for e in (ev_in[j], ev_comp[j], ev_out[j]):
            e.record(comp)

    def step_e2e(i):
        j = i % 2
        s_in.wait_event(ev_comp[j])  # buffer set j's last prefill has read its inputs
        with torch.cuda.stream(s_in):
            draw[j].copy_(hraw, non_blocking=True)
            ev_in[j].record(s_in)
        comp.wait_event(ev_in[j])
        comp.wait_event(ev_out[j])  # and its last outputs are copied out
        glinattn_prefill(dbuf[j]["q"], dbuf[j]["k"], dbuf[j]["v"], dbuf[j]["alpha"], None, None, variant=GLA,
                         o=o2[j], S_T=S2[j])
        ev_comp[j].record(comp)
        s_out.wait_event(ev_comp[j])
        with torch.cuda.stream(s_out):
            o_h[j].copy_(o2[j], non_blocking=True)
            S_h[j].copy_(S2[j], non_blocking=True)
            ev_out[j].record(s_out)

    def e2e_timed(steps, warmup):
        for i in range(warmup):
            step_e2e(i)
        torch.cuda.synchronize()
        barrier(dist)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(comp)
        s_in.wait_event(t0)
        for i in range(steps):
            step_e2e(warmup + i)
        for j in range(2):
            comp.wait_event(ev_out[j])
        t1.record(comp)
        torch.cuda.synchronize()
        barrier(dist)
        return max_over_ranks(dist, t0.elapsed_time(t1) / steps, dev)

    e2e_ms = e2e_timed(max(4, args.steps // 2), 2)
    h2d = hraw.numel()  # the bytes the one copy in moves (inputs plus alignment gaps)
    d2h = o_h[0].numel() * o_h[0].element_size() + S_h[0].numel() * S_h[0].element_size()

    # ---- Gated DeltaNet decode, batch 256 -----------------------------------------
    dc = DEC_CFG
    dx = inputs.gdn_decode(dc["N"], dc["H"], dc["d"], dc["P"], seed=rank, device=dev)
    od = torch.empty(dc["N"], dc["H"], dc["d"], dtype=torch.bfloat16, device=dev)

    def step_dec():
        glinattn_decode(dx["q"], dx["k"], dx["v"], dx["alpha"], dx["beta"], dx["pool"], dx["slot_ids"],
                        variant=GDN, conv_w=dx["conv_w"], conv_pool=dx["conv_pool"], qk_l2norm=True, o=od)

    dec_ms, dec_per = timed_steps(step_dec, max(args.steps, 20), max(args.warmup, 3), dist, dev)
    dsb = decode_state_bytes(dc["N"], dc["H"], dc["d"])
    dec_kms = statistics.mean(dec_per)

    # ---- Gated DeltaNet prefill -------------------------------------------------------
    g = GDN_CFG
    gx = inputs.gdn_prefill(g["B"], g["H"], g["T"], g["d"], seed=rank, device=dev)
    og = torch.empty(g["B"], g["T"], g["H"], g["d"], dtype=torch.bfloat16, device=dev)
    Sg = torch.empty(g["B"], g["H"], g["d"], g["d"], dtype=torch.float32, device=dev)

    from gated_deltanet_02_gb300.glinattn import prefill_workspace_size
    gws = torch.empty(max(1, prefill_workspace_size(g["B"], g["T"], g["H"], g["d"])), dtype=torch.uint8, device=dev)

    def step_gdn():
        glinattn_prefill(gx["q"], gx["k"], gx["v"], gx["alpha"], gx["beta"], gx["S0"], variant=GDN,
                         conv_w=gx["conv_w"], qk_l2norm=True, o=og, S_T=Sg, workspace=gws)

    gdn_ms, gdn_per = timed_steps(step_gdn, max(3, min(args.steps, 20)), 3, dist, dev)
    gdn_bytes, gdn_flops = gdn_bytes_flops(**g)

    # the same prefill keeping a prefix-cache checkpoint (state + conv cache) every 1024 tokens
    every = 1024
    nblk = g["T"] // every
    Sb = torch.empty(g["B"], nblk, g["H"], g["d"], g["d"], dtype=torch.float32, device=dev)
    cb = torch.empty(g["B"], nblk, 3, 3 * g["H"] * g["d"], dtype=torch.bfloat16, device=dev)

    def step_gdn_ck():
        glinattn_prefill(gx["q"], gx["k"], gx["v"], gx["alpha"], gx["beta"], gx["S0"], variant=GDN,
                         conv_w=gx["conv_w"], qk_l2norm=True, o=og, S_T=Sg, state_every=every, S_blocks=Sb,
                         conv_blocks=cb, workspace=gws)

    ck_ms, _ = timed_steps(step_gdn_ck, max(3, min(args.steps, 20)), 3, dist, dev)
    ck_bytes = Sb.numel() * 4 + cb.numel() * 2

    # ---- long context: 3-segment prefill, then 64 x 4 speculative decode -------------
    lc = long_context_run(args, dist, dev, rank)

    # ---- the SSD form: state 128 x head dim 64, one q / k group for 32 heads ---------
    ssd = ssd_run(args, dist, dev, rank)

    # ---- normalised kernelised linear attention ---------------------------------------
    nla = nla_run(args, dist, dev, rank)

    # ---- Mamba's selective scan -----------------------------------------------------------
    scan = scan_run(args, dist, dev, rank)

    # ---- CPU baseline: the oracle on this host's cores (rank 0) -----------------------
    cpu = cpu_baseline_run(ex, budget_s=args.cpu_seconds) if rank == 0 and not args.no_cpu else None

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    traffic = profiled_traffic("gla_prefill_kernel", ["prefill_tc.cu", "sm100.cuh", "tc_common.cuh"])
    prep_t = profiled_traffic("gdn_prep_kernel", ["gdn_tc.cu", "sm100.cuh", "tc_common.cuh", "frontend.cuh"])
    scan_t = profiled_traffic("gdn_scan_kernel", ["gdn_tc.cu", "sm100.cuh", "tc_common.cuh", "frontend.cuh"])
    gdn_traffic = prep_t + scan_t if prep_t is not None and scan_t is not None else None
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; q,k ~ N(0,1)/sqrt(d), v ~ N(0,1), alpha = sigmoid(N(0,1)+3))",
        "config": {"workload": "gated linear attention prefill, B=4 H=16 T=4096 d_k=d_v=128 C=64, "
                               "bf16 q/k/v/o, fp32 alpha and state, S0 = 0",
                   "global_batch": c["B"] * ws, "seq_len": c["T"], "parallelism": f"replicas x{ws}",
                   "l2": "inputs larger than L2 (no flush needed); smaller sub-benchmarks cycle over "
                         "disjoint buffer copies totalling ~3x L2"},
        "roofline": {"bound": "hbm", "achieved": gbytes / (kern_ms / 1e3) / 1e9, "peak": hbm,
                     "unit": "GB/s", "frac": gbytes / (kern_ms / 1e3) / 1e9 / hbm,
                     "traffic": traffic, "peak_kind": f"{pk_kind} burst copy",
                     "algorithmic_bytes": gbytes, "kernel": "gla_prefill_kernel"},
        "tensor": {"flops": gflops, "achieved_tflops": gflops / (kern_ms / 1e3) / 1e12,
                   "peak_tflops": tc, "frac": gflops / (kern_ms / 1e3) / 1e12 / tc,
                   "peak_kind": f"{pk_kind} bf16 burst",
                   # time at the roofline, max(FLOPs / tensor peak, bytes / HBM), over the measured time
                   "attainable_frac": max(gflops / (tc * 1e12), gbytes / (hbm * 1e9)) / (kern_ms / 1e3)},
        "e2e": {"value": tokens * ws / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "long_context": lc,
        "ssd": ssd,
        "normalized_linear_attention": nla,
        "selective_scan": scan,
        "cpu_baseline": cpu,
        "decode": {"value": dc["N"] * ws / (dec_ms / 1e3), "unit": "tokens/s",
                   "config": "Gated DeltaNet decode, 256 requests x 16 heads, d=128, 512-slot fp32 pool, "
                             "conv cache + L2 norm, in place",
                   "ms_per_step": dec_ms,
                   "roofline": {"bound": "hbm", "achieved": dsb / (dec_kms / 1e3) / 1e9, "peak": hbm,
                                "unit": "GB/s", "frac": dsb / (dec_kms / 1e3) / 1e9 / hbm,
                                "traffic": profiled_traffic("decode128_kernel", ["decode128.cu", "sm100.cuh", "frontend.cuh"]),
                                "algorithmic_bytes": dsb, "kernel": "decode128_kernel"}},
        "gdn_prefill": {"value": g["B"] * g["T"] * ws / (gdn_ms / 1e3), "unit": "tokens/s",
                        "config": "Gated DeltaNet prefill, B=2 H=16 T=8192 d=128, conv + L2 norm",
                        "ms_per_step": gdn_ms,
                        "roofline": {"bound": "hbm",
                                     "achieved": gdn_bytes / (statistics.mean(gdn_per) / 1e3) / 1e9,
                                     "peak": hbm, "unit": "GB/s",
                                     "frac": gdn_bytes / (statistics.mean(gdn_per) / 1e3) / 1e9 / hbm,
                                     "traffic": gdn_traffic, "algorithmic_bytes": gdn_bytes,
                                     "kernels": "gdn_prep_kernel + gdn_scan_kernel"},
                        "tensor_frac": gdn_flops / (statistics.mean(gdn_per) / 1e3) / 1e12 / tc,
                        "with_checkpoints": {"state_every": every, "ms_per_step": ck_ms,
                                             "checkpoint_bytes": ck_bytes,
                                             "overhead_frac": ck_ms / gdn_ms - 1.0}}
    }
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def long_context_run(args, dist, dev, rank):
    """Gated DeltaNet, B=1, H=32, T=32768 prefilled as segments of 6553 / 11468
    / 14747 tokens (state and conv cache handed on), then 64 requests each
    decoding 4 draft tokens from their own copy of the state, one state kept
    per draft position."""
    import torch

    from gated_deltanet_02_gb300 import (GDN, glinattn_prefill, glinattn_replay, glinattn_spec_decode,
                                         glinattn_state_copy, inputs)
    pk, _ = peaks()
    B, H, T, d = 1, 32, 32768, 128
    ex = inputs.gdn_prefill(B, H, T, d, seed=rank, device=dev, s0_std=0.0)
    segs = inputs.segment_lengths(T)
    parts, s0 = [], 0
    for L in segs:
        sl = slice(s0, s0 + L)
        parts.append({k: ex[k][:, sl].contiguous() for k in ("q", "k", "v", "alpha", "beta")})
        s0 += L
    outs = [torch.empty(B, L, H, d, dtype=torch.bfloat16, device=dev) for L in segs]
    S = torch.empty(B, H, d, d, device=dev)
    conv = [torch.empty(B, 3, 3 * H * d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    from gated_deltanet_02_gb300.glinattn import prefill_workspace_size
    ws = torch.empty(prefill_workspace_size(B, max(segs), H, d), dtype=torch.uint8, device=dev)

    def step_prefill():
        for i, part in enumerate(parts):
            glinattn_prefill(part["q"], part["k"], part["v"], part["alpha"], part["beta"],
                             None if i == 0 else S, variant=GDN, conv_w=ex["conv_w"],
                             conv_in=None if i == 0 else conv[(i - 1) % 2], conv_out=conv[i % 2],
                             qk_l2norm=True, o=outs[i], S_T=S, workspace=ws)

    pre_ms, _ = timed_steps(step_prefill, 2, 1, dist, dev)
    N, D = 64, 4
    P = N * (1 + D)
    pool = torch.zeros(P, H, d, d, device=dev)
    cpool = torch.zeros(P, 3, 3 * H * d, dtype=torch.bfloat16, device=dev)
    pool[:N] = S[0]
    cpool[:N] = conv[(len(segs) - 1) % 2][0]
    src = torch.arange(N, dtype=torch.int32, device=dev)
    dst = (N + torch.arange(N * D, dtype=torch.int32, device=dev)).view(N, D)
    dr = inputs.spec_drafts(N, D, H, d, seed=rank + 1, device=dev)
    od = torch.empty(N, D, H, d, dtype=torch.bfloat16, device=dev)

    def step_spec():
        glinattn_spec_decode(dr["q"], dr["k"], dr["v"], dr["alpha"], dr["beta"], pool, src, dst,
                             variant=GDN, conv_w=ex["conv_w"], conv_pool=cpool, qk_l2norm=True, o=od)

    spec_ms, spec_per = timed_steps(step_spec, max(10, args.steps), 3, dist, dev)
    spec_bytes = N * H * (1 + D) * d * d * 4
    k_ms = statistics.mean(spec_per)

    # the replay-buffer alternative: verify without per-draft states, then apply
    # each request's accepted drafts (a ~ U{0..4}) to its own slot in place
    accept = dr["accept"].to(torch.int32)
    # the 64 slots a round touches (134 MB) cycle over disjoint slot sets of the
    # pool (the states the speculative round above left in them)
    rsets = [torch.arange(i * N, (i + 1) * N, dtype=torch.int32, device=dev)
             for i in range(rotation(N * H * d * d * 4, most=P // N))]

    def replay_round(rs):
        glinattn_spec_decode(dr["q"], dr["k"], dr["v"], dr["alpha"], dr["beta"], pool, rs, None,
                             variant=GDN, conv_w=ex["conv_w"], conv_pool=cpool, qk_l2norm=True, o=od)
        glinattn_replay(dr["k"], dr["v"], dr["alpha"], dr["beta"], pool, rs, accept, q=dr["q"], variant=GDN,
                        conv_w=ex["conv_w"], conv_pool=cpool, qk_l2norm=True)

    step_replay = cycling([lambda rs=rs: replay_round(rs) for rs in rsets])
    rep_ms, rep_per = timed_steps(step_replay, max(10, args.steps), 3, dist, dev)
    n_acc = int((accept > 0).sum().item())
    rep_bytes = N * H * d * d * 4 + 2 * n_acc * H * d * d * 4

    # copy on write: 64 request slots copied whole (state + conv cache) into 64 others
    csrc = torch.arange(N, dtype=torch.int32, device=dev)
    cdst = N + csrc

    def step_copy():
        glinattn_state_copy(pool, csrc, cdst, conv_pool=cpool)

    copy_ms, copy_per = timed_steps(step_copy, max(10, args.steps), 3, dist, dev)
    copy_bytes = 2 * N * (H * d * d * 4 + 3 * 3 * H * d * 2)
    return {"config": "Gated DeltaNet, B=1 H=32 T=32768 in segments 6553/11468/14747 (conv + L2 norm), "
                      "then 64 requests x 4 draft tokens, one fp32 state per draft position",
            "prefill_tokens_per_s": T / (pre_ms / 1e3), "prefill_ms": pre_ms,
            "spec_draft_tokens_per_s": N * D / (spec_ms / 1e3), "spec_ms_per_round": spec_ms,
            "spec_roofline": {"bound": "hbm", "achieved": spec_bytes / (k_ms / 1e3) / 1e9,
                              "peak": pk["hbm_gbs"], "unit": "GB/s",
                              "frac": spec_bytes / (k_ms / 1e3) / 1e9 / pk["hbm_gbs"],
                              "algorithmic_bytes": spec_bytes},
            "replay_rollback": {"config": "verify-only speculative decode + replay of the accepted drafts "
                                          f"({n_acc} of {N} requests accept at least one), in place",
                                "ms_per_round": rep_ms, "pool_slots_needed": N,
                                "pool_slots_needed_per_draft_states": N * (1 + D),
                                "roofline": {"bound": "hbm",
                                             "achieved": rep_bytes / (statistics.mean(rep_per) / 1e3) / 1e9,
                                             "peak": pk["hbm_gbs"], "unit": "GB/s",
                                             "frac": rep_bytes / (statistics.mean(rep_per) / 1e3) / 1e9
                                             / pk["hbm_gbs"], "algorithmic_bytes": rep_bytes}},
            "slot_copy": {"config": "64 whole slots (32 heads x 128 x 128 fp32 + bf16 conv cache) copied",
                          "ms": copy_ms,
                          "roofline": {"bound": "hbm",
                                       "achieved": copy_bytes / (statistics.mean(copy_per) / 1e3) / 1e9,
                                       "peak": pk["hbm_gbs"], "unit": "GB/s",
                                       "frac": copy_bytes / (statistics.mean(copy_per) / 1e3) / 1e9
                                       / pk["hbm_gbs"], "algorithmic_bytes": copy_bytes}}}


def ssd_run(args, dist, dev, rank):
    """The SSD form of Mamba2 as gated linear attention: a B=2, T=4096 prefill
    of 32 heads (head dim 64, state size 128) sharing one q / k group, and a
    decode step of 256 requests x 32 heads from a 512-slot pool."""
    import torch

    from gated_deltanet_02_gb300 import GLA, glinattn_decode, glinattn_prefill, inputs
    pk, _ = peaks()
    B, H, G, T, dk, dv = 2, 32, 1, 4096, 128, 64
    pre_bytes = B * T * G * dk * 2 * 2 + B * T * H * (dv * 2 * 2 + 4) + B * H * dk * dv * 4
    steps = []
    for i in range(rotation(pre_bytes)):  # a step's 71 MB fit in L2: cycle over disjoint copies
        ex = inputs.ssd_prefill(B, H, G, T, seed=rank + 1000 * i, device=dev)
        o = torch.empty(B, T, H, dv, dtype=torch.bfloat16, device=dev)
        S = torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev)
        steps.append(lambda ex=ex, o=o, S=S: glinattn_prefill(ex["q"], ex["k"], ex["v"], ex["alpha"], None, None,
                                                              variant=GLA, o=o, S_T=S))
    pre_ms, pre_per = timed_steps(cycling(steps), max(3, min(args.steps, 10)), 2, dist, dev)
    N, P = 256, 512
    dx = inputs.ssd_decode(N, H, G, P, seed=rank, device=dev)
    od = torch.empty(N, H, dv, dtype=torch.bfloat16, device=dev)

    def step_dec():
        glinattn_decode(dx["q"], dx["k"], dx["v"], dx["alpha"], None, dx["pool"], dx["slot_ids"], variant=GLA,
                        o=od)

    dec_ms, dec_per = timed_steps(step_dec, max(10, args.steps), 3, dist, dev)
    dec_bytes = N * H * dk * dv * 4 * 2
    hbm = pk["hbm_gbs"]
    return {"config": "SSD form as gated linear attention: B=2 T=4096, 32 heads of head dim 64, state size 128, "
                      "one shared q / k group, bf16; decode 256 requests x 32 heads, 512-slot fp32 pool",
            "prefill_tokens_per_s": B * T / (pre_ms / 1e3), "prefill_ms": pre_ms,
            "prefill_roofline": {"bound": "hbm", "achieved": pre_bytes / (statistics.mean(pre_per) / 1e3) / 1e9,
                                 "peak": hbm, "unit": "GB/s",
                                 "frac": pre_bytes / (statistics.mean(pre_per) / 1e3) / 1e9 / hbm,
                                 "algorithmic_bytes": pre_bytes},
            "decode_tokens_per_s": N / (dec_ms / 1e3), "decode_ms": dec_ms,
            "decode_roofline": {"bound": "hbm", "achieved": dec_bytes / (statistics.mean(dec_per) / 1e3) / 1e9,
                                "peak": hbm, "unit": "GB/s",
                                "frac": dec_bytes / (statistics.mean(dec_per) / 1e3) / 1e9 / hbm,
                                "algorithmic_bytes": dec_bytes}}


def scan_run(args, dist, dev, rank):
    """Mamba's selective scan on B=2, T=4096, D=2048 channels (d_model 1024
    expanded twice), N=16 states, bf16 in and out; decode of 256 requests from
    a 512-slot fp32 pool."""
    import torch

    from gated_deltanet_02_gb300 import glinattn_selective_scan, glinattn_selective_scan_decode, inputs
    pk, _ = peaks()
    B, T, D, N = 2, 4096, 2048, 16
    sc_bytes = B * T * (2 * D + 2 * N) * 2 + B * T * D * 2 + B * D * N * 4 + D * N * 4
    # a step touches ~135 MB (inputs, y and the chunk end / start states the
    # workspace holds for its 64-token chunks): cycle over disjoint copies
    chunk_states = 2 * B * (T // 64) * D * N * 4
    steps = []
    for i in range(rotation(sc_bytes + chunk_states)):
        ex = inputs.selective_scan_inputs(B, T, D, N, seed=rank + 1000 * i, device=dev, dtype=torch.bfloat16)
        y = torch.empty(B, T, D, dtype=torch.bfloat16, device=dev)
        h = torch.empty(B, D, N, dtype=torch.float32, device=dev)
        ws = torch.empty(64 << 20, dtype=torch.uint8, device=dev)
        steps.append(lambda ex=ex, y=y, h=h, ws=ws: glinattn_selective_scan(ex["x"], ex["delta"], ex["Bm"], ex["Cm"],
                                                                           ex["A"], None, y=y, h_T=h, workspace=ws))
    sc_ms, sc_per = timed_steps(cycling(steps), max(3, min(args.steps, 10)), 2, dist, dev)
    R = 256
    dec_bytes = R * D * N * 4 * 2
    # a step's 256 state rows (34 MB) fit in L2: cycle over disjoint slot sets
    # of a pool holding rotation(...) x 256 slots
    nsets = rotation(dec_bytes)
    P = R * nsets
    gen = torch.Generator(device=dev)
    gen.manual_seed(rank + 7)
    dx = inputs.selective_scan_inputs(R, 1, D, N, seed=rank + 3, device=dev, dtype=torch.bfloat16)
    pool = torch.randn(P, D, N, device=dev, generator=gen) * 0.1
    slot_sets = torch.randperm(P, device=dev, generator=gen).to(torch.int32).view(nsets, R)
    xd, dd, bd, cd = (dx[k][:, 0].contiguous() for k in ("x", "delta", "Bm", "Cm"))
    yd = torch.empty(R, D, dtype=torch.bfloat16, device=dev)
    step_dec = cycling([lambda sl=sl: glinattn_selective_scan_decode(xd, dd, bd, cd, dx["A"], pool, sl, y=yd)
                        for sl in slot_sets])
    dec_ms, dec_per = timed_steps(step_dec, max(10, args.steps), 3, dist, dev)
    hbm = pk["hbm_gbs"]
    exps = B * T * D * N
    return {"config": "selective scan B=2 T=4096 D=2048 N=16, bf16 x / delta / B / C / y, fp32 A and state; "
                      f"decode 256 requests x 2048 channels x 16 states from a {P}-slot fp32 pool",
            "tokens_per_s": B * T / (sc_ms / 1e3), "ms_per_step": sc_ms,
            "roofline": {"bound": "hbm", "achieved": sc_bytes / (statistics.mean(sc_per) / 1e3) / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": sc_bytes / (statistics.mean(sc_per) / 1e3) / 1e9 / hbm,
                         "algorithmic_bytes": sc_bytes,
                         "kernels": "ssm_chunk_kernel x2 + ssm_carry_kernel"},
            "exp_per_s": 2 * exps / (statistics.mean(sc_per) / 1e3),
            "decode_tokens_per_s": R / (dec_ms / 1e3), "decode_ms": dec_ms,
            "decode_roofline": {"bound": "hbm", "achieved": dec_bytes / (statistics.mean(dec_per) / 1e3) / 1e9,
                                "peak": hbm, "unit": "GB/s",
                                "frac": dec_bytes / (statistics.mean(dec_per) / 1e3) / 1e9 / hbm,
                                "algorithmic_bytes": dec_bytes}}


def nla_run(args, dist, dev, rank):
    """Normalised kernelised linear attention (phi = elu + 1): prefill on the
    gated linear attention shape B=4 H=16 T=4096 d=128, and decode of 256
    requests x 16 heads from a 512-slot pool of states and normalisers."""
    import torch

    from gated_deltanet_02_gb300 import NLA, glinattn_decode, glinattn_prefill, inputs
    from gated_deltanet_02_gb300.glinattn import prefill_workspace_size
    pk, _ = peaks()
    B, H, T, d = 4, 16, 4096, 128
    ex = inputs.nla_prefill(B, H, T, d, seed=rank, device=dev)
    o = torch.empty(B, T, H, d, dtype=torch.bfloat16, device=dev)
    S = torch.empty(B, H, d, d, dtype=torch.float32, device=dev)
    z = torch.empty(B, H, d, dtype=torch.float32, device=dev)
    ws = torch.empty(prefill_workspace_size(B, T, H, d, variant=NLA, out_dtype=1), dtype=torch.uint8, device=dev)

    def step_prefill():
        glinattn_prefill(ex["q"], ex["k"], ex["v"], None, None, None, variant=NLA, o=o, S_T=S, z_T=z,
                         workspace=ws)

    pre_ms, pre_per = timed_steps(step_prefill, max(3, min(args.steps, 20)), 3, dist, dev)
    # q, k, v in (bf16), o out (bf16), S_T and z_T out: the layer's own bytes
    pre_bytes = B * T * H * d * 2 * 4 + B * H * (d * d + d) * 4
    N, P = 256, 512
    dx = inputs.nla_decode(N, H, d, P, seed=rank, device=dev)
    od = torch.empty(N, H, d, dtype=torch.bfloat16, device=dev)

    def step_dec():
        glinattn_decode(dx["q"], dx["k"], dx["v"], None, None, dx["pool"], dx["slot_ids"], variant=NLA,
                        z_pool=dx["zpool"], o=od)

    dec_ms, dec_per = timed_steps(step_dec, max(10, args.steps), 3, dist, dev)
    dec_bytes = N * H * (d * d + d) * 4 * 2
    hbm = pk["hbm_gbs"]
    return {"config": "normalised linear attention (phi = elu + 1, eps = 1e-6): prefill B=4 H=16 T=4096 d=128 bf16; "
                      "decode 256 requests x 16 heads, 512-slot fp32 pool of states and normalisers",
            "prefill_tokens_per_s": B * T / (pre_ms / 1e3), "prefill_ms": pre_ms,
            "prefill_roofline": {"bound": "hbm", "achieved": pre_bytes / (statistics.mean(pre_per) / 1e3) / 1e9,
                                 "peak": hbm, "unit": "GB/s",
                                 "frac": pre_bytes / (statistics.mean(pre_per) / 1e3) / 1e9 / hbm,
                                 "algorithmic_bytes": pre_bytes,
                                 "kernels": "nla_feature_kernel + gla_prefill_kernel (normalising instance, z carried in it)"},
            "decode_tokens_per_s": N / (dec_ms / 1e3), "decode_ms": dec_ms,
            "decode_roofline": {"bound": "hbm", "achieved": dec_bytes / (statistics.mean(dec_per) / 1e3) / 1e9,
                                "peak": hbm, "unit": "GB/s",
                                "frac": dec_bytes / (statistics.mean(dec_per) / 1e3) / 1e9 / hbm,
                                "algorithmic_bytes": dec_bytes}}


# ----------------------------------------------------------------------------
# the oracle on the host cores
# ----------------------------------------------------------------------------

def cpu_baseline_run(ex, budget_s=10.0):
    """Times the fp64 oracle recurrence on a bounded sample of the GLA prefill
    workload: whole sequences (T = 4096) of as many (batch, head) units as fit
    the time budget, on all host cores.  Throughput is layer tokens/s: the
    head-tokens processed divided by the H heads of a token."""
    import oracle
    cores = os.cpu_count() or 1
    q, k, v, a = (ex[n] for n in ("q", "k", "v", "alpha"))
    B, T, H, d = q.shape

    def run(nu):
        bs, hs = (nu // H, H) if nu >= H else (1, nu)
        qs, ks, vs = (x[:bs, :, :hs].double().cpu().numpy() for x in (q, k, v))
        al = a[:bs, :, :hs].double().cpu().numpy()
        t0 = time.perf_counter()
        oracle.recurrence(oracle.GLA, qs, ks, vs, al, nthreads=cores)
        return time.perf_counter() - t0, bs * hs

    dt1, nu1 = run(1)  # one (batch, head) unit: one thread
    target = int(budget_s * cores / max(dt1 / nu1, 1e-9))
    target = max(1, min(B * H, target))
    dt, nu = run(target)
    return {"value": nu * T / H / dt, "unit": "tokens/s", "cores": min(cores, nu), "kind": "oracle",
            "one_thread_value": nu1 * T / H / dt1,
            "sample": f"fp64 recurrence over {nu} of {B * H} (batch, head) units, full T={T}, "
                      f"of the GLA prefill workload ({dt:.1f} s)"}


def run_reference(args):
    """The oracle arm: rank 0 times the fp64 CPU oracle; other ranks exit."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch

    from gated_deltanet_02_gb300 import inputs
    import oracle
    cores = os.cpu_count() or 1
    c = GLA_CFG
    ex = inputs.gla_prefill(c["B"], c["H"], c["T"], c["d"], seed=0, device="cpu")
    # per step: a bounded sample of (batch, head) units of the workload
    nu = max(1, min(c["B"] * c["H"], cores))
    hs = min(nu, c["H"])
    bs = max(1, nu // c["H"])
    qs, ks, vs = (ex[n][:bs, :, :hs].double().numpy() for n in ("q", "k", "v"))
    al = ex["alpha"][:bs, :, :hs].double().numpy()
    for _ in range(args.warmup):
        oracle.recurrence(oracle.GLA, qs[:, :256], ks[:, :256], vs[:, :256], al[:, :256], nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.recurrence(oracle.GLA, qs, ks, vs, al, nthreads=cores)
    dt = (time.perf_counter() - t0) / args.steps
    # tokens/s of the whole layer: head-tokens processed / heads per token
    value = bs * hs * c["T"] / c["H"] / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "gated linear attention prefill, B=4 H=16 T=4096 d_k=d_v=128 C=64"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": min(cores, bs * hs),
                             "kind": "oracle",
                             "sample": f"{bs * hs} of {c['B'] * c['H']} (batch, head) units per step, "
                                       f"full T={c['T']}, fp64 recurrence"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_profile(args):
    """One workload alone, for a profiler: `launches` calls of the chosen hot
    kernel on the bench's own inputs, nothing timed, no JSON line."""
    import torch

    from gated_deltanet_02_gb300 import GDN, GLA, glinattn_decode, glinattn_prefill, inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.profile == "gla":
        c = GLA_CFG
        ex = inputs.gla_prefill(c["B"], c["H"], c["T"], c["d"], seed=0, device=dev)
        o = torch.empty(c["B"], c["T"], c["H"], c["d"], dtype=torch.bfloat16, device=dev)
        S = torch.empty(c["B"], c["H"], c["d"], c["d"], dtype=torch.float32, device=dev)

        def step():
            glinattn_prefill(ex["q"], ex["k"], ex["v"], ex["alpha"], None, None, variant=GLA, o=o, S_T=S)
    elif args.profile == "decode":
        dc = DEC_CFG
        dx = inputs.gdn_decode(dc["N"], dc["H"], dc["d"], dc["P"], seed=0, device=dev)
        od = torch.empty(dc["N"], dc["H"], dc["d"], dtype=torch.bfloat16, device=dev)

        def step():
            glinattn_decode(dx["q"], dx["k"], dx["v"], dx["alpha"], dx["beta"], dx["pool"], dx["slot_ids"],
                            variant=GDN, conv_w=dx["conv_w"], conv_pool=dx["conv_pool"], qk_l2norm=True,
                            o=od)
    elif args.profile in ("spec", "verify"):
        from gated_deltanet_02_gb300 import glinattn_spec_decode
        N, D, H, d = 64, 4, 32, 128
        g = torch.Generator(device=dev)
        g.manual_seed(0)
        pool = torch.randn(N * (1 + D), H, d, d, device=dev, generator=g) * 0.01
        cpool = torch.randn(N * (1 + D), 3, 3 * H * d, device=dev, generator=g).to(torch.bfloat16)
        conv_w = torch.randn(3 * H * d, 4, device=dev, generator=g) * 0.5
        src = torch.arange(N, dtype=torch.int32, device=dev)
        dst = (N + torch.arange(N * D, dtype=torch.int32, device=dev)).view(N, D)
        if args.profile == "verify":  # verify only: outputs, no per-draft states
            dst = None
        dr = inputs.spec_drafts(N, D, H, d, seed=1, device=dev)
        od = torch.empty(N, D, H, d, dtype=torch.bfloat16, device=dev)

        def step():
            glinattn_spec_decode(dr["q"], dr["k"], dr["v"], dr["alpha"], dr["beta"], pool, src, dst, variant=GDN,
                                 conv_w=conv_w, conv_pool=cpool, qk_l2norm=True, o=od)
    elif args.profile == "replay":  # the accepted drafts (0..4 per request, seeded) applied in place
        from gated_deltanet_02_gb300 import glinattn_replay
        N, D, H, d = 64, 4, 32, 128
        g = torch.Generator(device=dev)
        g.manual_seed(0)
        pool = torch.randn(N, H, d, d, device=dev, generator=g) * 0.01
        cpool = torch.randn(N, 3, 3 * H * d, device=dev, generator=g).to(torch.bfloat16)
        conv_w = torch.randn(3 * H * d, 4, device=dev, generator=g) * 0.5
        src = torch.arange(N, dtype=torch.int32, device=dev)
        dr = inputs.spec_drafts(N, D, H, d, seed=1, device=dev)
        accept = dr["accept"]

        def step():
            glinattn_replay(dr["k"], dr["v"], dr["alpha"], dr["beta"], pool, src, accept, q=dr["q"], variant=GDN,
                            conv_w=conv_w, conv_pool=cpool, qk_l2norm=True)
    elif args.profile == "ssd":
        ex = inputs.ssd_prefill(2, 32, 1, 4096, seed=0, device=dev)
        o = torch.empty(2, 4096, 32, 64, dtype=torch.bfloat16, device=dev)
        S = torch.empty(2, 32, 128, 64, dtype=torch.float32, device=dev)

        def step():
            glinattn_prefill(ex["q"], ex["k"], ex["v"], ex["alpha"], None, None, variant=GLA, o=o, S_T=S)
    elif args.profile == "nla":
        from gated_deltanet_02_gb300 import NLA
        from gated_deltanet_02_gb300.glinattn import prefill_workspace_size
        ex = inputs.nla_prefill(4, 16, 4096, 128, seed=0, device=dev)
        o = torch.empty(4, 4096, 16, 128, dtype=torch.bfloat16, device=dev)
        S = torch.empty(4, 16, 128, 128, dtype=torch.float32, device=dev)
        z = torch.empty(4, 16, 128, dtype=torch.float32, device=dev)
        ws = torch.empty(prefill_workspace_size(4, 4096, 16, 128, variant=NLA, out_dtype=1), dtype=torch.uint8,
                         device=dev)

        def step():
            glinattn_prefill(ex["q"], ex["k"], ex["v"], None, None, None, variant=NLA, o=o, S_T=S, z_T=z,
                             workspace=ws)
    elif args.profile == "scan":
        from gated_deltanet_02_gb300 import glinattn_selective_scan
        ex = inputs.selective_scan_inputs(2, 4096, 2048, 16, seed=0, device=dev, dtype=torch.bfloat16)
        y = torch.empty(2, 4096, 2048, dtype=torch.bfloat16, device=dev)
        h = torch.empty(2, 2048, 16, dtype=torch.float32, device=dev)
        ws = torch.empty(64 << 20, dtype=torch.uint8, device=dev)

        def step():
            glinattn_selective_scan(ex["x"], ex["delta"], ex["Bm"], ex["Cm"], ex["A"], None, y=y, h_T=h,
                                    workspace=ws)
    elif args.profile == "nla_decode":
        from gated_deltanet_02_gb300 import NLA
        dx = inputs.nla_decode(256, 16, 128, 512, seed=0, device=dev)
        od = torch.empty(256, 16, 128, dtype=torch.bfloat16, device=dev)

        def step():
            glinattn_decode(dx["q"], dx["k"], dx["v"], None, None, dx["pool"], dx["slot_ids"], variant=NLA,
                            z_pool=dx["zpool"], o=od)
    elif args.profile == "scan_decode":
        from gated_deltanet_02_gb300 import glinattn_selective_scan_decode
        R, D, N, P = 256, 2048, 16, 1536
        gen = torch.Generator(device=dev)
        gen.manual_seed(7)
        dx = inputs.selective_scan_inputs(R, 1, D, N, seed=3, device=dev, dtype=torch.bfloat16)
        pool = torch.randn(P, D, N, device=dev, generator=gen) * 0.1
        slots = torch.randperm(P, device=dev, generator=gen)[:R].to(torch.int32)
        xd, dd, bd, cd = (dx[k][:, 0].contiguous() for k in ("x", "delta", "Bm", "Cm"))
        yd = torch.empty(R, D, dtype=torch.bfloat16, device=dev)

        def step():
            glinattn_selective_scan_decode(xd, dd, bd, cd, dx["A"], pool, slots, y=yd)
    else:
        g = GDN_CFG
        gx = inputs.gdn_prefill(g["B"], g["H"], g["T"], g["d"], seed=0, device=dev)
        og = torch.empty(g["B"], g["T"], g["H"], g["d"], dtype=torch.bfloat16, device=dev)
        Sg = torch.empty(g["B"], g["H"], g["d"], g["d"], dtype=torch.float32, device=dev)
        from gated_deltanet_02_gb300.glinattn import prefill_workspace_size
        wsb = torch.empty(prefill_workspace_size(g["B"], g["T"], g["H"], g["d"]), dtype=torch.uint8,
                          device=dev)

        def step():
            glinattn_prefill(gx["q"], gx["k"], gx["v"], gx["alpha"], gx["beta"], gx["S0"], variant=GDN,
                             conv_w=gx["conv_w"], qk_l2norm=True, o=og, S_T=Sg, workspace=wsb)
    for _ in range(args.launches):
        step()
    torch.cuda.synchronize()
    print(f"profile {args.profile}: {args.launches} launches done")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile", choices=["gla", "decode", "gdn", "spec", "verify", "replay", "ssd", "nla", "scan",
                                          "nla_decode", "scan_decode"], default=None,
                    help="run one workload's kernel a few times for a profiler, then exit")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
