#!/usr/bin/env python3
"""Benchmark of the HYPIC linear-attention hot path on GB300.

Headline workload (one "step"): a batch of 8 independently prefilled segments
of L = 8192 tokens, 32 heads, d_k = d_v = 128, bf16 k/v with fp32 state,
scanned once with the scalar (RetNet-style fixed gamma_h) gate and once with
the diagonal (GLA-style per-channel) gate: per segment and head the
transition operator T_C and the zero-start state S(C|0).  Metric: segment
tokens per second (each family's batch counts its B x L tokens).

Extra rows in the same JSON line (own units and rooflines):
  dense_scan -- gated delta rule on a 30-layer x 32-head x 128 stack, one
                segment per layer;
  rag_chain  -- composes/s: 64 requests x 20 cached segments (Zipf(1.1) from a
                pool of 200) folded in order through 30 layers x 32 heads.

Timing: CUDA events on the launching stream, warm-up first, inputs resident
in HBM and larger than L2; ``e2e`` repeats the headline step from pinned host
buffers with the copies inside the timed region.  ``--impl reference`` times
the fp64 oracle on host cores instead (bounded sample, same metric).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

MEASURED = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0


# ------------------------------------------------------------------ helpers

def peaks():
    try:
        with open(MEASURED) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), float(m.get("bf16_tflops_sustained", m["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = [r.split(",") for r in open(self.path).read().strip().splitlines() if r.strip()]
        os.unlink(self.path)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Max of a per-rank timing over all ranks (the job's wall time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, t_max):
    """Whole-job throughput of independent replicas: units of all ranks / slowest rank's time."""
    return units_per_rank * world / t_max


def profiled_traffic(summary, source):
    """DRAM bytes per launch recorded in a committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    import hashlib
    try:
        vals = {}
        for line in open(os.path.join(ROOT, "profiles", summary)):
            if ":" in line and not line.startswith(("|", "#", " ")):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
        sha = hashlib.sha256(open(os.path.join(ROOT, source), "rb").read()).hexdigest()[:16]
        if vals.get("source_sha256_prefix") != sha:
            return None
        return float(vals["traffic_bytes_per_launch_L8192"])
    except Exception:
        return None


# ------------------------------------------------------------------ workloads

HEAD = dict(B=8, H=32, d=128)


def headline_inputs(L, seed=1):
    from linear_attention_state_gated_gb300 import workloads as wl
    return {fam: wl.scalar_diag(fam, seg_len=L, n_seg=HEAD["B"], H=HEAD["H"], d=HEAD["d"], seed=seed)
            for fam in (wl.SCALAR, wl.DIAG)}


def pinned(x, bf16=False):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x))
    if bf16:
        t = t.to(torch.bfloat16)
    return t.pin_memory()


def scan_bytes(fam, n_tok_heads, n_units, d=128, in_bytes=2):
    """Algorithmic HBM bytes of one scan launch: read k, v (and the gate) once,
    write lambda and S(C|0) (and M for dense) once per (layer, segment, head)."""
    gate = 4 * d if fam == 1 else 4
    beta = 4 if fam == 2 else 0
    per_tok = 2 * d * in_bytes + gate + beta
    per_unit = 4 * d * d + (4 * d if fam == 1 else 4) + (4 * d * d if fam == 2 else 0)
    return n_tok_heads * per_tok + n_units * per_unit


# The pages' own figures, quoted as context (HYPIC evaluation on 8x H20 nodes,
# model level; xix.ai/fr, evaluation and linear-layer paragraphs).  Not comparable
# with the kernel measurements of this bench.
PAGES_CONTEXT = {
    "mean_ttft_vs_prefix_caching": "3.25x lower (2.77-4.05x)",
    "slo_qps_vs_prefix_caching": "1.66x at a 1 s TTFT SLO (1.49-1.85x)",
    "composed_vs_recompute_difference": 6e-5,
    "state_construction_cost": "5.2-6.7 % of segment prefill (Qwen3.5-35B-A3B)",
    "hardware": "8x H20 nodes (evaluation as a whole)",
}


# ------------------------------------------------------------------ our arm

def run_headline(args, rank, world):
    import torch
    import linear_attention_state_gated_gb300 as hy

    L = args.L
    B, H, d = HEAD["B"], HEAD["H"], HEAD["d"]
    inp = headline_inputs(L, seed=1 + rank)
    dev = torch.device("cuda")
    host, devt, outs = {}, {}, {}
    for fam, w in inp.items():
        host[fam] = {"k": pinned(w["k"], True), "v": pinned(w["v"], True),
                     "alpha": pinned(w["alpha"]), "offs": pinned(w["seg_offsets"])}
        devt[fam] = {key: t.to(dev, non_blocking=False) for key, t in host[fam].items()}
        n_seg = B
        lam_shape = (1, n_seg, H, d) if fam == 1 else (1, n_seg, H)
        outs[fam] = {"lam": torch.empty(lam_shape, dtype=torch.float32, device=dev),
                     "S": torch.empty((1, n_seg, H, d, d), dtype=torch.float32, device=dev)}
    # scratch of the workspace form (the diagonal scan's balanced schedule), allocated once
    wsp = {fam: hy.segment_scan_workspace_bytes(fam, torch.bfloat16, 1, B, B * L, H, d, d) for fam in (0, 1)}
    wsb = {fam: torch.empty(n, dtype=torch.uint8, device=dev) if n > 0 else None for fam, n in wsp.items()}
    launches_per_step = sum(2 if wsp[fam] > 0 else 1 for fam in (0, 1))   # scan (+ combine)
    torch.cuda.synchronize()

    def step(events=None):
        for fam in (0, 1):
            t = devt[fam]
            if events is not None:
                events[fam][0].record()
            hy.segment_scan(fam, t["k"], t["v"], t["alpha"], t["offs"], out=outs[fam], workspace=wsb[fam])
            if events is not None:
                events[fam][1].record()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)

    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")) if world > 1 else 0)
    if rank == 0:
        clocks.start()
    per_kernel = {0: [], 1: []}
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)] for _ in range(2)]
    barrier(world)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for i in range(args.steps):
        step(events={0: ev[0][i], 1: ev[1][i]})
    stop.record()
    torch.cuda.synchronize()
    elapsed = start.elapsed_time(stop) / 1e3
    barrier(world)
    clk = clocks.stop() if rank == 0 else None
    for fam in (0, 1):
        per_kernel[fam] = [a.elapsed_time(b) / 1e3 for a, b in ev[fam]]
    t_max = max_over_ranks(elapsed, world)
    tokens_per_step = 2 * B * L
    value = job_throughput(tokens_per_step * args.steps, world, t_max)

    # end to end: pinned host inputs -> device -> scan -> host results, every step
    e2e_steps = max(3, min(args.steps, 10))
    res_host = {fam: {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                      for k, v in outs[fam].items()} for fam in (0, 1)}
    h2d = sum(t.numel() * t.element_size() for fam in (0, 1) for t in host[fam].values())
    d2h = sum(t.numel() * t.element_size() for fam in (0, 1) for t in res_host[fam].values())

    # host -> device copies spread over several streams (one copy stream does not fill
    # the host link), each family's scan waits for its own inputs only
    n_cs = 4
    cstreams = [torch.cuda.Stream() for _ in range(n_cs)]
    main = torch.cuda.current_stream()

    def e2e_step():
        ready = {}
        for fam in (0, 1):
            evs = []
            for j, key in enumerate(devt[fam]):
                src, dst = host[fam][key].view(-1), devt[fam][key].view(-1)
                parts = n_cs if dst.numel() >= (1 << 20) * n_cs else 1
                bounds = [dst.numel() * q // parts for q in range(parts + 1)]
                for q in range(parts):
                    cs = cstreams[(j + q) % n_cs]
                    cs.wait_stream(main)           # the previous step's scan has read the buffer
                    with torch.cuda.stream(cs):
                        dst[bounds[q]:bounds[q + 1]].copy_(src[bounds[q]:bounds[q + 1]], non_blocking=True)
                        ev = torch.cuda.Event()
                        ev.record(cs)
                        evs.append(ev)
            ready[fam] = evs
        for fam in (0, 1):
            for ev in ready[fam]:
                main.wait_event(ev)
            hy.segment_scan(fam, devt[fam]["k"], devt[fam]["v"], devt[fam]["alpha"],
                            devt[fam]["offs"], out=outs[fam], workspace=wsb[fam])
            for key in outs[fam]:
                res_host[fam][key].copy_(outs[fam][key], non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    # the host link on this machine: one plain pinned -> device copy of the largest input
    big_h, big_d = max(((host[f][k], devt[f][k]) for f in (0, 1) for k in host[f]), key=lambda x: x[0].numel() *
                       x[0].element_size())
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0.record()
    big_d.copy_(big_h, non_blocking=True)
    l1.record()
    torch.cuda.synchronize()
    link_gbs = big_h.numel() * big_h.element_size() / (l0.elapsed_time(l1) / 1e3) / 1e9
    barrier(world)
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record()
    for _ in range(e2e_steps):
        e2e_step()
    e2.record()
    torch.cuda.synchronize()
    e2e_t = max_over_ranks(s2.elapsed_time(e2) / 1e3, world)
    e2e_value = job_throughput(tokens_per_step * e2e_steps, world, e2e_t)

    hbm, bf16, bf16_sus, src = peaks()
    n_tok_heads = B * L * H
    kern = {}
    for fam in (0, 1):
        avg = sum(per_kernel[fam]) / len(per_kernel[fam])
        by = scan_bytes(fam, n_tok_heads, B * H, d)
        kern[fam] = dict(avg_s=avg, bytes=by, gbs=by / avg / 1e9)
    dom = max((0, 1), key=lambda f: kern[f]["avg_s"])
    return dict(value=value, elapsed=t_max, clocks=clk, kern=kern, dom=dom, launches_per_step=launches_per_step,
                e2e=dict(value=e2e_value, unit="tokens/s", h2d_bytes_per_step=h2d,
                         d2h_bytes_per_step=d2h, steps=e2e_steps,
                         h2d_gbs=round(h2d / (e2e_t / e2e_steps) / 1e9, 1),
                         link_copy_gbs=round(link_gbs, 1)),
                hbm=hbm, src=src)


# tensor work one chunk of 64 tokens of one (layer, head) chain issues, in flops
# (bf16 products, including the hi / lo splits); the algorithmic count is 180 k
# per token-head (Gram, U and W, W X and K^T Delta at C = 64)
DENSE_ALG_FLOP_PER_TOKEN_HEAD = 180e3


def dense_issued_flop_per_chunk():
    mm = lambda m, n, k: 2.0 * m * n * k   # noqa: E731
    gram = mm(128, 64, 128)                  # [K; K or Q] K^T in the preparation pass
    w = 2 * mm(128, 64, 64)                  # W^T = K^T (A diag(beta b))^T, A split hi / lo
    u = 2 * mm(128, 64, 64)                  # U^T (state half only)
    delta = 3 * mm(128, 64, 128)             # U^T - X0^T W^T, three-term split, per half
    upd = 2 * mm(128, 128, 64)               # X^T += Delta~^T K, Delta~ split, per half
    return gram + 2 * (w + delta + upd) + u


def run_dense(args, L):
    import torch
    import linear_attention_state_gated_gb300 as hy
    from linear_attention_state_gated_gb300 import workloads as wl
    Lyr, H, d = 30, 32, 128
    dev = torch.device("cuda")
    w = wl.dense_stack_device(L, n_layers=Lyr, H=H, d=d, seed=2)
    k, v, a, b = w["k"], w["v"], w["alpha"], w["beta"]
    offs = torch.tensor([0, L], dtype=torch.int64, device=dev)
    out = {"lam": torch.empty((Lyr, 1, H), dtype=torch.float32, device=dev),
           "S": torch.empty((Lyr, 1, H, d, d), dtype=torch.float32, device=dev),
           "M": torch.empty((Lyr, 1, H, d, d), dtype=torch.float32, device=dev)}
    del w
    # two passes over a workspace (the default) or the single-pass kernel
    ws = None
    if args.dense_form == "two_pass":
        ws = torch.empty(hy.segment_scan_workspace_bytes(2, torch.bfloat16, Lyr, 1, L, H, d, d),
                         dtype=torch.uint8, device=dev)
    for _ in range(2):
        hy.segment_scan(2, k, v, a, offs, beta=b, out=out, workspace=ws)
    torch.cuda.synchronize()
    reps = 3
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for s0, e0 in evs:
        s0.record()
        hy.segment_scan(2, k, v, a, offs, beta=b, out=out, workspace=ws)
        e0.record()
    torch.cuda.synchronize()
    t = sum(s0.elapsed_time(e0) for s0, e0 in evs) / reps / 1e3
    tok_heads = Lyr * L * H
    flops = tok_heads * DENSE_ALG_FLOP_PER_TOKEN_HEAD
    issued = Lyr * H * (L // 64) * dense_issued_flop_per_chunk()
    _, bf16, bf16_sus, src = peaks()
    del k, v, a, b, offs, out, ws
    torch.cuda.empty_cache()
    return {"workload": f"gated delta rule, {Lyr} layers x {H} heads x {d}, one segment of {L} tokens per layer "
                        "(inputs drawn on the device)",
            "value": L / t, "unit": "tokens/s (all 30 layers)", "head_tokens_per_s": tok_heads / t,
            "ms": t * 1e3, "form": args.dense_form,
            "roofline": {"bound": "tensor", "achieved": flops / t / 1e12, "peak": bf16,
                         "unit": "TFLOP/s", "frac": flops / t / 1e12 / bf16, "traffic": None,
                         "peak_kind": f"bf16 burst, {src}",
                         "algorithmic_flop_per_token_head": DENSE_ALG_FLOP_PER_TOKEN_HEAD,
                         "issued_tflops": issued / t / 1e12, "issued_frac": issued / t / 1e12 / bf16}}


def run_dense_rows(args):
    rows = {str(L): run_dense(args, L) for L in args.dense_lengths}
    if args.dense_form == "two_pass":
        rows["varlen"] = run_dense_varlen(args)
    return rows


def run_dense_varlen(args):
    """A varlen batch: 16 segments, lengths U{1024..4096} (seeded), gated delta rule,
    2 layers x 32 heads x 128 (1024 chains: the ragged tail is visible), one call
    (the two-pass form)."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    from linear_attention_state_gated_gb300 import workloads as wl
    Lyr, H, d = 2, 32, 128
    lens = [int(x) for x in np.random.default_rng(12).integers(1024, 4097, size=16)]
    w = wl.dense_stack(lengths=lens, n_layers=Lyr, H=H, d=d, seed=12)
    dev = torch.device("cuda")
    k = torch.from_numpy(w["k"]).to(torch.bfloat16).to(dev)
    v = torch.from_numpy(w["v"]).to(torch.bfloat16).to(dev)
    a = torch.from_numpy(w["alpha"]).to(dev)
    b = torch.from_numpy(w["beta"]).to(dev)
    offs = torch.from_numpy(w["seg_offsets"]).to(dev)
    N = int(w["seg_offsets"][-1])
    del w
    ws = torch.empty(hy.segment_scan_workspace_bytes(2, torch.bfloat16, Lyr, len(lens), N, H, d, d),
                     dtype=torch.uint8, device=dev)
    out = hy.segment_scan(2, k, v, a, offs, beta=b, workspace=ws)
    hy.segment_scan(2, k, v, a, offs, beta=b, out=out, workspace=ws)
    torch.cuda.synchronize()
    reps = 3
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        hy.segment_scan(2, k, v, a, offs, beta=b, out=out, workspace=ws)
    e.record()
    torch.cuda.synchronize()
    t = s.elapsed_time(e) / reps / 1e3
    return {"segments": len(lens), "layers": Lyr, "tokens": N, "ms": t * 1e3, "tokens_per_s": N / t}




# KDA-style gates, chunked form: per chunk of 64 tokens the pair (T_c, S_c) --
# the Gram [Ck'; Ek'] Aq^T (128 x 64 x 128), P (128 x 64 x 64), P Ka (128 x 128 x 64),
# P Le (128 x 64 x 64), Q V (128 x 128 x 64) -- then its composition into the
# segment's pair (M_c S and M_c M_acc, 128 x 128 x 128 each): flops per token-head
KDA_ALG_FLOP_PER_TOKEN_HEAD = (2.0 * (128 * 64 * 128 + 128 * 64 * 64 + 128 * 128 * 64 + 128 * 64 * 64
                                      + 128 * 128 * 64) + 2 * 2.0 * 128 ** 3) / 64


def kda_issued_flop_per_chunk():
    mm = lambda m, n, k: 2.0 * m * n * k   # noqa: E731
    pair = 3 * (mm(128, 64, 128) + mm(128, 64, 64) + mm(128, 128, 64) + mm(128, 64, 64)) + 2 * mm(128, 128, 64)
    chains = 2 * 3 * mm(128, 128, 128)     # state and operator chains, three-term splits
    return pair + chains


def run_kda(args, L):
    """KDA-style gates (a gate per channel inside the erasing update), 30 layers x
    32 heads x 128, one segment of L tokens per layer: every chunk's pair on the
    tensor cores, then the per-segment chains of the composed-prefix kernels."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    from linear_attention_state_gated_gb300 import workloads as wl
    Lyr, H, d = args.kda_layers, 32, 128
    w = wl.kda_stack(seg_len=L, n_layers=Lyr, H=H, d=d)
    dev = torch.device("cuda")
    k = torch.from_numpy(w["k"]).to(torch.bfloat16).to(dev)
    v = torch.from_numpy(w["v"]).to(torch.bfloat16).to(dev)
    a = torch.from_numpy(w["alpha"]).to(dev)
    b = torch.from_numpy(w["beta"]).to(dev)
    offs = torch.from_numpy(w["seg_offsets"]).to(dev)
    out = {"lam": torch.empty((Lyr, 1, H), dtype=torch.float32, device=dev),
           "S": torch.empty((Lyr, 1, H, d, d), dtype=torch.float32, device=dev),
           "M": torch.empty((Lyr, 1, H, d, d), dtype=torch.float32, device=dev)}
    del w
    ws = torch.empty(hy.segment_scan_workspace_bytes(hy.KDA, torch.bfloat16, Lyr, 1, L, H, d, d),
                     dtype=torch.uint8, device=dev)
    for _ in range(2):
        hy.segment_scan(hy.KDA, k, v, a, offs, beta=b, out=out, workspace=ws)
    torch.cuda.synchronize()
    reps = 3
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        hy.segment_scan(hy.KDA, k, v, a, offs, beta=b, out=out, workspace=ws)
    e.record()
    torch.cuda.synchronize()
    t = s.elapsed_time(e) / reps / 1e3
    tok_heads = Lyr * L * H
    flops = tok_heads * KDA_ALG_FLOP_PER_TOKEN_HEAD
    issued = Lyr * H * (L // 64) * kda_issued_flop_per_chunk()
    _, bf16, _, src = peaks()
    del k, v, a, b, offs, out, ws
    torch.cuda.empty_cache()
    return {"workload": f"KDA-style gates, {Lyr} layers x {H} heads x {d}, one segment of {L} tokens per layer",
            "value": L / t, "unit": f"tokens/s (all {Lyr} layers)", "head_tokens_per_s": tok_heads / t,
            "ms": t * 1e3,
            "kernel": "chunk pairs on tcgen05 (scan_kda_chunk_kernel), then the composed-prefix chains",
            "roofline": {"bound": "tensor", "achieved": flops / t / 1e12, "peak": bf16, "unit": "TFLOP/s",
                         "frac": flops / t / 1e12 / bf16, "traffic": None, "peak_kind": f"bf16 burst, {src}",
                         "algorithmic_flop_per_token_head": KDA_ALG_FLOP_PER_TOKEN_HEAD,
                         "issued_tflops": issued / t / 1e12, "issued_frac": issued / t / 1e12 / bf16},
            "token_by_token_equivalent": {"flop_per_token_head": 12 * d * d,
                                          "tflops": tok_heads * 12 * d * d / t / 1e12,
                                          "note": "the recurrence's own count (12 d^2) against the same time"}}


def run_compose(args):
    """One composition step S = T S_prev + S_C (hypic_compose) over 64 requests x
    30 layers = 1920 items x 32 heads x 128 x 128, per family; synthetic fp32
    states drawn on the device (values do not change the work)."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    res = {}
    hbm, _, _, src = peaks()
    n, H, d = args.compose_n, 32, 128
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    S_prev = torch.randn((n, H, d, d), generator=g, device=dev)
    S_C = torch.randn((n, H, d, d), generator=g, device=dev)
    S_out = torch.empty_like(S_prev)
    for fam, name in ((0, "scalar"), (1, "diag"), (2, "dense")):
        lam = -torch.rand((n, H, d) if fam == 1 else (n, H), generator=g, device=dev) * 50
        M = torch.randn((n, H, d, d), generator=g, device=dev) * 0.1 if fam == 2 else None
        for _ in range(3):
            hy.compose(fam, lam, S_C, S_prev=S_prev, M=M, S_out=S_out)
        torch.cuda.synchronize()
        reps = 5
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            hy.compose(fam, lam, S_C, S_prev=S_prev, M=M, S_out=S_out)
        e.record()
        torch.cuda.synchronize()
        t = s.elapsed_time(e) / reps / 1e3
        by = n * H * (3 * 4 * d * d + (4 * d if fam == 1 else 4) + (4 * d * d if fam == 2 else 0))
        res[name] = {"value": n / t, "unit": "composes/s (all 32 heads)", "ms": t * 1e3, "items": n,
                     "roofline": {"bound": "hbm", "achieved": by / t / 1e9, "peak": hbm, "unit": "GB/s",
                                  "frac": by / t / 1e9 / hbm, "traffic": None, "peak_kind": f"copy, {src}"}}
        del M, lam
    del S_prev, S_C, S_out
    torch.cuda.empty_cache()
    return res


def run_seam(args):
    """Reuse with a seam window (hypic_seam_compose): per item, the first 8 tokens
    of a reused segment advance the running state from S_prev (emitting their
    outputs), then the cached rest of the segment is composed; 1920 items x 32
    heads x 128 x 128 per family, inputs drawn on the device (values do not change
    the work)."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    res = {}
    hbm, _, _, src = peaks()
    n, w, H, d = args.compose_n, 8, 32, 128
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(6)
    f = dict(device=dev, generator=g)
    k = torch.nn.functional.normalize(torch.randn((n, w, H, d), **f), dim=-1).to(torch.bfloat16)
    q = torch.randn((n, w, H, d), **f).to(torch.bfloat16)
    v = torch.randn((n, w, H, d), **f).to(torch.bfloat16)
    beta = torch.sigmoid(torch.randn((n, w, H), **f))
    S_prev = torch.randn((n, H, d, d), **f)
    S_C = torch.randn((n, H, d, d), **f)
    S_out = torch.empty_like(S_prev)
    o = torch.empty((n, w, H, d), dtype=torch.bfloat16, device=dev)
    for fam, name in ((0, "scalar"), (1, "diag"), (2, "dense")):
        alpha = 0.85 + 0.15 * torch.rand((n, w, H, d) if fam == 1 else (n, w, H), **f)
        lam = -torch.rand((n, H, d) if fam == 1 else (n, H), **f) * 5
        M = torch.randn((n, H, d, d), **f) * 0.1 if fam == 2 else None
        call = lambda: hy.seam_compose(fam, k, v, alpha, lam, S_C, S_prev=S_prev, M=M, beta=beta, q=q,
                                       want_o=True, S_out=S_out, o_out=o)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        reps = 5
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            call()
        e.record()
        torch.cuda.synchronize()
        t = s.elapsed_time(e) / reps / 1e3
        # states in and out (S_prev, S_C, S_out; M for dense), lambda, the window's
        # q, k, v (bf16), alpha, beta and outputs
        per_head = 3 * 4 * d * d + (4 * d * d if fam == 2 else 0) + (4 * d if fam == 1 else 4) + \
            w * (3 * 2 * d + (4 * d if fam == 1 else 4) + 4 + 2 * d)
        by = n * H * per_head
        res[name] = {"value": n / t, "unit": "seam composes/s (all 32 heads, w = 8)", "ms": t * 1e3,
                     "items": n, "window": w,
                     "roofline": {"bound": "hbm", "achieved": by / t / 1e9, "peak": hbm, "unit": "GB/s",
                                  "frac": by / t / 1e9 / hbm, "traffic": None, "peak_kind": f"copy, {src}"}}
        del alpha, lam, M
    del k, q, v, beta, S_prev, S_C, S_out, o
    torch.cuda.empty_cache()
    return res


def run_prefix(args):
    """Composed prefix (hypic_compose_prefix): the cached pair of a whole 64-segment
    prompt, 64 pool entries in order, 30 layers x 32 heads x 128 x 128, per family;
    synthetic pool drawn on the device (values do not change the work)."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    res = {}
    hbm, _, _, src = peaks()
    P, Lyr, H, d = 64, 30, 32, 128
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    clen = torch.tensor([P], dtype=torch.int32, device=dev)
    idx = torch.arange(P, dtype=torch.int32, device=dev)[None]
    pool_S = torch.randn((P, Lyr, H, d, d), generator=g, device=dev)
    for fam, name in ((0, "scalar"), (1, "diag"), (2, "dense")):
        lam = -torch.rand((P, Lyr, H, d) if fam == 1 else (P, Lyr, H), generator=g, device=dev) * 5
        M = torch.randn((P, Lyr, H, d, d), generator=g, device=dev) * 0.1 if fam == 2 else None
        out = {}
        call = lambda: hy.compose_prefix(fam, clen, idx, lam, pool_S, pool_M=M, out=out)   # noqa: E731
        out = call()
        for _ in range(2):
            call()
        torch.cuda.synchronize()
        reps = 3
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            call()
        e.record()
        torch.cuda.synchronize()
        t = s.elapsed_time(e) / reps / 1e3
        # each entry's S_p (and M_p) once, lambda, and the outputs (S, M) once per (layer, head)
        per_entry = 4 * d * d + (4 * d * d if fam == 2 else 0) + (4 * d if fam == 1 else 4)
        by = Lyr * H * (P * per_entry + 4 * d * d + (4 * d * d if fam == 2 else 0))
        res[name] = {"value": P * Lyr / t, "unit": "composes/s folded into the prefix (all 32 heads)",
                     "ms": t * 1e3, "entries": P, "layers": Lyr,
                     "roofline": {"bound": "hbm", "achieved": by / t / 1e9, "peak": hbm, "unit": "GB/s",
                                  "frac": by / t / 1e9 / hbm, "traffic": None, "peak_kind": f"copy, {src}"}}
        del lam, M, out
    del pool_S
    torch.cuda.empty_cache()
    return res


def scan_rag_pool(fam, n_layers, H=32, d=128, P=200, timed=None):
    """The RAG pool: P segments of U{1024..4096} tokens under the scalar/diagonal
    law, drawn on the device layer by layer and scanned (hypic_segment_scan with
    a workspace) into pool tensors lam [P, Lyr, H(, d)] and S [P, Lyr, H, d, d].
    ``timed`` (a list) collects each layer's scan time in seconds."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    from linear_attention_state_gated_gb300 import workloads as wl
    dev = torch.device("cuda")
    lens = wl.rag_pool_lengths(P)
    lam_shape = (P, n_layers, H, d) if fam == 1 else (P, n_layers, H)
    pool_lam = torch.empty(lam_shape, dtype=torch.float32, device=dev)
    pool_S = torch.empty((P, n_layers, H, d, d), dtype=torch.float32, device=dev)
    N = int(lens.sum())
    need = hy.segment_scan_workspace_bytes(fam, torch.bfloat16, 1, P, N, H, d, d)
    ws = torch.empty(need, dtype=torch.uint8, device=dev) if need > 0 else None
    for l in range(n_layers):
        k, v, a, offs = wl.scalar_diag_layer_device(fam, lens, l, H=H, d=d)
        offs = torch.from_numpy(offs).to(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        out = hy.segment_scan(fam, k, v, a, offs, workspace=ws)
        e1.record()
        pool_lam[:, l].copy_(out["lam"][0])
        pool_S[:, l].copy_(out["S"][0])
        if timed is not None:
            torch.cuda.synchronize()
            timed.append(e0.elapsed_time(e1) / 1e3)
        del k, v, a, out
    torch.cuda.synchronize()
    return lens, pool_lam, pool_S


def run_chain(args):
    """RAG-style composition: 64 requests x 20 distinct pool entries (Zipf(1.1), in
    draw order) folded through all layers, over a pool of 200 segments scanned on
    the device (lengths U{1024..4096}, scalar / diagonal law)."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    from linear_attention_state_gated_gb300 import workloads as wl
    res = {}
    hbm, _, _, src = peaks()
    clen, idx = wl.rag_requests()
    dev = torch.device("cuda")
    cl, ix = torch.from_numpy(clen).to(dev), torch.from_numpy(idx).to(dev)
    Lyr = args.chain_layers
    for fam, name in ((0, "scalar"), (1, "diag")):
        scan_t = []
        lens, pl, pS = scan_rag_pool(fam, Lyr, timed=scan_t)
        R, H, d = 64, 32, 128
        out = torch.empty((R, Lyr, H, d, d), dtype=torch.float32, device=dev)
        for _ in range(3):
            hy.compose_chain(fam, cl, ix, pl, pS, S_out=out)
        torch.cuda.synchronize()
        reps = 5
        s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(reps):
            hy.compose_chain(fam, cl, ix, pl, pS, S_out=out)
        e0.record()
        torch.cuda.synchronize()
        t = s0.elapsed_time(e0) / reps / 1e3
        n_steps = int(clen.sum())
        composes = n_steps * Lyr                       # (request, segment, layer) triples
        lam_b = 4 * d if fam == 1 else 4
        by = n_steps * Lyr * H * (4 * d * d + lam_b) + R * Lyr * H * 4 * d * d
        pool_tok = int(lens.sum())
        res[name] = {"value": composes / t, "unit": "composes/s (all 32 heads)", "ms": t * 1e3,
                     "layers": Lyr,
                     "pool": {"segments": len(lens), "tokens": pool_tok, "layers": Lyr,
                              "scan_ms_per_layer": 1e3 * sum(scan_t) / len(scan_t),
                              "scan_tokens_per_s": pool_tok * Lyr / sum(scan_t),
                              "note": "pool segments drawn on the device and scanned (untimed set-up of the chain)"},
                     "roofline": {"bound": "hbm", "achieved": by / t / 1e9, "peak": hbm,
                                  "unit": "GB/s", "frac": by / t / 1e9 / hbm, "traffic": None,
                                  "peak_kind": f"copy, {src}"}}
        del pl, pS, out
        torch.cuda.empty_cache()
    return res


def run_scan_sd_o(args, L=2048):
    """Scalar and diagonal scans with the per-token outputs o_t = S_t^T q_t: 8 segments
    x L tokens x 32 heads, bf16 q/k/v/o, each family timed alone."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    from linear_attention_state_gated_gb300 import workloads as wl
    B, H, d = HEAD["B"], HEAD["H"], HEAD["d"]
    hbm, _, _, src = peaks()
    dev = torch.device("cuda")
    res = {"workload": f"scalar / diagonal scan with o_t, batch {B} x {L} tokens, {H} heads, d_k=d_v={d}"}
    for fam in (0, 1):
        w = wl.scalar_diag(fam, seg_len=L, n_seg=B, H=H, d=d, seed=1, with_q=True)
        k = torch.from_numpy(w["k"]).to(torch.bfloat16).to(dev)
        v = torch.from_numpy(w["v"]).to(torch.bfloat16).to(dev)
        q = torch.from_numpy(w["q"]).to(torch.bfloat16).to(dev)
        a = torch.from_numpy(w["alpha"]).to(dev)
        offs = torch.from_numpy(w["seg_offsets"]).to(dev)
        out = hy.segment_scan(fam, k, v, a, offs, q=q, want_o=True)
        torch.cuda.synchronize()
        reps = 5
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            hy.segment_scan(fam, k, v, a, offs, q=q, want_o=True, out=out)
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / reps / 1e3
        by = scan_bytes(fam, B * L * H, B * H, d) + B * L * H * d * 2 * 2   # + q read, o written
        res[{0: "scalar", 1: "diag"}[fam]] = {
            "tokens_per_s": B * L / t, "ms": t * 1e3,
            "roofline": {"bound": "hbm", "achieved": by / t / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": by / t / 1e9 / hbm, "peak_kind": f"HBM copy, {src}"}}
        del k, v, q, a, offs, out
    return res


def run_tree(args):
    """Few units, long chains: 1 layer x 4 heads, one request folding 64 pool entries
    in order, per family; the plain chain (one CTA per (request, layer, head)) against
    the two-level tree of hypic_compose_chain_ws.  Pool pairs drawn on the device
    (decaying operators); the 16-32 MB pool stays in L2 between launches."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    P, Lyr, H, d, n = 64, 1, 4, 128, 64
    res = {"workload": f"1 request x {Lyr} layer x {H} heads x d={d}, chains of {n} pool entries"}
    clen = torch.tensor([n], dtype=torch.int32, device=dev)
    idx = torch.arange(n, dtype=torch.int32, device=dev)[None]
    for fam, name in ((0, "scalar"), (1, "diag"), (2, "dense")):
        lam = -0.05 * torch.rand((P, Lyr, H, d) if fam == 1 else (P, Lyr, H), generator=g, device=dev)
        S = torch.randn((P, Lyr, H, d, d), generator=g, device=dev)
        M = None
        if fam == 2:
            M = torch.randn((P, Lyr, H, d, d), generator=g, device=dev) / d ** 0.5
            M = M / M.abs().amax(dim=(-2, -1), keepdim=True)
        ws = torch.empty(max(1, hy.compose_chain_workspace_bytes(fam, 1, Lyr, H, d, d, n)), dtype=torch.uint8,
                         device=dev)
        out = torch.empty((1, Lyr, H, d, d), device=dev)
        times = {}
        for mode in ("chain", "tree"):
            kw = {"workspace": ws} if mode == "tree" else {}
            for _ in range(3):
                hy.compose_chain(fam, clen, idx, lam, S, pool_M=M, S_out=out, **kw)
            torch.cuda.synchronize()
            reps = 20
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                hy.compose_chain(fam, clen, idx, lam, S, pool_M=M, S_out=out, **kw)
            e1.record()
            torch.cuda.synchronize()
            times[mode] = e0.elapsed_time(e1) / reps
        res[name] = {"chain_ms": times["chain"], "tree_ms": times["tree"], "speedup": times["chain"] / times["tree"],
                     "composes_per_s_tree": n * Lyr / (times["tree"] / 1e3)}
    return res


def run_scan_sd(args, L):
    """Scalar and diagonal scans of 8 segments x L tokens x 32 heads (the headline's
    kernels at a shorter length), each family timed alone."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    B, H, d = HEAD["B"], HEAD["H"], HEAD["d"]
    hbm, _, _, src = peaks()
    dev = torch.device("cuda")
    res = {}
    for fam, w in headline_inputs(L, seed=1).items():
        k = torch.from_numpy(w["k"]).to(torch.bfloat16).to(dev)
        v = torch.from_numpy(w["v"]).to(torch.bfloat16).to(dev)
        a = torch.from_numpy(w["alpha"]).to(dev)
        offs = torch.from_numpy(w["seg_offsets"]).to(dev)
        need = hy.segment_scan_workspace_bytes(fam, torch.bfloat16, 1, B, B * L, H, d, d)
        ws = torch.empty(need, dtype=torch.uint8, device=dev) if need > 0 else None
        out = hy.segment_scan(fam, k, v, a, offs, workspace=ws)
        torch.cuda.synchronize()
        reps = 20
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for s0, e0 in evs:
            s0.record()
            hy.segment_scan(fam, k, v, a, offs, out=out, workspace=ws)
            e0.record()
        torch.cuda.synchronize()
        t = sum(s0.elapsed_time(e0) for s0, e0 in evs) / reps / 1e3
        by = scan_bytes(fam, B * L * H, B * H, d)
        res[{0: "scalar", 1: "diag"}[fam]] = {
            "tokens_per_s": B * L / t, "ms": t * 1e3,
            "roofline": {"bound": "hbm", "achieved": by / t / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": by / t / 1e9 / hbm, "peak_kind": f"HBM copy, {src}",
                         "l2": "inputs below 129 MB stay in L2 between launches" if by < 129e6 else "inputs exceed L2"}}
        del k, v, a, offs, ws, out
    return {"workload": f"scalar / diagonal scan, batch {B} x {L} tokens, {H} heads, d_k=d_v={d}", **res}


def run_long_mix(args):
    """131072-token prompt = 64 x 2048-token segments, gated delta rule, 30 layers
    x 32 heads: 48 cached segments (scanned before the timed region), then per
    step: scan the 16 uncached segments in parallel with o_t (one call: every
    (layer, uncached segment) a segment of one token array) and fold all 64 pairs
    in prompt order (one chain per (layer, head); the layers are the chain's
    requests over a pool with the layout of ``workloads.long_mix_layout``)."""
    import torch
    import linear_attention_state_gated_gb300 as hy
    from linear_attention_state_gated_gb300 import workloads as wl
    n_seg, L, Lyr, H, d = 64, 2048, args.mix_layers, 32, 128
    unc, cached, rows = wl.long_mix_layout(n_seg=n_seg, n_layers=Lyr)
    nu = len(unc)
    dev = torch.device("cuda")
    P = Lyr * n_seg
    pool_lam = torch.empty((P, 1, H), dtype=torch.float32, device=dev)
    pool_M = torch.empty((P, 1, H, d, d), dtype=torch.float32, device=dev)
    pool_S = torch.empty((P, 1, H, d, d), dtype=torch.float32, device=dev)
    offs1 = torch.tensor([0, L], dtype=torch.int64, device=dev)
    for c, s_ in enumerate(cached):   # the cached pairs (untimed): one scan call per segment
        w = wl.long_mix_segment_device(s_, seg_len=L, n_layers=Lyr, H=H, d=d, with_q=False)
        r0 = Lyr * nu + c * Lyr
        out = {"lam": pool_lam[r0:r0 + Lyr].view(Lyr, 1, H), "M": pool_M[r0:r0 + Lyr].view(Lyr, 1, H, d, d),
               "S": pool_S[r0:r0 + Lyr].view(Lyr, 1, H, d, d)}
        hy.segment_scan(2, w["k"], w["v"], w["alpha"], offs1, beta=w["beta"], out=out)
        del w
    flat, offs_np = wl.long_mix_uncached_flat(unc, seg_len=L, n_layers=Lyr, H=H, d=d)
    offs = torch.from_numpy(offs_np).to(dev)
    o = torch.empty((1, Lyr * nu * L, H, d), dtype=torch.bfloat16, device=dev)
    out_u = {"lam": pool_lam[:Lyr * nu].view(1, Lyr * nu, H), "M": pool_M[:Lyr * nu].view(1, Lyr * nu, H, d, d),
             "S": pool_S[:Lyr * nu].view(1, Lyr * nu, H, d, d), "o": o}
    ws = torch.empty(hy.segment_scan_workspace_bytes(2, torch.bfloat16, 1, Lyr * nu, Lyr * nu * L, H, d, d, True),
                     dtype=torch.uint8, device=dev)
    clen = torch.full((Lyr,), n_seg, dtype=torch.int32, device=dev)
    idx = torch.from_numpy(rows).to(dev)
    S_fin = torch.empty((Lyr, 1, H, d, d), dtype=torch.float32, device=dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record()
        hy.segment_scan(2, flat["k"], flat["v"], flat["alpha"], offs, beta=flat["beta"], q=flat["q"],
                        want_o=True, out=out_u, workspace=ws)
        if ev is not None:
            ev[1].record()
        hy.compose_chain(2, clen, idx, pool_lam, pool_S, pool_M=pool_M, S_out=S_fin)
        if ev is not None:
            ev[2].record()

    step()
    torch.cuda.synchronize()
    reps = 2
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
    for e in evs:
        step(e)
    torch.cuda.synchronize()
    t_scan = sum(e[0].elapsed_time(e[1]) for e in evs) / reps / 1e3
    t_chain = sum(e[1].elapsed_time(e[2]) for e in evs) / reps / 1e3
    t = t_scan + t_chain
    # state-only scan of one uncached segment (the tensor-core path) for reference
    w = wl.long_mix_segment_device(unc[0], seg_len=L, n_layers=Lyr, H=H, d=d, with_q=False)
    tmp = {"lam": torch.empty((Lyr, 1, H), device=dev), "M": torch.empty((Lyr, 1, H, d, d), device=dev),
           "S": torch.empty((Lyr, 1, H, d, d), device=dev)}
    hy.segment_scan(2, w["k"], w["v"], w["alpha"], offs1, beta=w["beta"], out=tmp)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    hy.segment_scan(2, w["k"], w["v"], w["alpha"], offs1, beta=w["beta"], out=tmp)
    e1.record()
    torch.cuda.synchronize()
    t_state_only = e0.elapsed_time(e1) / 1e3
    hbm, _, _, src = peaks()
    chain_bytes = n_seg * Lyr * H * (2 * 4 * d * d + 4) + Lyr * H * 4 * d * d
    res = {"workload": "131072-token prompt, 64 x 2048-token segments (48 cached, 16 uncached), gated delta "
                       f"rule, {Lyr} layers x 32 heads x 128",
           "value": n_seg * L / t, "unit": "prompt tokens/s", "ms": t * 1e3,
           "scan_uncached_with_o_ms": t_scan * 1e3, "chain_ms": t_chain * 1e3,
           "uncached_scan": f"one call, 16 x {Lyr} (layer, segment) units of 2048 tokens",
           "composes_per_s": n_seg * Lyr / t_chain,
           "scan_state_only_one_segment_ms": t_state_only * 1e3,
           "chain_roofline": {"bound": "hbm", "achieved": chain_bytes / t_chain / 1e9, "peak": hbm,
                              "unit": "GB/s", "frac": chain_bytes / t_chain / 1e9 / hbm,
                              "peak_kind": f"copy, {src}"}}
    del flat, pool_M, pool_S, o, w, ws
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------ oracle (CPU)

_SAMPLE_CACHE = {}


def oracle_sample_rate(L, families=(0, 1), seg_tokens=None, heads=None):
    """Time the fp64 oracle on the headline workload: by default the whole
    workload (every segment, every head, both gates), else every segment's
    first `seg_tokens` tokens for a subset of heads.  Head groups of 8 are
    scanned one call at a time to bound host memory.  Returns (tokens/s in the
    headline unit, seconds, threads, description)."""
    import oracle
    if L not in _SAMPLE_CACHE:
        _SAMPLE_CACHE[L] = headline_inputs(L, seed=1)
    inp = _SAMPLE_CACHE[L]
    hs = list(range(HEAD["H"])) if heads is None else list(heads)
    tok_heads = 0
    t_total = 0.0
    for fam in families:
        w = inp[fam]
        offs = w["seg_offsets"]
        n = seg_tokens or int(offs[1] - offs[0])
        idx = np.concatenate([np.arange(offs[s], offs[s] + n) for s in range(len(offs) - 1)])
        so = np.arange(len(offs), dtype=np.int64) * n
        for g0 in range(0, len(hs), 8):
            hg = hs[g0:g0 + 8]
            k = np.ascontiguousarray(w["k"][:, idx][:, :, hg])
            v = np.ascontiguousarray(w["v"][:, idx][:, :, hg])
            a = np.ascontiguousarray(w["alpha"][:, idx][:, :, hg])
            t0 = time.perf_counter()
            oracle.segment_scan(fam, k, v, a, so)
            t_total += time.perf_counter() - t0
            tok_heads += len(idx) * len(hg)
    # a token counts once all heads have passed
    rate = tok_heads / HEAD["H"] / t_total
    what = ("the whole workload" if seg_tokens is None and heads is None else
            f"first {n} tokens of each segment x {len(hs)} of {HEAD['H']} heads")
    desc = (f"fp64 oracle (token-by-token C, OpenMP over (segment, head) units), {len(families)} gates "
            f"x {HEAD['B']} segments, {what}; tokens/s = token-heads/s / {HEAD['H']}")
    return rate, t_total, oracle.max_threads(), desc


def run_reference(args, rank, world):
    if rank != 0:
        return
    rates, times = [], []
    for i in range(args.warmup + args.steps):
        rate, t, cores, desc = oracle_sample_rate(args.L, heads=range(0, HEAD["H"], 4))
        if i >= args.warmup:
            rates.append(rate)
            times.append(t)
    value = statistics.median(rates)
    line = {"impl": "reference", "metric": "segment-scan tokens/s (T_C+S_C)", "value": value,
            "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": headline_config(args.L),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def headline_config(L):
    return {"workload": (f"scalar (RetNet gamma_h) + diagonal (GLA) segment scan, batch "
                         f"{HEAD['B']} x {L} tokens, {HEAD['H']} heads, d_k=d_v={HEAD['d']}, "
                         "bf16 k/v, fp32 state"),
            "global_batch": HEAD["B"], "seq_len": L, "parallelism": "replicas",
            "l2": "inputs (>= 1 GB per step) exceed the 129 MB L2; no flush"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="hypic", choices=["hypic", "reference"])
    ap.add_argument("--L", type=int, default=8192)
    ap.add_argument("--rows", default="sd,sdo,dense,kda,compose,seam,prefix,chain,tree,mix",
                    help="extra rows: sd,sdo,dense,kda,compose,seam,prefix,chain,tree,mix or none")
    ap.add_argument("--dense-lengths", default="512,2048,8192,32768",
                    help="dense rows: segment lengths of the 30-layer stack")
    ap.add_argument("--sd-lengths", default="512,2048",
                    help="scalar / diagonal rows at lengths other than the headline's")
    ap.add_argument("--kda-L", type=int, default=2048)
    ap.add_argument("--kda-layers", type=int, default=30,
                    help="layers of the KDA row (30: the dense stack's shape; fewer for a profiling capture)")
    ap.add_argument("--dense-form", choices=["two_pass", "single"], default="two_pass",
                    help="dense row: two passes over a workspace, or the single-pass kernel")
    ap.add_argument("--compose-n", type=int, default=1920,
                    help="compose row: items (64 requests x 30 layers by default)")
    ap.add_argument("--chain-layers", type=int, default=30,
                    help="RAG chain row: layers of the pool (30 by default)")
    ap.add_argument("--mix-layers", type=int, default=30,
                    help="layers of the long-mix row (fewer for a profiling capture; 30 in the benchmark)")
    ap.add_argument("--no-cpu", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    args.dense_lengths = [int(x) for x in args.dense_lengths.split(",") if x]
    args.sd_lengths = [int(x) for x in args.sd_lengths.split(",") if x]

    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        run_reference(args, rank, world)
        return

    import torch
    import linear_attention_state_gated_gb300 as hy
    hy.library()   # raises if the CUDA library is missing: no fallback
    rank, world, local = dist_setup(args.gpus)
    h = run_headline(args, rank, world)
    rows = {}
    # the extra rows and the oracle baseline run at N = 1 only (with N GPUs every
    # GPU would wait for rank 0 meanwhile)
    solo = rank == 0 and world == 1
    if solo and "sd" in args.rows:
        rows["scan_sd"] = {str(L): run_scan_sd(args, L) for L in args.sd_lengths}
    if solo and "dense" in args.rows:
        rows["dense_scan"] = run_dense_rows(args)
    if solo and "kda" in args.rows:
        rows["kda_scan"] = run_kda(args, args.kda_L)
    if solo and "compose" in args.rows:
        rows["compose"] = run_compose(args)
    if solo and "seam" in args.rows:
        rows["seam"] = run_seam(args)
    if solo and "prefix" in args.rows:
        rows["prefix"] = run_prefix(args)
    if solo and "chain" in args.rows:
        rows["rag_chain"] = run_chain(args)
    if solo and "sdo" in args.rows:
        rows["scan_sd_o"] = run_scan_sd_o(args)
    if solo and "tree" in args.rows:
        rows["tree"] = run_tree(args)
    if solo and "mix" in args.rows:
        rows["long_mix"] = run_long_mix(args)
    if rank != 0:
        barrier(world)
        return
    cpu = None
    if solo and not args.no_cpu:
        rate, t, cores, desc = oracle_sample_rate(args.L)
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc,
               "seconds": round(t, 2)}
    kd = h["kern"][h["dom"]]
    fam_name = {0: "scalar", 1: "diag"}
    line = {
        "metric": "segment-scan tokens/s (T_C+S_C)", "value": h["value"], "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * h["elapsed"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": headline_config(args.L),
        "roofline": {"bound": "hbm", "achieved": kd["gbs"], "peak": h["hbm"], "unit": "GB/s",
                     "frac": kd["gbs"] / h["hbm"],
                     "traffic": (profiled_traffic("scan_sd_tc_diag_B8x2048_H32.md",
                                                  "linear_attention_state_gated_gb300/csrc/scan_sd_tc.cu")
                                 if h["dom"] == 1 and args.L == 8192 else None),
                     "kernel": f"segment scan, {fam_name[h['dom']]} gate",
                     "algorithmic_bytes": kd["bytes"], "avg_launch_ms": kd["avg_s"] * 1e3,
                     "peak_kind": f"HBM copy, {h['src']}"},
        "kernels": {fam_name[f]: {"avg_launch_ms": h["kern"][f]["avg_s"] * 1e3,
                                  "tokens_per_s": HEAD["B"] * args.L / h["kern"][f]["avg_s"],
                                  "GB/s": h["kern"][f]["gbs"], "frac": h["kern"][f]["gbs"] / h["hbm"],
                                  "algorithmic_bytes": h["kern"][f]["bytes"]} for f in (0, 1)},
        "pages_context": PAGES_CONTEXT,
        "cpu_baseline": cpu, "e2e": h["e2e"], "clocks": h["clocks"],
        "gpu_launches": h["launches_per_step"] * args.steps, "rows": rows,
    }
    barrier(world)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
