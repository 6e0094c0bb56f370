#!/usr/bin/env python
"""Throughput of the gated delta rule on GB300: one JSON line.

One step = the whole hot path once:
  * gdr_prefill     KDA prefill, 1 sequence x 32768 tokens, H = 32, d_k = d_v = 128, bf16 q/k/v,
                    per-channel alpha, S0 ~ N(0, 0.01), outputs and final states;
  * gdr_linear_attn the alpha = 1, no-erase pass over the same q/k/v/S0;
  * gdr_decode_step one token for each of 256 sequences x 32 heads (d = 128, bf16, per-channel
                    alpha) on fp32 states pre-filled by a 2048-token prefill.
value = prefill tokens/s (sequence tokens, all heads); decode tokens/s and the linear pass are
reported beside it.  Every input is larger than L2 (the prefill reads 1.35 GB, the decode state
is 1.07 GB), so no L2 flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the CPU oracle (fp64, all host cores) on a bounded sample of the same
prefill workload; it is a deliberately slow baseline, not a target.
"""
from __future__ import annotations

import argparse
import hashlib
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

import gdr_inputs as gi  # noqa: E402

PREFILL = "kda_b1_h32_t32768"
DECODE = "decode_n256_h32"
SMALL, GDN, VARLEN = "kda_t256_d64_f32", "gdn_b4_h16_t4096", "varlen_n64_h16"
CONFIG_WORKLOADS = (SMALL, GDN, VARLEN)
DECODE_PREFILL_LEN = 2048
SAMPLE_TOKENS = 32768  # oracle sample: tokens of each sampled head
METRIC = "gated-delta prefill tokens/s + decode tokens/s; % of TC/HBM roofline"
CSRC = os.path.join(ROOT, "gated_delta_rule_prefill_gb300", "csrc")


# ----------------------------------------------------------------------------------------------
# algorithmic counts (per launch)
# ----------------------------------------------------------------------------------------------
def prefill_bytes(T, H, d, n_seqs, channel=True, linear=False, elt=2, beta=True):
    per_tok_head = (3 * d * elt + d * elt)  # q, k, v in; out
    if not linear:
        per_tok_head += (d if channel else 1) * 4 + (4 if beta else 0)  # alpha, beta
    return T * H * per_tok_head + 2 * n_seqs * H * d * d * 4  # + S0 in, S_final out


def prefill_flops(T, H, d, C=64, linear=False):
    """Algorithmic flops (2 per multiply-add), counting only the triangle entries a chunk needs.
    Gated delta rule: W S, Q~ S, K^^T U (3 d^2), A (strict lower, (C-1)/2 d), M (lower incl. the
    diagonal, (C+1)/2 d), the solve applied to [beta K~ | beta V] ((C-1)/2 2d) and M U
    ((C+1)/2 d).  Linear attention, and gated linear attention (whose decay-weighted M has the
    same triangle as Q K^T): Q S and K^T V (2 d^2), the score triangle and its product with V
    ((C+1) d)."""
    if linear:
        return T * H * 2 * (2 * d * d + (C + 1) * d)
    f = 3 * d * d + (C - 1) / 2 * d + (C + 1) / 2 * d + (C - 1) / 2 * 2 * d + (C + 1) / 2 * d
    return T * H * 2 * f


def gated_linear_flops(T, H, d, C=64):
    """Gated linear attention: Q~ S and K^^T V (2 d^2), the decay-weighted M (lower triangle
    with the diagonal, (C+1)/2 d) and M V ((C+1)/2 d)."""
    return T * H * 2 * (2 * d * d + (C + 1) / 2 * d + (C + 1) / 2 * d)


def decode_bytes(N, H, d, elt=2):
    return N * H * (2 * d * d * 4 + 3 * d * elt + d * 4 + 4 + d * elt)


def decode_flops(N, H, d):
    return N * H * 2 * (3 * d * d + 2 * d)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        return m["hbm_gbs"], m["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# the files that hold each measured kernel's device code (the bench's KDA prefill, its gated
# variant and its gated-linear pass run the clustered kernel)
KERNEL_SOURCES = {"gated_linear_attn": ["prefill_cluster.cu", "tc_common.cuh", "umma.cuh"],
                  "prefill_output_gate": ["prefill_cluster.cu", "tc_common.cuh", "umma.cuh"],
                  "prefill_prologue": ["prefill_cluster.cu", "tc_common.cuh", "umma.cuh"],
                  "layer_prologue": ["prologue.cu", "gdr_internal.cuh"],
                  "normalized_linear_attn": ["linear_tc.cu", "tc_common.cuh", "umma.cuh"],
                  "gated_linear_decode": ["decode.cu"],
                  "normalized_linear_decode": ["decode.cu"],
                  "prefill": ["prefill_cluster.cu", "tc_common.cuh", "umma.cuh"],
                  "linear_attn": ["linear_tc.cu", "tc_common.cuh", "umma.cuh"],
                  "decode": ["decode.cu"]}


def ncu_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    if kernel not in KERNEL_SOURCES:
        return None
    with open(p) as f:
        t = json.load(f).get(kernel)
    if not t or t.get("source_digest") != source_digest(KERNEL_SOURCES[kernel]):
        return None
    return t.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------------------------
# ranks: every rank runs its own replica of the workload (independent problems, weak scaling);
# the only cross-rank traffic is this max-reduction of the timings and the barriers around them
# ----------------------------------------------------------------------------------------------
def max_over_ranks(values, device, world):
    """Element-wise maximum of per-rank float timings (no-op for one rank)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, device=device, dtype=torch.float64)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tokens_per_s(world, tokens_per_rank, seconds_max):
    """Whole-job throughput: the tokens all ranks processed over the slowest rank's time."""
    return world * tokens_per_rank / seconds_max


# ----------------------------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = None
        self.offset = 0

    def start(self):
        """Start sampling every 20 ms and return once the first sample has been written."""
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            t0 = time.time()
            while os.path.getsize(self.path) == 0 and time.time() - t0 < 5:
                time.sleep(0.01)
        except Exception:
            self.proc = None

    def begin(self):
        """Mark the start of the timed region: earlier samples are dropped (but one is kept)."""
        if self.path:
            self.offset = os.path.getsize(self.path)

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows, before = [], []
        with open(self.path) as f:
            pos = 0
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    (rows if pos >= self.offset else before).append(parts)
                pos += len(line)
        os.unlink(self.path)
        if not rows and before:  # region shorter than the sampling interval: the last sample
            rows = before[-1:]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        dev = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0]
        idx = {r[0] for r in rows}
        if dev in idx:
            rows = [r for r in rows if r[0] == dev]
        elif len(idx) > 1:
            rows = [r for r in rows if r[0] == sorted(idx)[0]]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------------------------------
# the oracle leg (CPU)
# ----------------------------------------------------------------------------------------------
def workload_config(n_ranks):
    """The `config` of the bench line (both arms): the prefill and decode workloads of a step."""
    wp, wd = gi.workload(PREFILL), gi.workload(DECODE)
    return {"workload": "%s + %s" % (PREFILL, DECODE),
            "prefill": {"n_seqs": wp.n_seqs, "T": wp.total_tokens, "H": wp.H, "d_k": wp.d_k,
                        "d_v": wp.d_v, "gate": "channel",
                        "dtype": "bf16 q/k/v, fp32 alpha/beta/state"},
            "decode": {"n_seqs": wd.n_seqs, "H": wd.H, "d": wd.d_k,
                       "state_prefill_tokens": DECODE_PREFILL_LEN},
            "l2": "no flush: every step's inputs exceed L2 (129 MB)",
            "parallelism": "replicas" if n_ranks > 1 else "1 GPU"}


def oracle_sample(cores):
    """Inputs of the bounded oracle sample: the first SAMPLE_TOKENS tokens of min(H, cores) heads of the
    prefill workload (work scales linearly in tokens and heads)."""
    wl = gi.workload(PREFILL)
    heads = list(range(min(wl.H, cores)))
    sub = gi.Workload(wl.name, wl.seed, wl.H, wl.d_k, wl.d_v, wl.dtype, wl.gate,
                      np.array([SAMPLE_TOKENS]), wl.s0)
    a = gi.gen_full(sub, heads=heads, threads=cores)
    desc = "first %d of %d tokens x %d of %d heads of %s (oracle fp64, %d threads)" % (
        SAMPLE_TOKENS, wl.total_tokens, len(heads), wl.H, wl.name, cores)
    scale = (SAMPLE_TOKENS * len(heads)) / float(wl.total_tokens * wl.H)  # fraction of the workload
    return a, desc, scale, wl


def time_oracle(a, cores):
    import oracle
    t = time.perf_counter()
    oracle.gated_delta(a["q"], a["k"], a["v"], a["alpha"], a["beta"], S0=a["S0"],
                       cu_seqlens=a["cu_seqlens"], threads=cores)
    return time.perf_counter() - t


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.build_oracle()
    cores = oracle.default_threads()
    a, desc, scale, wl = oracle_sample(cores)
    for _ in range(args.warmup):
        time_oracle(a, cores)
    ts = [time_oracle(a, cores) for _ in range(args.steps)]
    tot = sum(ts)
    value = wl.total_tokens * scale * args.steps / tot
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_config(1), sample=desc),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------------------------
# the GPU leg
# ----------------------------------------------------------------------------------------------
def run_gpu(args):
    import torch
    import torch.distributed as dist

    import gated_delta_rule_prefill_gb300 as g

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    # cpu baseline first (host work, before any heavy GPU allocation), rank 0 only
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build_oracle()
        cores = oracle.default_threads()
        a, desc, scale, wl = oracle_sample(cores)
        t = time_oracle(a, cores)
        cpu = {"value": wl.total_tokens * scale / t, "unit": "tokens/s", "cores": cores,
               "kind": "oracle", "sample": desc, "seconds": round(t, 3)}
        del a

    # ---- inputs (drawn on the device; same distributions as the parity inputs)
    wp = gi.workload(PREFILL)
    P = gi.device_full(wp, dev, seed_offset=rank)
    T, H, d = wp.total_tokens, wp.H, wp.d_k
    out = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    Sf = torch.empty_like(P["S0"])
    out_l = torch.empty_like(out)
    Sf_l = torch.empty_like(P["S0"])
    ws = torch.empty(g.gdr_prefill_workspace_size(wp.n_seqs, H, d, d), dtype=torch.uint8,
                     device=dev)

    wd = gi.workload(DECODE)
    wd_pre = gi.Workload(wd.name, wd.seed, wd.H, wd.d_k, wd.d_v, wd.dtype, wd.gate,
                         np.full(wd.n_seqs, DECODE_PREFILL_LEN, dtype=np.int64), "zeros")
    S_dec = torch.empty((wd.n_seqs, wd.H, wd.d_k, wd.d_v), dtype=torch.float32, device=dev)
    # states pre-filled by a seeded 2048-token prefill, 32 sequences at a time
    ws_d = torch.empty(g.gdr_prefill_workspace_size(32, wd.H, wd.d_k, wd.d_v), dtype=torch.uint8,
                       device=dev)
    for s0 in range(0, wd.n_seqs, 32):
        part = gi.Workload(wd.name, wd.seed + s0, wd.H, wd.d_k, wd.d_v, wd.dtype, wd.gate,
                           wd_pre.seqlens[s0:s0 + 32], "zeros")
        X = gi.device_full(part, dev, seed_offset=rank)
        g.gdr_prefill(X["q"], X["k"], X["v"], X["alpha"], X["beta"], S0=None,
                      cu_seqlens=X["cu_seqlens"], S_final=S_dec[s0:s0 + 32], workspace=ws_d)
        del X
    steps_in = gi.device_decode_steps(wd, 4, dev)
    out_d = torch.empty((wd.n_seqs, wd.H, wd.d_v), dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()

    def step(i, ev=None):
        if ev:
            ev[0].record(stream)
        g.gdr_prefill(P["q"], P["k"], P["v"], P["alpha"], P["beta"], S0=P["S0"],
                      cu_seqlens=P["cu_seqlens"], out=out, S_final=Sf, workspace=ws)
        if ev:
            ev[1].record(stream)
        g.gdr_linear_attn(P["q"], P["k"], P["v"], S0=P["S0"], cu_seqlens=P["cu_seqlens"],
                          out=out_l, S_final=Sf_l, workspace=ws)
        if ev:
            ev[2].record(stream)
        x = steps_in[i % len(steps_in)]
        g.gdr_decode_step(x["q"], x["k"], x["v"], x["alpha"], x["beta"], S_dec, out=out_d)
        if ev:
            ev[3].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler()
    clocks.start()
    torch.cuda.synchronize()
    clocks.begin()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(i, evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    # every bounded wait in the timed launches completed (a wait that gave up records a status;
    # its launch would have run ~2 s and its results would be invalid)
    checks = {"workspace": g.gdr_workspace_status(ws), "device": g.gdr_query_device_status()}
    if checks["workspace"] or checks["device"]:
        print("bench: a device-side check failed in the timed region: %s" % checks, file=sys.stderr)
    if world > 1:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    pre_ms = [e[0].elapsed_time(e[1]) for e in evs]
    lin_ms = [e[1].elapsed_time(e[2]) for e in evs]
    dec_ms = [e[2].elapsed_time(e[3]) for e in evs]
    total_ms, pre_tot, lin_tot, dec_tot = max_over_ranks(
        [total_ms, sum(pre_ms), sum(lin_ms), sum(dec_ms)], dev, world)

    # ---- gated linear attention (S <- Diag(alpha) S + k v^T) on the prefill inputs: reported
    # beside the step, timed on its own after it (not part of the step or of gpu_launches)
    out_g = torch.empty_like(out)
    Sf_g = torch.empty_like(P["S0"])

    def gla():
        g.gdr_gated_linear_attn(P["q"], P["k"], P["v"], P["alpha"], S0=P["S0"],
                                cu_seqlens=P["cu_seqlens"], out=out_g, S_final=Sf_g, workspace=ws)

    gla_steps = max(1, min(args.steps, 10))
    for _ in range(3):
        gla()
    torch.cuda.synchronize()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(gla_steps):
        gla()
    g1.record(stream)
    torch.cuda.synchronize()
    gla_ms = max_over_ranks([g0.elapsed_time(g1) / gla_steps], dev, world)[0]

    # ---- the same prefill with the KDA output gate (out = o * sigmoid(g)), also outside the step
    gen = torch.Generator(device=dev)
    gen.manual_seed(4242 + rank)
    gate_in = torch.randn(out.shape, generator=gen, device=dev).mul_(2.0).to(torch.bfloat16)

    def pre_gated():
        g.gdr_prefill_output_gate(P["q"], P["k"], P["v"], P["alpha"], P["beta"], gate_in,
                                  S0=P["S0"], cu_seqlens=P["cu_seqlens"], out=out_g,
                                  S_final=Sf_g, workspace=ws)

    for _ in range(3):
        pre_gated()
    torch.cuda.synchronize()
    g0.record(stream)
    for _ in range(gla_steps):
        pre_gated()
    g1.record(stream)
    torch.cuda.synchronize()
    og_ms = max_over_ranks([g0.elapsed_time(g1) / gla_steps], dev, world)[0]
    del gate_in

    # ---- the prefill with the layer prologue on load (raw projections in: q, k =
    # normalize(silu(.)), alpha, beta = sigmoid(.) inside the kernels), also outside the step
    R = gi.device_full(wp, dev, seed_offset=7 + rank, raw=True)

    def pre_prologue():
        g.gdr_prefill(R["q"], R["k"], P["v"], R["alpha"], R["beta"], S0=P["S0"],
                      cu_seqlens=P["cu_seqlens"], out=out_g, S_final=Sf_g, workspace=ws,
                      prologue=True)

    for _ in range(3):
        pre_prologue()
    torch.cuda.synchronize()
    g0.record(stream)
    for _ in range(gla_steps):
        pre_prologue()
    g1.record(stream)
    torch.cuda.synchronize()
    pro_ms = max_over_ranks([g0.elapsed_time(g1) / gla_steps], dev, world)[0]

    # ... and unfused: the prologue as its own pass (raw -> mapped tensors in HBM), then the
    # prefill on the mapped tensors; both kernels timed per step, the pass also on its own
    M = {kk: torch.empty_like(R[kk]) for kk in ("q", "k", "alpha", "beta")}

    def pass_only():
        g.gdr_layer_prologue(R["q"], R["k"], R["alpha"], R["beta"], q=M["q"], k=M["k"],
                             alpha=M["alpha"], beta=M["beta"])

    def pre_unfused():
        pass_only()
        g.gdr_prefill(M["q"], M["k"], P["v"], M["alpha"], M["beta"], S0=P["S0"],
                      cu_seqlens=P["cu_seqlens"], out=out_g, S_final=Sf_g, workspace=ws)

    for _ in range(3):
        pre_unfused()
    torch.cuda.synchronize()
    g0.record(stream)
    for _ in range(gla_steps):
        pre_unfused()
    g1.record(stream)
    torch.cuda.synchronize()
    unf_ms = max_over_ranks([g0.elapsed_time(g1) / gla_steps], dev, world)[0]
    g0.record(stream)
    for _ in range(gla_steps):
        pass_only()
    g1.record(stream)
    torch.cuda.synchronize()
    lp_ms = max_over_ranks([g0.elapsed_time(g1) / gla_steps], dev, world)[0]
    del R, M

    # ---- normalised phi-linear attention (phi = elu + 1, normaliser z) on the same q, k, v
    Zf = torch.empty((wp.n_seqs, H, d), dtype=torch.float32, device=dev)

    def nla():
        g.gdr_normalized_linear_attn(P["q"], P["k"], P["v"], eps=1e-6, S0=P["S0"],
                                     cu_seqlens=P["cu_seqlens"], out=out_g, S_final=Sf_g,
                                     z_final=Zf, workspace=ws)

    for _ in range(3):
        nla()
    torch.cuda.synchronize()
    g0.record(stream)
    for _ in range(gla_steps):
        nla()
    g1.record(stream)
    torch.cuda.synchronize()
    nla_ms = max_over_ranks([g0.elapsed_time(g1) / gla_steps], dev, world)[0]
    del out_g, Sf_g, Zf

    # ---- the decode steps of gated linear and normalised linear attention on the decode
    # workload's states (z: the first states' channel sums, only its magnitude matters)
    Zd = S_dec.sum(dim=3).abs_().add_(1.0)
    dec_steps = max(10, min(args.steps, 100))

    def time_dec(fn):
        for i in range(3):
            fn(steps_in[i % len(steps_in)])
        torch.cuda.synchronize()
        g0.record(stream)
        for i in range(dec_steps):
            fn(steps_in[i % len(steps_in)])
        g1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks([g0.elapsed_time(g1) / dec_steps], dev, world)[0]

    gld_ms = time_dec(lambda x: g.gdr_gated_linear_decode_step(x["q"], x["k"], x["v"], x["alpha"],
                                                                 S_dec, out=out_d))
    nld_ms = time_dec(lambda x: g.gdr_normalized_linear_decode_step(x["q"], x["k"], x["v"], S_dec,
                                                                      Zd, eps=1e-6, out=out_d))
    del Zd

    # ---- end to end through the public API with host buffers (prefill), rank-local
    host_in = {k: P[k].cpu().pin_memory() for k in ("q", "k", "v", "alpha", "beta", "S0")}
    host_cu = P["cu_seqlens"].cpu().pin_memory()
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    host_sf = torch.empty(Sf.shape, dtype=Sf.dtype).pin_memory()
    hbuf = torch.empty(g.gdr_prefill_host_buffer_size(wp.n_seqs, H, T, d, d), dtype=torch.uint8,
                       device=dev)
    e2e_steps = max(1, min(args.steps, 5))

    def e2e_step():  # one call: host inputs in, out and S_final back, copies inside the call
        g.gdr_prefill_host(host_in["q"], host_in["k"], host_in["v"], host_in["alpha"],
                           host_in["beta"], S0=host_in["S0"], cu_seqlens=host_cu, out=host_out,
                           S_final=host_sf, buffer=hbuf)

    e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / e2e_steps], dev, world)[0]
    if world > 1:
        dist.barrier()
    h2d = sum(t.numel() * t.element_size() for t in host_in.values()) + host_cu.numel() * 4
    d2h = host_out.numel() * host_out.element_size() + host_sf.numel() * host_sf.element_size()

    # ---- the other named workloads, each timed on its own (parity cases of the same path): the
    # 256-token fp32 KDA prefill (latency only), the scalar-gate prefill of 4 x 4096 tokens and
    # the packed variable-length prefill of 64 sequences with its linear-attention pass
    cfg_ms = {}
    cfg_iters = max(1, min(args.steps, 10))

    def time_fn(fn, iters=cfg_iters):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        g0.record(stream)
        for _ in range(iters):
            fn()
        g1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks([g0.elapsed_time(g1) / iters], dev, world)[0]

    cfg_wl = {}
    for name in CONFIG_WORKLOADS:
        wl = gi.workload(name)
        cfg_wl[name] = wl
        X = gi.device_full(wl, dev, seed_offset=rank)
        o = torch.empty((wl.total_tokens, wl.H, wl.d_v),
                        dtype=torch.bfloat16 if wl.dtype == "bf16" else torch.float32, device=dev)
        sf = torch.empty_like(X["S0"])
        w = torch.empty(g.gdr_prefill_workspace_size(wl.n_seqs, wl.H, wl.d_k, wl.d_v,
                                                     wl.dtype), dtype=torch.uint8, device=dev)
        cfg_ms[name] = time_fn(lambda: g.gdr_prefill(
            X["q"], X["k"], X["v"], X["alpha"], X["beta"], S0=X["S0"],
            cu_seqlens=X["cu_seqlens"], out=o, S_final=sf, workspace=w))
        if name == VARLEN:
            cfg_ms[name + " linear"] = time_fn(lambda: g.gdr_linear_attn(
                X["q"], X["k"], X["v"], S0=X["S0"], cu_seqlens=X["cu_seqlens"], out=o,
                S_final=sf, workspace=w))
        del X, o, sf, w
    torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    hbm, tc, peak_kind = peaks()
    K = args.steps
    pre_s, lin_s, dec_s = pre_tot / K / 1e3, lin_tot / K / 1e3, dec_tot / K / 1e3
    n = world
    prefill_tps = job_tokens_per_s(n, T, pre_s)
    decode_tps = job_tokens_per_s(n, wd.n_seqs, dec_s)
    linear_tps = job_tokens_per_s(n, T, lin_s)

    def roof(name, bytes_, flops, secs):
        gbs = bytes_ / secs / 1e9
        tfs = flops / secs / 1e12
        return {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                "frac": gbs / hbm, "traffic": ncu_traffic(name),
                "algorithmic_bytes": bytes_, "algorithmic_flops": flops,
                "tensor_tflops": tfs, "tensor_frac": tfs / tc,
                "launch_us": secs * 1e6, "peak_source": peak_kind + " (MEASURED_PEAKS.json)"
                if peak_kind == "measured" else "fallback"}

    kern = {
        "prefill": roof("prefill", prefill_bytes(T, H, d, wp.n_seqs), prefill_flops(T, H, d),
                        pre_s),
        "linear_attn": roof("linear_attn", prefill_bytes(T, H, d, wp.n_seqs, linear=True),
                            prefill_flops(T, H, d, linear=True), lin_s),
        "decode": roof("decode", decode_bytes(wd.n_seqs, wd.H, wd.d_k),
                       decode_flops(wd.n_seqs, wd.H, wd.d_k), dec_s),
    }
    kern_extra = {
        "gated_linear_attn": roof("gated_linear_attn",
                                  prefill_bytes(T, H, d, wp.n_seqs, beta=False),
                                  gated_linear_flops(T, H, d), gla_ms / 1e3),
        "prefill_output_gate": roof("prefill_output_gate",
                                    prefill_bytes(T, H, d, wp.n_seqs) + T * H * d * 2,
                                    prefill_flops(T, H, d), og_ms / 1e3),
        "prefill_prologue": roof("prefill_prologue", prefill_bytes(T, H, d, wp.n_seqs),
                                 prefill_flops(T, H, d), pro_ms / 1e3),
        "normalized_linear_attn": roof("normalized_linear_attn",
                                       prefill_bytes(T, H, d, wp.n_seqs, linear=True),
                                       prefill_flops(T, H, d, linear=True), nla_ms / 1e3),
        # the delta decode's bytes without beta (gated linear); without alpha and beta, with
        # z read and written (normalised linear)
        "gated_linear_decode": roof("gated_linear_decode",
                                    decode_bytes(wd.n_seqs, wd.H, wd.d_k) - wd.n_seqs * wd.H * 4,
                                    decode_flops(wd.n_seqs, wd.H, wd.d_k), gld_ms / 1e3),
        "normalized_linear_decode": roof("normalized_linear_decode",
                                         decode_bytes(wd.n_seqs, wd.H, wd.d_k) +
                                         wd.n_seqs * wd.H * (wd.d_k * 4 - 4),
                                         decode_flops(wd.n_seqs, wd.H, wd.d_k), nld_ms / 1e3),
        # read xq, xk (bf16), a (fp32 per channel), b; write q, k, alpha, beta
        "layer_prologue": roof("layer_prologue", 2 * T * H * (2 * d * 2 + d * 4 + 4), 0.0,
                               lp_ms / 1e3),
    }
    cfg = {}
    for name, wl in cfg_wl.items():
        ms = cfg_ms[name]
        ch = wl.gate == "channel"
        elt = 2 if wl.dtype == "bf16" else 4
        e = {"tokens_per_s": job_tokens_per_s(n, wl.total_tokens, ms / 1e3), "ms": ms,
             "total_tokens": int(wl.total_tokens), "n_seqs": int(wl.n_seqs), "H": wl.H,
             "d": wl.d_k, "gate": wl.gate, "dtype": wl.dtype,
             "compute_dtype": g.compute_dtype(wl.dtype, wl.d_k)}
        if name == SMALL:
            e["note"] = "latency-bound (256 tokens, one head): time only"
        else:
            e["roofline"] = roof("cfg:" + name, prefill_bytes(wl.total_tokens, wl.H, wl.d_k,
                                                               wl.n_seqs, channel=ch, elt=elt),
                                 prefill_flops(wl.total_tokens, wl.H, wl.d_k), ms / 1e3)
        cfg[name] = e
        if name == VARLEN:
            lms = cfg_ms[name + " linear"]
            cfg[name + " linear"] = {
                "tokens_per_s": job_tokens_per_s(n, wl.total_tokens, lms / 1e3), "ms": lms,
                "roofline": roof("cfg:" + name + " linear",
                                 prefill_bytes(wl.total_tokens, wl.H, wl.d_k, wl.n_seqs,
                                               linear=True, elt=elt),
                                 prefill_flops(wl.total_tokens, wl.H, wl.d_k, linear=True),
                                 lms / 1e3)}
    dominant = max(kern, key=lambda k: kern[k]["launch_us"])
    main_roof = {k: kern[dominant][k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                                 "traffic")}
    main_roof["kernel"] = dominant
    line = {
        "metric": METRIC, "value": prefill_tps, "unit": "tokens/s", "n_gpus": n, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": g.compute_dtype(wp.dtype, d),
        "data": "synthetic (seeded, drawn on the device; distributions of the workload spec)",
        "config": workload_config(n),
        "decode_tokens_per_s": decode_tps,
        "linear_attn_tokens_per_s": linear_tps,
        "gated_linear_attn_tokens_per_s": job_tokens_per_s(n, T, gla_ms / 1e3),
        "prefill_output_gate_tokens_per_s": job_tokens_per_s(n, T, og_ms / 1e3),
        "prefill_prologue_tokens_per_s": job_tokens_per_s(n, T, pro_ms / 1e3),
        "prefill_unfused_prologue_tokens_per_s": job_tokens_per_s(n, T, unf_ms / 1e3),
        "normalized_linear_attn_tokens_per_s": job_tokens_per_s(n, T, nla_ms / 1e3),
        "gated_linear_decode_tokens_per_s": job_tokens_per_s(n, wd.n_seqs, gld_ms / 1e3),
        "normalized_linear_decode_tokens_per_s": job_tokens_per_s(n, wd.n_seqs, nld_ms / 1e3),
        "roofline": main_roof,
        "kernels": kern,
        "kernels_outside_step": kern_extra,
        "configs": cfg,
        "e2e": {"value": job_tokens_per_s(n, T, e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "what": "gdr_prefill_host: pinned host inputs in, "
                "out and S_final back, copies pipelined with the kernels inside the call"},
        "gpu_launches": 6 * K,  # per step: prep + prefill, prep + linear run sums + linear runs, decode
        "clocks": clk,
        "device_checks": checks,
    }
    if cpu:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_profile(args):
    """Profiler target: `--warmup` launches each of the step's three kernels on a smaller KDA
    prefill (1 x `--profile-tokens` tokens, 32 heads, the KDA workload's distributions; the
    linear pass on the same q/k/v) and one decode step on the decode workload's shape, then exit.
    For ncu captures that must stay small; it prints no bench line."""
    import torch

    import gated_delta_rule_prefill_gb300 as g

    torch.cuda.set_device(0)
    wp = gi.custom(name="kda_profile", seed=1002, seqlens=[args.profile_tokens], H=32, d_k=128,
                   d_v=128, dtype="bf16", gate="channel", s0="normal")
    d = gi.device_full(wp, "cuda")
    wd = gi.workload(DECODE)
    x = gi.device_decode_steps(wd, 1, "cuda")[0]
    S = torch.randn((wd.n_seqs, wd.H, wd.d_k, wd.d_v), dtype=torch.float32, device="cuda") * 0.1
    n = max(1, args.warmup)
    for _ in range(n):
        g.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], S0=d["S0"],
                      cu_seqlens=d["cu_seqlens"])
        g.gdr_linear_attn(d["q"], d["k"], d["v"], S0=d["S0"], cu_seqlens=d["cu_seqlens"])
        g.gdr_decode_step(x["q"], x["k"], x["v"], x["alpha"], x["beta"], S)
    if args.profile_variants:  # then the rows timed outside the step, in the bench's order
        gate_in = torch.randn(d["v"].shape, device="cuda").mul_(2.0).to(torch.bfloat16)
        R = gi.device_full(wp, "cuda", seed_offset=7, raw=True)
        M = {kk: torch.empty_like(R[kk]) for kk in ("q", "k", "alpha", "beta")}
        Z = S.sum(dim=3).abs_().add_(1.0)
        for _ in range(n):
            g.gdr_gated_linear_attn(d["q"], d["k"], d["v"], d["alpha"], S0=d["S0"],
                                    cu_seqlens=d["cu_seqlens"])
            g.gdr_prefill_output_gate(d["q"], d["k"], d["v"], d["alpha"], d["beta"], gate_in,
                                      S0=d["S0"], cu_seqlens=d["cu_seqlens"])
            g.gdr_prefill(R["q"], R["k"], d["v"], R["alpha"], R["beta"], S0=d["S0"],
                          cu_seqlens=d["cu_seqlens"], prologue=True)
            g.gdr_layer_prologue(R["q"], R["k"], R["alpha"], R["beta"], q=M["q"], k=M["k"],
                                 alpha=M["alpha"], beta=M["beta"])
            g.gdr_normalized_linear_attn(d["q"], d["k"], d["v"], eps=1e-6, S0=d["S0"],
                                         cu_seqlens=d["cu_seqlens"])
            g.gdr_gated_linear_decode_step(x["q"], x["k"], x["v"], x["alpha"], S)
            g.gdr_normalized_linear_decode_step(x["q"], x["k"], x["v"], S, Z, eps=1e-6)
    torch.cuda.synchronize()
    print("profile case done: 1 x %d tokens x 32 heads, %d launches of each kernel"
          % (args.profile_tokens, n))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-tokens", type=int, default=0,
                    help="profiler target only: the step's kernels on 1 x T tokens, then exit")
    ap.add_argument("--profile-variants", action="store_true",
                    help="with --profile-tokens: also the rows timed outside the step")
    args = ap.parse_args()
    if args.profile_tokens > 0:
        return run_profile(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
