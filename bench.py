"""Benchmark of the KDA state path on GB300.

One JSON line on stdout (rank 0).  A step is one pass of the path over one
batch of seeded synthetic input with everything resident in HBM:

  varlen (default headline): kda_chunk_prefill over 8 sequences with lengths
      uniform in [64, 2048] (seed 1), H = 64, bf16, resuming from checkpointed
      fp32 states; metric = prefill tokens/s.
  decode:  69 x (copy-on-write restores for 10% of 384 requests, then
      kda_decode_step on 384 requests x 64 heads over a 512-slot pool).
  verify:  69 kda_verify_store_inputs launches (64 requests x 8 draft tokens x
      64 heads) and one kda_replay_fold over all 69 layers.

The decode and verify+fold workloads are measured in the same run and reported
under "also".  --impl reference times the oracle (fp64 CPU) on the same
workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import kda_inputs as gen  # noqa: E402

KD = VD = 128
STATE_B = KD * VD * 4


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------
# clocks sampler (nvidia-smi during the timed region)
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        t0, t1 = (self.marks[0], self.marks[-1]) if len(self.marks) >= 2 else (0, 1e30)
        inside = [s for t, s in self.samples if t0 <= t <= t1] or [s for _, s in self.samples]
        sm = [float(s[0]) for s in inside if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in inside if s[1].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in inside:
            for n, v in zip(names, s[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(inside)}


# ---------------------------------------------------------------------------
# distributed helpers (one process per GPU; replicas only)
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units, ms, ws):
    """Whole-job rate: every rank runs the same replica workload of `units`
    units, and ms is the slowest rank's time per step."""
    return units / (ms / 1e3) * ws


def timed(fn, steps, warmup, ws, sampler=None, stream=None):
    """W warm-up steps, then exactly K timed steps between barrier+synchronize;
    CUDA events on the launching stream.  Returns ms per step (max over ranks)."""
    stream = stream or torch.cuda.current_stream()
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    if sampler:
        sampler.mark()
    ms = e0.elapsed_time(e1) / steps
    return max_over_ranks(ms, ws)


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

def varlen_workload(device, seed=1, H=64):
    return gen.varlen_batch(device, seed=seed, H=H)


NOMINAL_HBM_GBS = 8000.0   # the nominal HBM3e bandwidth the fractions are also quoted against
CHUNK = 32                 # chunk length of the tensor-core prefill


def chunked_flops_per_token_head(C=CHUNK, d=KD):
    """Tensor-core work of the chunked form per token and head: the state
    products (read-out of Q e^G S, U = U~ - W S, the state increment) 6 d^2, the
    intra-chunk Gram and WY products 10 C d, the triangular solve 2 C^2 / 3."""
    return 6 * d * d + 10 * C * d + 2 * C * C / 3


def with_nominal(d, hbm):
    """Copy of a result dict in which every HBM fraction of measured peak (a key
    ending in "_frac" or "frac", not a tensor fraction) is also given against the
    nominal 8 TB/s."""
    if not isinstance(d, dict):
        return d
    out = {}
    for k, v in d.items():
        out[k] = with_nominal(v, hbm)
        if (k == "frac" or k.endswith("_frac")) and "tensor" not in k and "nominal" not in k \
                and isinstance(v, (int, float)):
            nk = k + "_of_nominal_8tbs"
            if nk not in d and "frac_of_nominal_8tbs" not in d:
                out[nk] = v * hbm / NOMINAL_HBM_GBS
    return out


def varlen_config(T, lengths, alg_bytes):
    """The config dict of the headline line; both arms print the same one."""
    return {"workload": "varlen prefill: 8 seqs, lengths U[64,2048] (seed 1), H=64, K=V=128, "
                        "bf16 inputs, fp32 states resumed from checkpoints",
            "total_tokens": int(T), "lengths": [int(x) for x in lengths],
            "l2": "inputs larger than L2 (%.2f GB per step)" % (alg_bytes / 1e9)}


def algorithmic_prefill_bytes(T, H, N, es=2, init_read=True, snap=False):
    per_tok = H * (3 * KD * es + VD * es + es + VD * es)   # q, k, gk, v, beta in; o out
    states = N * H * STATE_B * ((1 if init_read else 0) + 1 + (1 if snap else 0))
    return T * per_tok + states


def bench_varlen(args, ws, sampler):
    import kda_state_gb300 as kda
    dev = "cuda"
    w = varlen_workload(dev)
    x, N, H, T = w["x"], w["N"], w["H"], w["T"]
    pool = torch.empty(2 * N, H, KD, VD, device=dev)
    pool[:N] = w["ck"]
    cu_d = w["cu"].to(dev)
    init = torch.arange(N, dtype=torch.int32, device=dev)
    out = torch.arange(N, 2 * N, dtype=torch.int32, device=dev)
    o = torch.empty(T, H, VD, dtype=torch.bfloat16, device=dev)
    cu_h = w["cu"]

    def step():
        kda.kda_chunk_prefill(x["q"], x["k"], x["v"], x["gk"], x["beta"], cu_d, cu_h, pool, init,
                              out, o=o)

    ms = timed(step, args.steps, args.warmup, ws, sampler)
    # end to end: every step copies its inputs from pinned host memory to the
    # device and its output back.  The steps are pipelined as a server would
    # run them: step i+1's inputs move in (two streams, so two copy engines)
    # while step i computes and step i-1's output moves out (a third stream),
    # with device inputs and outputs double-buffered and events ordering each
    # buffer's reuse.
    hx = {n: t.cpu().pin_memory() for n, t in x.items()}
    cu_pin = cu_h.pin_memory()
    ho = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    dx = [{n: torch.empty_like(t) for n, t in x.items()} for _ in range(2)]
    cu_dd = [torch.empty_like(cu_d) for _ in range(2)]
    do = [torch.empty_like(o) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in hx.values()) + cu_h.numel() * 4
    d2h = ho[0].numel() * ho[0].element_size()
    s_cmp = torch.cuda.current_stream()
    s_in = [torch.cuda.Stream(), torch.cuda.Stream()]
    s_out = torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    ev_in = [[ev(), ev()] for _ in range(2)]     # [buffer][input stream]
    ev_cmp = [ev(), ev()]
    ev_out = [ev(), ev()]
    lanes = [("q", "k"), ("v", "gk", "beta")]    # inputs per input stream
    count = {"k": 0}

    def step_e2e():
        j = count["k"] & 1
        count["k"] += 1
        for a, st in enumerate(s_in):
            st.wait_event(ev_cmp[j])              # the compute that last read dx[j] is done
            with torch.cuda.stream(st):
                for n in lanes[a]:
                    dx[j][n].copy_(hx[n], non_blocking=True)
                if a == 0:
                    cu_dd[j].copy_(cu_pin, non_blocking=True)
                ev_in[j][a].record(st)
        for a in range(2):
            s_cmp.wait_event(ev_in[j][a])
        s_cmp.wait_event(ev_out[j])               # the copy that last read do[j] is done
        d = dx[j]
        kda.kda_chunk_prefill(d["q"], d["k"], d["v"], d["gk"], d["beta"], cu_dd[j], cu_h, pool,
                              init, out, o=do[j])
        ev_cmp[j].record(s_cmp)
        s_out.wait_event(ev_cmp[j])
        with torch.cuda.stream(s_out):
            ho[j].copy_(do[j], non_blocking=True)
            ev_out[j].record(s_out)

    K_e2e = max(3, args.steps // 4)
    for _ in range(3):
        step_e2e()
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_cmp)
    for st in s_in + [s_out]:
        st.wait_stream(s_cmp)                     # nothing of the timed steps starts before e0
    for _ in range(K_e2e):
        step_e2e()
    for st in s_in + [s_out]:
        s_cmp.wait_stream(st)                     # every copy of the timed steps ends before e1
    e1.record(s_cmp)
    torch.cuda.synchronize()
    barrier(ws)
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / K_e2e, ws)
    alg = algorithmic_prefill_bytes(T, H, N)
    return dict(ms=ms, ms_e2e=ms_e2e, T=T, H=H, N=N, lengths=w["lengths"], alg_bytes=alg,
                h2d=h2d, d2h=d2h, launches_per_step=1)


def bench_varlen_checkpoints(args, ws, interval=256):
    """The varlen workload with the state also written after every 256 tokens
    of each sequence (the prefix cache's block) into a slot list."""
    import kda_state_gb300 as kda
    dev = "cuda"
    w = varlen_workload(dev)
    x, N, H, T = w["x"], w["N"], w["H"], w["T"]
    lengths = list(w["lengths"])
    cap = max(lengths) // interval
    made = sum(min(L // interval, cap) for L in lengths)
    pool = torch.empty(2 * N + N * cap, H, KD, VD, device=dev)
    pool[:N] = w["ck"]
    slots = torch.arange(2 * N, 2 * N + N * cap, dtype=torch.int32, device=dev).view(N, cap)
    cu_d = w["cu"].to(dev)
    init = torch.arange(N, dtype=torch.int32, device=dev)
    out = torch.arange(N, 2 * N, dtype=torch.int32, device=dev)
    o = torch.empty(T, H, VD, dtype=torch.bfloat16, device=dev)
    cu_h = w["cu"]

    def step():
        kda.kda_chunk_prefill_checkpoints(x["q"], x["k"], x["v"], x["gk"], x["beta"], cu_d, cu_h,
                                          pool, init, out, interval, slots, o=o)

    ms = timed(step, args.steps, args.warmup, ws)
    alg = algorithmic_prefill_bytes(T, H, N) + made * H * STATE_B
    del pool
    torch.cuda.empty_cache()
    return dict(ms=ms, T=T, alg_bytes=alg, checkpoints=made, interval=interval)


def bench_long(args, ws, N=4, T=24576, H=96, piece=4096, steps=None):
    """Six 4096-token pieces of 4 x 24576 tokens (H = 96), each piece one
    kda_chunk_prefill over the 4 sequences resuming in place from the working
    slots, with a snapshot to a slot alternating between two (ping-pong)."""
    import kda_state_gb300 as kda
    dev = "cuda"
    P = T // piece
    gd = gen.make_gen(1002, dev)
    xs = [gen.token_inputs(N * piece, H, torch.bfloat16, gd, device=dev) for _ in range(P)]
    ck = gen.checkpoint((N, H, KD, VD), gd, device=dev)
    pool = torch.zeros(3 * N, H, KD, VD, device=dev)
    work = torch.arange(N, dtype=torch.int32, device=dev)
    snaps = [torch.arange(N, 2 * N, dtype=torch.int32, device=dev),
             torch.arange(2 * N, 3 * N, dtype=torch.int32, device=dev)]
    cu = gen.cu_seqlens([piece] * N)
    cu_d = cu.to(dev)
    o = torch.empty(N * piece, H, VD, dtype=torch.bfloat16, device=dev)

    def step():
        pool[:N].copy_(ck)
        for pc in range(P):
            x = xs[pc]
            kda.kda_chunk_prefill(x["q"], x["k"], x["v"], x["gk"], x["beta"], cu_d, cu, pool, work,
                                  work, snaps[pc % 2], o=o)

    K = steps or max(3, min(args.steps, 10))
    ms = timed(step, K, 3, ws)
    alg = P * algorithmic_prefill_bytes(N * piece, H, N, snap=True)
    del xs, pool
    torch.cuda.empty_cache()
    return dict(ms=ms, tokens=N * T, alg_bytes=alg, pieces=P)


def bench_decode(args, ws, layers=69, B=384, H=64, slots=512, cow_frac=0.10, steps=None):
    import kda_state_gb300 as kda
    dev = "cuda"
    g = gen.make_gen(3)
    perm = gen.slot_permutation(slots, g)
    ids = perm[:B].to(dev)
    unused = perm[B:]
    n_cow = int(cow_frac * B)
    cow_req = torch.randperm(B, generator=g)[:n_cow]
    cow_dst = perm[:B][cow_req].to(torch.int32).to(dev)
    cow_src = unused[torch.randint(0, slots - B, (n_cow,), generator=g)].to(torch.int32).to(dev)
    gd = gen.make_gen(1003, dev)
    pools = [gen.checkpoint((slots, H, KD, VD), gd, device=dev) for _ in range(layers)]
    xs = [gen.token_inputs(B, H, torch.bfloat16, gd, device=dev) for _ in range(layers)]
    o = torch.empty(B, H, VD, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(layers)]
    record = {"on": False}

    def step():
        for l in range(layers):
            kda.kda_slot_copy([pools[l]], cow_src, cow_dst)
            x = xs[l]
            if record["on"]:
                ev[l][0].record(stream)
            kda.kda_decode_step(x["q"], x["k"], x["v"], x["gk"], x["beta"], ids, pools[l], o=o)
            if record["on"]:
                ev[l][1].record(stream)

    K = steps or max(3, min(args.steps, 10))
    ms = timed(step, K, max(3, min(args.warmup, 3)), ws)
    record["on"] = True
    step()
    torch.cuda.synchronize()
    record["on"] = False
    dec_ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    per_unit = 2 * STATE_B + (3 * KD + VD) * 2 + 2 + VD * 2
    dec_bytes = B * H * per_unit
    cow_bytes = 2 * n_cow * H * STATE_B
    del pools, xs
    torch.cuda.empty_cache()
    return dict(ms=ms, dec_ms=dec_ms, dec_bytes=dec_bytes, cow_bytes=cow_bytes, B=B, H=H,
                layers=layers, n_cow=n_cow)


def bench_decode_fused(args, ws, layers=69, B=384, H=64, slots=512, steps=None):
    """Conv + KDA + onorm decode (one kda_decode_fused launch per layer) against
    the unfused path (kda_conv_prologue + kda_decode_step + kda_gated_rmsnorm per
    layer) on the same pools, conv states and raw inputs."""
    import kda_state_gb300 as kda
    dev = "cuda"
    g = gen.make_gen(3)
    ids = gen.slot_permutation(slots, g)[:B].to(dev)
    gd = gen.make_gen(1007, dev)
    pools = [gen.checkpoint((slots, H, KD, VD), gd, device=dev) for _ in range(layers)]
    convs = [gen.checkpoint((slots, 3, 3, H, KD), gd, device=dev, std=1.0).to(torch.bfloat16)
             for _ in range(layers)]
    xs = [{n: t[:, 0] for n, t in gen.raw_projections(1, H, torch.bfloat16, gd, device=dev,
                                                        lead=(B,)).items()} for _ in range(layers)]
    wts = [gen.fused_weights(H, torch.bfloat16, gd, device=dev) for _ in range(layers)]
    out = torch.empty(B, H, VD, dtype=torch.bfloat16, device=dev)
    q, k, v = (torch.empty(B, H, KD, dtype=torch.bfloat16, device=dev) for _ in range(3))
    beta = torch.empty(B, H, dtype=torch.bfloat16, device=dev)
    o = torch.empty(B, H, VD, dtype=torch.bfloat16, device=dev)
    cu = torch.arange(B + 1, dtype=torch.int32)
    cu_d = cu.to(dev)
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(layers)]
    record = {"on": False}
    scale = KD ** -0.5

    def step_fused():
        for l in range(layers):
            x, w = xs[l], wts[l]
            if record["on"]:
                ev[l][0].record(stream)
            kda.kda_decode_fused(x["qkv"][:, 0], x["qkv"][:, 1], x["qkv"][:, 2], x["gk"], x["b"],
                                 w["conv_w"], convs[l], x["gate"], w["w_norm"], ids, pools[l],
                                 out=out, scale=scale)
            if record["on"]:
                ev[l][1].record(stream)

    def step_unfused():
        for l in range(layers):
            x, w = xs[l], wts[l]
            kda.kda_conv_prologue(x["qkv"][:, 0], x["qkv"][:, 1], x["qkv"][:, 2], x["b"],
                                  w["conv_w"], convs[l], ids, ids, cu_d, cu, out=(q, k, v, beta))
            kda.kda_decode_step(q, k, v, x["gk"], beta, ids, pools[l], o=o, scale=scale)
            kda.kda_gated_rmsnorm(o, x["gate"], w["w_norm"], out=out)

    K = steps or max(3, min(args.steps, 10))
    ms_unfused = timed(step_unfused, K, 3, ws)
    ms = timed(step_fused, K, 3, ws)
    record["on"] = True
    step_fused()
    torch.cuda.synchronize()
    record["on"] = False
    fused_ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    # per unit: state in + out, raw q k v, b, gk, gate, conv state in + out, normed o out
    per_unit = 2 * STATE_B + 3 * KD * 2 + 2 + KD * 2 + VD * 2 + 2 * 3 * 3 * KD * 2 + VD * 2
    del pools, convs, xs
    torch.cuda.empty_cache()
    return dict(ms=ms, ms_unfused=ms_unfused, fused_ms=fused_ms, fused_bytes=B * H * per_unit,
                B=B, H=H, layers=layers)


def bench_prefill_fused(args, ws):
    """The varlen batch from raw projections: kda_conv_prologue, then
    kda_chunk_prefill, then kda_gated_rmsnorm (the pages' prefill fusions around
    FlashKDA), each timed on its own."""
    import kda_state_gb300 as kda
    dev = "cuda"
    w = varlen_workload(dev)
    N, H, T, cu_h = w["N"], w["H"], w["T"], w["cu"]
    cu_d = cu_h.to(dev)
    gd = gen.make_gen(1008, dev)
    x = gen.raw_projections(T, H, torch.bfloat16, gd, device=dev)
    wt = gen.fused_weights(H, torch.bfloat16, gd, device=dev)
    conv = gen.checkpoint((2 * N, 3, 3, H, KD), gd, device=dev, std=1.0).to(torch.bfloat16)
    pool = torch.empty(2 * N, H, KD, VD, device=dev)
    pool[:N] = w["ck"]
    init = torch.arange(N, dtype=torch.int32, device=dev)
    out_s = torch.arange(N, 2 * N, dtype=torch.int32, device=dev)
    q, k, v = (torch.empty(T, H, KD, dtype=torch.bfloat16, device=dev) for _ in range(3))
    beta = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    o = torch.empty(T, H, VD, dtype=torch.bfloat16, device=dev)
    out = torch.empty(T, H, VD, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    # per-kernel times: five consecutive steps, each with its own events, queued
    # behind two unrecorded steps so that no host launch gap falls inside them
    ev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(5)]
    record = {"ev": None}
    scale = KD ** -0.5

    def mark(i):
        if record["ev"] is not None:
            record["ev"][i].record(stream)

    def step():
        mark(0)
        kda.kda_conv_prologue(x["qkv"][:, 0], x["qkv"][:, 1], x["qkv"][:, 2], x["b"], wt["conv_w"],
                              conv, init, out_s, cu_d, cu_h, out=(q, k, v, beta))
        mark(1)
        kda.kda_chunk_prefill(q, k, v, x["gk"], beta, cu_d, cu_h, pool, init, out_s, o=o,
                              scale=scale)
        mark(2)
        kda.kda_gated_rmsnorm(o, x["gate"], wt["w_norm"], out=out)
        mark(3)

    K = max(3, min(args.steps, 200))
    ms = timed(step, K, 3, ws)
    step()
    step()
    for evs in ev_sets:
        record["ev"] = evs
        step()
    record["ev"] = None
    torch.cuda.synchronize()
    times = [[evs[i].elapsed_time(evs[i + 1]) for i in range(3)] for evs in ev_sets]
    med = [statistics.median(t[i] for t in times) for i in range(3)]
    th = T * H
    pro_bytes = th * (3 * KD * 2 + 2 + 3 * KD * 2 + 2) + 2 * N * H * 3 * 3 * KD * 2
    norm_bytes = th * 3 * VD * 2
    return dict(ms=ms, T=T, prologue_ms=med[0], prefill_ms=med[1], norm_ms=med[2],
                prologue_bytes=pro_bytes, norm_bytes=norm_bytes)


def bench_verify_fold(args, ws, layers=69, B=64, G=8, H=64, slots=128, R=16, steps=None,
                      ragged=False):
    """Verify of B requests x G drafts on every layer, then one fold.  ragged:
    each request verifies its own G_b <= G drafts (uniform on 1..G, packed by
    cu_drafts) and accepts at most G_b."""
    import kda_state_gb300 as kda
    dev = "cuda"
    g = gen.make_gen(4)
    ids = gen.slot_permutation(slots, g)[:B].to(dev)
    accept = gen.accept_lengths(B, G, 0.64, g)
    Gb = gen.draft_lengths(B, G, g) if ragged else torch.full((B,), G, dtype=torch.int32)
    accept = torch.minimum(accept, Gb)
    acc_d = accept.to(dev)
    cu_d = torch.cat([torch.zeros(1, dtype=torch.int32), Gb.cumsum(0).to(torch.int32)]).to(dev)
    n_tok = int(Gb.sum())
    gd = gen.make_gen(1004, dev)
    pools = [gen.checkpoint((slots, H, KD, VD), gd, device=dev) for _ in range(layers)]
    rings = [kda.make_ring(slots, R, H, torch.bfloat16, dev) for _ in range(layers)]
    if ragged:
        xs = [gen.token_inputs(n_tok, H, torch.bfloat16, gd, device=dev) for _ in range(layers)]
        o = torch.empty(n_tok, H, VD, dtype=torch.bfloat16, device=dev)
    else:
        xs = [gen.token_inputs(G, H, torch.bfloat16, gd, device=dev, lead=(B,)) for _ in range(layers)]
        o = torch.empty(B, G, H, VD, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    ev_v = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(layers)]
    ev_f = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    record = {"on": False}

    def step():
        for l in range(layers):
            x = xs[l]
            if record["on"]:
                ev_v[l][0].record(stream)
            if ragged:
                kda.kda_verify_store_inputs_ragged(x["q"], x["k"], x["v"], x["gk"], x["beta"], cu_d,
                                                   G, ids, pools[l], rings[l], o=o)
            else:
                kda.kda_verify_store_inputs(x["q"], x["k"], x["v"], x["gk"], x["beta"], ids,
                                            pools[l], rings[l], o=o)
            if record["on"]:
                ev_v[l][1].record(stream)
        if record["on"]:
            ev_f[0].record(stream)
        kda.kda_replay_fold(pools, rings, ids, acc_d, max_accept=G)
        if record["on"]:
            ev_f[1].record(stream)

    K = steps or max(3, min(args.steps, 10))
    ms = timed(step, K, max(3, min(args.warmup, 3)), ws)
    record["on"] = True
    step()
    torch.cuda.synchronize()
    record["on"] = False
    ver_ms = statistics.median(a.elapsed_time(b) for a, b in ev_v)
    fold_ms = ev_f[0].elapsed_time(ev_f[1])
    rec = 2 * KD + 2 * VD + 4 * KD + 4
    n_units = int((Gb > 0).sum())
    ver_bytes = H * (n_units * STATE_B + n_tok * (3 * KD * 2 + VD * 2 + 2 + VD * 2 + rec))
    acc_sum = int(accept.sum())
    fold_bytes = layers * H * (2 * STATE_B * int((accept > 0).sum()) + acc_sum * rec)
    del pools, rings, xs
    torch.cuda.empty_cache()
    return dict(ms=ms, ver_ms=ver_ms, fold_ms=fold_ms, ver_bytes=ver_bytes, fold_bytes=fold_bytes,
                accepted=acc_sum, mean_accept=acc_sum / B, B=B, G=G, layers=layers, H=H,
                verified=n_tok, mean_draft=n_tok / B)


def bench_snapshot_ab(args, ws, layers=69, B=64, G=8, H=64, slots=128, R=16, steps=None):
    """A/B of the two ways to make speculation reversible, on one workload:
    ReplaySSM (verify storing ~1 KB records, then one fold) against the
    snapshot-per-step baseline (verify writing the 64 KB state after every
    draft step, then one commit copy).  Same drafts, pools and accept lengths."""
    import kda_state_gb300 as kda
    dev = "cuda"
    g = gen.make_gen(4)
    ids = gen.slot_permutation(slots, g)[:B].to(dev)
    acc_d = gen.accept_lengths(B, G, 0.64, g).to(dev)
    snap_ids = torch.arange(B, dtype=torch.int32, device=dev)
    gd = gen.make_gen(1004, dev)
    pools = [gen.checkpoint((slots, H, KD, VD), gd, device=dev) for _ in range(layers)]
    rings = [kda.make_ring(slots, R, H, torch.bfloat16, dev) for _ in range(layers)]
    snaps = [torch.empty(B, G, H, KD, VD, device=dev) for _ in range(layers)]
    xs = [gen.token_inputs(G, H, torch.bfloat16, gd, device=dev, lead=(B,)) for _ in range(layers)]
    o = torch.empty(B, G, H, VD, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    ev = {k: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(layers)] for k in ("ver", "snap")}
    ev1 = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for k in ("fold", "commit")}
    record = {"on": False}

    def mark(pair, i):
        if record["on"]:
            pair[i].record(stream)

    def step_replay():
        for l in range(layers):
            x = xs[l]
            mark(ev["ver"][l], 0)
            kda.kda_verify_store_inputs(x["q"], x["k"], x["v"], x["gk"], x["beta"], ids, pools[l],
                                        rings[l], o=o)
            mark(ev["ver"][l], 1)
        mark(ev1["fold"], 0)
        kda.kda_replay_fold(pools, rings, ids, acc_d, max_accept=G)
        mark(ev1["fold"], 1)

    def step_snap():
        for l in range(layers):
            x = xs[l]
            mark(ev["snap"][l], 0)
            kda.kda_verify_snapshot(x["q"], x["k"], x["v"], x["gk"], x["beta"], ids, pools[l],
                                    snaps[l], snap_ids, o=o)
            mark(ev["snap"][l], 1)
        mark(ev1["commit"], 0)
        kda.kda_snapshot_commit(pools, snaps, ids, snap_ids, acc_d)
        mark(ev1["commit"], 1)

    K = steps or max(3, min(args.steps, 10))
    res = {}
    for name, fn in (("replayssm", step_replay), ("snapshot", step_snap)):
        ms = timed(fn, K, 3, ws)
        record["on"] = True
        fn()
        torch.cuda.synchronize()
        record["on"] = False
        vk, ck = ("ver", "fold") if name == "replayssm" else ("snap", "commit")
        res[name] = {"ms_per_step": ms,
                     "verify_kernel_us": statistics.median(a.elapsed_time(b) for a, b in ev[vk]) * 1e3,
                     "commit_kernel_us": ev1[ck][0].elapsed_time(ev1[ck][1]) * 1e3}
    rec = 2 * KD * 2 + 4 * KD + 4
    res["replayssm"]["draft_bytes_per_request"] = layers * H * R * rec
    res["snapshot"]["draft_bytes_per_request"] = layers * H * G * STATE_B
    del pools, rings, snaps, xs
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline / reference arm)
# ---------------------------------------------------------------------------

class OracleVarlen:
    """The oracle (fp64, host cores) on a bounded sample of the varlen workload:
    whole heads (all 8 sequences of a head) of the same-shaped inputs."""

    def __init__(self):
        import oracle
        self.oracle = oracle
        w = varlen_workload("cpu")
        self.cu = w["cu"].numpy()
        self.H = w["H"]
        self.T = int(self.cu[-1])
        self.x = {n: t.double().numpy() for n, t in w["x"].items()}
        self.S0 = w["ck"].double().numpy()
        self.threads = os.cpu_count() or 1
        # calibrate the per-token cost on the shortest sequence, one thread
        n0 = int(np.argmin(np.diff(self.cu)))
        t0 = time.time()
        self._run([n0], [0], 1)
        self.sec_per_tok = (time.time() - t0) / max(1, self.cu[n0 + 1] - self.cu[n0])

    def _run(self, seqs, heads, threads):
        x = self.x
        self.oracle.prefill_varlen(x["q"], x["k"], x["v"], x["gk"], x["beta"], self.cu, self.S0,
                                   seqs=seqs, heads=heads, nthreads=threads)

    def heads_for(self, seconds):
        return max(1, min(self.H, int(seconds * self.threads / (self.sec_per_tok * self.T))))

    def rate(self, n_heads):
        """tokens/s: token-heads processed / H / wall time."""
        t0 = time.time()
        self._run(list(range(8)), list(range(n_heads)), self.threads)
        dt = time.time() - t0
        return self.T * n_heads / self.H / dt, dt


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

CSRC = os.path.join(ROOT, "kda_state_gb300", "csrc")


def _device_headers(name, seen):
    """The local device headers (.cuh) a source includes, depth first, in order."""
    for line in open(os.path.join(CSRC, name)):
        m = re.match(r'\s*#include\s+"([^"/]+\.cuh)"', line)
        if m and m.group(1) not in seen:
            seen.append(m.group(1))
            _device_headers(m.group(1), seen)
    return seen


def source_sha1(kernel_file):
    """First 12 hex digits of the sha1 over a kernel's source file followed by
    the device headers it includes (the hash the profile summaries record as
    source_sha1)."""
    h = hashlib.sha1()
    for f in [kernel_file] + _device_headers(kernel_file, []):
        h.update(open(os.path.join(CSRC, f), "rb").read())
    return h.hexdigest()[:12]


def profile_traffic(kernel_file, summary_name, key="dram_bytes_per_launch"):
    """DRAM bytes (read + write) from a committed ncu summary, if it was taken
    on the current kernel source (matched by hash); else None."""
    path = os.path.join(ROOT, "profiles", summary_name)
    try:
        txt = open(path).read()
    except OSError:
        return None
    m_h = re.search(r"source_sha1:\s*([0-9a-f]+)", txt)
    m_t = re.search(key + r":\s*([0-9.eE+]+)", txt)
    if not m_h or not m_t or m_h.group(1) != source_sha1(kernel_file):
        return None
    return float(m_t.group(1))


def run_reference(args, ws, rank):
    if rank != 0:
        return
    orc = OracleVarlen()
    n_heads = orc.heads_for(max(0.2, 120.0 / (args.steps + args.warmup)))
    rates, secs = [], 0.0
    for i in range(args.warmup + args.steps):
        r, dt = orc.rate(n_heads)
        if i >= args.warmup:
            rates.append(r)
            secs += dt
    v = statistics.mean(rates)
    lengths = np.diff(orc.cu).tolist()
    alg = algorithmic_prefill_bytes(orc.T, orc.H, len(lengths))
    desc = ("per step: %d (sequence, head) units (8 sequences x %d heads) = %d token-heads of the "
            "varlen workload" % (8 * n_heads, n_heads, orc.T * n_heads))
    line = {"impl": "reference", "metric": "KDA prefill tok/s (varlen chunked prefill)",
            "value": v, "unit": "tok/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": varlen_config(orc.T, lengths, alg),
            "cpu_baseline": {"value": v, "unit": "tok/s", "cores": orc.threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-also", action="store_true", help="skip the decode / verify+fold runs")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--only", choices=["decode", "decode_fused", "prefill_fused", "verify",
                                       "verify_ragged", "snapshot_ab", "checkpoints"],
                    default=None,
                    help="run one of the secondary workloads alone (for profiling)")
    ap.add_argument("--layers", type=int, default=69,
                    help="layers of the --only workload (a smaller case for profiling)")
    args = ap.parse_args()
    ws, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    if args.only:
        torch.cuda.set_device(local)
        from kda_state_gb300 import _build
        _build.build()
        if args.only == "checkpoints":
            r = bench_varlen_checkpoints(args, 1)
        elif args.only == "decode_fused":
            r = bench_decode_fused(args, 1, layers=args.layers, steps=args.steps)
        elif args.only == "prefill_fused":
            r = bench_prefill_fused(args, 1)
        elif args.only == "snapshot_ab":
            r = bench_snapshot_ab(args, 1, layers=args.layers, steps=args.steps)
            r = {f"{a}_{k}": v for a, d in r.items() for k, v in d.items()}
        elif args.only == "verify_ragged":
            r = bench_verify_fold(args, 1, layers=args.layers, steps=args.steps, ragged=True)
        else:
            fn = bench_decode if args.only == "decode" else bench_verify_fold
            r = fn(args, 1, layers=args.layers, steps=args.steps)
        print(json.dumps({"only": args.only, **{k: v for k, v in r.items()
                                                 if isinstance(v, (int, float))}}), flush=True)
        return
    if ws > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    # CPU baseline first (before the first GPU call, no fork after CUDA init)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        try:
            orc = OracleVarlen()
            nh = orc.heads_for(10.0)
            tok, secs, passes = 0.0, 0.0, 0
            while secs < 10.0 and passes < 50:     # repeat the sample to about 10 s
                r, dt = orc.rate(nh)
                tok += r * dt
                secs += dt
                passes += 1
            cpu = {"value": tok / secs, "unit": "tok/s", "cores": orc.threads, "kind": "oracle",
                   "sample": "%d pass(es) over %d (sequence, head) units (8 sequences x %d of 64 "
                             "heads, %d token-heads each), %.1f s" % (passes, 8 * nh, nh, orc.T * nh,
                                                                      secs)}
        except Exception as e:  # noqa: BLE001
            cpu = {"value": None, "unit": "tok/s", "cores": None, "kind": "oracle",
                   "sample": "failed: %s" % e}
    from kda_state_gb300 import _build
    _build.build()
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    res = bench_varlen(args, ws, sampler)
    if sampler:
        time.sleep(0.3)
        sampler.stop()
    hbm, tc_peak, peak_kind = peaks()
    ms = res["ms"]
    value = aggregate_rate(res["T"], ms, ws)
    achieved = res["alg_bytes"] / (ms / 1e3) / 1e9
    tflops = res["T"] * res["H"] * chunked_flops_per_token_head() / (ms / 1e3) / 1e12
    traffic = profile_traffic("kda_prefill_tc.cu", "prefill_tc_kernel.varlen.md")
    line = {
        "metric": "KDA prefill tok/s (varlen chunked prefill)",
        "value": value, "unit": "tok/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": varlen_config(res["T"], res["lengths"], res["alg_bytes"]),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic,
                     "peak_kind": peak_kind, "kernel": "kda_chunk_prefill",
                     "algorithmic_bytes_per_launch": res["alg_bytes"],
                     "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                     "tensor": {"achieved": tflops, "peak": tc_peak, "unit": "TFLOP/s",
                                "frac": tflops / tc_peak, "peak_kind": peak_kind + " bf16 burst",
                                "flops_per_token_head": chunked_flops_per_token_head(),
                                "flops_per_launch": res["T"] * res["H"] * chunked_flops_per_token_head(),
                                "note": "chunked-form flops (C = %d) over the launch time; the "
                                        "kernel is HBM-bound, so this fraction is the smaller one"
                                        % CHUNK}},
        "e2e": {"value": aggregate_rate(res["T"], res["ms_e2e"], ws), "unit": "tok/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "ms_per_step": res["ms_e2e"],
                "schedule": "pinned host inputs in and o out every step; steps pipelined: the "
                            "next step's inputs copy in (two streams) while this step computes "
                            "and the previous step's output copies out"},
        "gpu_launches": res["launches_per_step"] * args.steps,
        "clocks": sampler.summary() if sampler else None,
        "cpu_baseline": cpu,
    }
    if not args.no_also:
        also = {}
        try:
            c = bench_varlen_checkpoints(args, ws)
            also["varlen_checkpoints"] = {
                "tok_per_s": aggregate_rate(c["T"], c["ms"], ws), "ms_per_step": c["ms"],
                "workload": "the varlen batch above with the state written every %d tokens "
                            "(%d checkpoints per head) into a slot list"
                            % (c["interval"], c["checkpoints"]),
                "GBps": c["alg_bytes"] / (c["ms"] / 1e3) / 1e9,
                "frac": c["alg_bytes"] / (c["ms"] / 1e3) / 1e9 / hbm,
                "frac_of_nominal_8tbs": c["alg_bytes"] / (c["ms"] / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                "time_vs_plain": c["ms"] / res["ms"],
                "traffic": profile_traffic("kda_prefill_tc.cu", "prefill_tc_kernel.varlen_checkpoints.md"),
            }
        except Exception as e:  # noqa: BLE001
            also["varlen_checkpoints"] = {"error": repr(e)}
        try:
            lg = bench_long(args, ws)
            also["long_prefill"] = {
                "tok_per_s": aggregate_rate(lg["tokens"], lg["ms"], ws), "ms_per_step": lg["ms"],
                "workload": "4 seqs x 24576 tok, H=96, bf16, from checkpoints, 6 pieces of 4096 "
                            "resuming in place, ping-pong snapshot per piece",
                "GBps": lg["alg_bytes"] / (lg["ms"] / 1e3) / 1e9,
                "frac": lg["alg_bytes"] / (lg["ms"] / 1e3) / 1e9 / hbm,
                "frac_of_nominal_8tbs": lg["alg_bytes"] / (lg["ms"] / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                "tensor_frac": lg["tokens"] * 96 * chunked_flops_per_token_head() / (lg["ms"] / 1e3)
                               / 1e12 / tc_peak,
                "note": "step includes a 48 MB checkpoint restore before the first piece",
            }
        except Exception as e:  # noqa: BLE001
            also["long_prefill"] = {"error": repr(e)}
        try:
            d = bench_decode(args, ws)
            also["decode"] = {
                "tok_per_s": aggregate_rate(d["B"], d["ms"], ws), "ms_per_step": d["ms"],
                "workload": "384 req x 1 tok, H=64, 512-slot pools, 69 layers, %d CoW copies/layer"
                            % d["n_cow"],
                "decode_kernel_us": d["dec_ms"] * 1e3,
                "decode_kernel_GBps": d["dec_bytes"] / (d["dec_ms"] / 1e3) / 1e9,
                "decode_kernel_frac": d["dec_bytes"] / (d["dec_ms"] / 1e3) / 1e9 / hbm,
                "decode_kernel_traffic": profile_traffic("kda_decode.cu", "decode_kernel.decode.md"),
                "step_GBps": (d["dec_bytes"] + d["cow_bytes"]) * d["layers"] / (d["ms"] / 1e3) / 1e9,
            }
        except Exception as e:  # noqa: BLE001
            also["decode"] = {"error": repr(e)}
        try:
            v = bench_verify_fold(args, ws)
            also["verify_fold"] = {
                "accepted_tok_per_s": aggregate_rate(v["accepted"], v["ms"], ws),
                "verified_tok_per_s": aggregate_rate(v["B"] * v["G"], v["ms"], ws),
                "ms_per_step": v["ms"], "mean_accept": v["mean_accept"],
                "workload": "64 req x 8 draft tok, 69 layers, H=64, 128-slot pools, ring 16",
                "verify_kernel_us": v["ver_ms"] * 1e3,
                "verify_kernel_GBps": v["ver_bytes"] / (v["ver_ms"] / 1e3) / 1e9,
                "verify_kernel_frac": v["ver_bytes"] / (v["ver_ms"] / 1e3) / 1e9 / hbm,
                "verify_kernel_traffic": profile_traffic("kda_verify.cu", "verify_block_kernel.verify.md"),
                "fold_kernel_us": v["fold_ms"] * 1e3,
                "fold_kernel_GBps": v["fold_bytes"] / (v["fold_ms"] / 1e3) / 1e9,
                "fold_kernel_frac": v["fold_bytes"] / (v["fold_ms"] / 1e3) / 1e9 / hbm,
                "fold_kernel_traffic": profile_traffic("kda_fold.cu", "fold_kernel.verify.md"),
            }
        except Exception as e:  # noqa: BLE001
            also["verify_fold"] = {"error": repr(e)}
        try:
            df = bench_decode_fused(args, ws)
            also["decode_fused"] = {
                "tok_per_s": aggregate_rate(df["B"], df["ms"], ws), "ms_per_step": df["ms"],
                "unfused_ms_per_step": df["ms_unfused"],
                "workload": "384 req x 1 tok, H=64, 512-slot pools, 69 layers: conv + KDA + onorm "
                            "in one launch per layer (unfused: prologue + decode + norm)",
                "fused_kernel_us": df["fused_ms"] * 1e3,
                "fused_kernel_GBps": df["fused_bytes"] / (df["fused_ms"] / 1e3) / 1e9,
                "fused_kernel_frac": df["fused_bytes"] / (df["fused_ms"] / 1e3) / 1e9 / hbm,
                "fused_kernel_traffic": profile_traffic("kda_decode_fused.cu",
                                                        "decode_fused_kernel.decode_fused.md"),
            }
        except Exception as e:  # noqa: BLE001
            also["decode_fused"] = {"error": repr(e)}
        try:
            pf = bench_prefill_fused(args, ws)
            also["prefill_fused_path"] = {
                "tok_per_s": aggregate_rate(pf["T"], pf["ms"], ws), "ms_per_step": pf["ms"],
                "workload": "the varlen batch from raw projections: conv prologue, chunked "
                            "prefill, gated RMSNorm",
                "prologue_us": pf["prologue_ms"] * 1e3,
                "prologue_frac": pf["prologue_bytes"] / (pf["prologue_ms"] / 1e3) / 1e9 / hbm,
                "prefill_us": pf["prefill_ms"] * 1e3,
                "norm_us": pf["norm_ms"] * 1e3,
                "norm_frac": pf["norm_bytes"] / (pf["norm_ms"] / 1e3) / 1e9 / hbm,
                "prologue_traffic": profile_traffic(
                    "kda_prologue.cu", "conv_prologue_kernel_gated_rmsnorm_kernel.prefill_fused.md"),
                "norm_traffic": profile_traffic(
                    "kda_prologue.cu", "conv_prologue_kernel_gated_rmsnorm_kernel.prefill_fused.md",
                    "norm_dram_bytes_per_launch"),
            }
        except Exception as e:  # noqa: BLE001
            also["prefill_fused_path"] = {"error": repr(e)}
        try:
            ab = bench_snapshot_ab(args, ws)
            ab["workload"] = ("64 req x 8 draft tok, 69 layers, H=64, 128-slot pools: ReplaySSM "
                              "(records + fold) vs snapshot per draft step (+ commit copy)")
            ab["draft_memory_ratio"] = (ab["snapshot"]["draft_bytes_per_request"]
                                        / ab["replayssm"]["draft_bytes_per_request"])
            also["snapshot_ab"] = ab
        except Exception as e:  # noqa: BLE001
            also["snapshot_ab"] = {"error": repr(e)}
        try:
            v = bench_verify_fold(args, ws, ragged=True)
            also["verify_fold_ragged"] = {
                "accepted_tok_per_s": aggregate_rate(v["accepted"], v["ms"], ws),
                "verified_tok_per_s": aggregate_rate(v["verified"], v["ms"], ws),
                "ms_per_step": v["ms"], "mean_accept": v["mean_accept"],
                "mean_draft": v["mean_draft"],
                "workload": "64 req x G_b ~ U{1..8} draft tok (trimmed windows), 69 layers, H=64, "
                            "128-slot pools, ring 16",
                "verify_kernel_us": v["ver_ms"] * 1e3,
                "verify_kernel_GBps": v["ver_bytes"] / (v["ver_ms"] / 1e3) / 1e9,
                "verify_kernel_frac": v["ver_bytes"] / (v["ver_ms"] / 1e3) / 1e9 / hbm,
                "fold_kernel_us": v["fold_ms"] * 1e3,
            }
        except Exception as e:  # noqa: BLE001
            also["verify_fold_ragged"] = {"error": repr(e)}
        line["also"] = {k: with_nominal(v, hbm) for k, v in also.items()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
