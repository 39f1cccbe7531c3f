"""Throughput of the GDN token-mixer hot path on the serving-mix sweep.

Workload (one "step" of this benchmark = one full sweep): 24 GDN layers of the
Qwen3.5-4B shape (conv over 8192 channels = q 16x128 | k 16x128 | v 32x128,
width 4, SiLU; delta rule with 32 v-heads over 16 q/k-heads, d = 128), 32
sequences with prompt lengths U[512, 1024] (seed 4) packed in order into
prefill steps of at most 2048 tokens, then 128 decode steps over all 32
sequences. Every prefill step builds its exact 8-token conv descriptors once
and reuses them in all 24 layers; each layer runs the conv (prefill or update)
and the delta rule (chunked prefill or decode) on q/k/v read in place from the
conv output, q/k L2-normalised and the gates activated from their logits
(a = exp(-softplus(z_a)), b = sigmoid(z_b)) in the kernel. Inputs are synthetic
(seeded normal x and gate logits) and distinct for every layer and step (about
11 GB per sweep, far larger than L2).

The sweep is captured once as a CUDA graph and replayed; `value` is tokens
through the 24-layer stack per second with inputs resident in HBM. `e2e` runs
the same sweep with every layer input copied from pinned host memory and every
layer output copied back inside the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

LAYERS = 24
N_SEQS = 32
STEP_TOKENS = 2048
DECODE_STEPS = 128
HK, HV, D = 16, 32, 128
C = 2 * HK * D + HV * D
CHUNK = 64
METRIC = "GDN tokens/s per step mix (prefill+decode) and achieved HBM GB/s / % roofline"
WORKLOAD = ("serving-mix sweep: 24 GDN layers (conv 8192 ch K=4 + gated delta rule 32v/16k "
            "heads d=128), 32 seqs, prompts U[512,1024] seed 4 packed into 2048-token prefill "
            "steps, then 128 decode steps")
KINDS = ("build_chunks", "conv_prefill", "delta_prefill", "conv_update", "delta_decode")
KERNEL_SOURCES = {
    "build_chunks": "gated_deltanet_linear_build_gb300/csrc/conv.cu",
    "conv_prefill": "gated_deltanet_linear_build_gb300/csrc/conv.cu",
    "conv_update": "gated_deltanet_linear_build_gb300/csrc/conv.cu",
    "delta_decode": "gated_deltanet_linear_build_gb300/csrc/decode.cu",
    "delta_prefill": "gated_deltanet_linear_build_gb300/csrc/prefill_tc.cu",
}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--case", default="mix",
                   choices=["mix", "conv_prefill", "conv_update", "decode", "prefill",
                            "decode_step", "mixed_step", "decode_units"],
                   help="mix = the serving-mix sweep (the benchmark); decode_step and "
                        "mixed_step compare two ways of running one engine step (CUDA "
                        "graphs over 24 layers); decode_units times the decode over a "
                        "range of sequence counts (units per CTA); the others time one "
                        "hot-path call on its own workload shape (per-kernel studies, ncu)")
    return p.parse_args(argv)


# ----------------------------------------------------------------------------
# Multi-rank plumbing (weak scaling: every rank runs its own independent mix)
# ----------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def reduce_over_ranks(x: float, op: str, dist=None, device="cpu") -> float:
    """MAX or SUM of a per-rank scalar (identity on one rank)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def rank_lengths_seed(rank: int) -> int:
    """Rank 0 serves the seed-4 prompt mix; rank r its own mix (seed 4 + r)."""
    return 4 + rank


# ----------------------------------------------------------------------------
# Peaks, clocks, stored ncu traffic
# ----------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return (float(pk["hbm_gbs"]), float(pk["bf16_tflops"]),
                float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), "measured")
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


def source_digest(relpath: str) -> str:
    with open(os.path.join(ROOT, relpath), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def stored_traffic(kind: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's source changed after the counters were taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kind]
        if source_digest(rec["source"]) != rec["source_sha256_16"]:
            return None
        return float(rec["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
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
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t_end = time.time() + 5.0          # let sampling start before timing
            while not self.lines and time.time() < t_end and self.proc.poll() is None:
                time.sleep(0.02)
        except OSError:
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
            self.thread.join(timeout=2)

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                mhz.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


# ----------------------------------------------------------------------------
# Algorithmic work per launch (bytes / flops), for the rooflines
# ----------------------------------------------------------------------------

def decode_delta_bytes(n=N_SEQS):
    state = 2 * n * HV * D * D * 4                 # S read + write (float32)
    qkv = n * (2 * HK * D + HV * D) * 2            # q, k, v (BF16)
    gates = 2 * n * HV * 4
    out = n * HV * D * 2
    return state + qkv + gates + out


def conv_prefill_bytes(T, n_seqs):
    return 2 * T * C * 2 + C * 4 * 2 + 2 * n_seqs * C * 3 * 2


def conv_update_bytes(n=N_SEQS):
    return 2 * n * C * 2 + 2 * n * C * 3 * 2 + C * 4 * 2


def prefill_flops(chunk_lengths, d=D, hv=HV):
    """Algorithmic flops of the chunked prefill over chunks of the given sizes,
    all v-heads: K K^T, Q K^T, Tm K, Tm V and (M o QK^T) Delta at c^2 d MACs;
    W S^T, Q S^T and Delta^T K at c d^2 MACs; forward substitution c^3 / 6."""
    macs = 0.0
    for c in chunk_lengths:
        macs += 5 * c * c * d + 3 * c * d * d + c ** 3 / 6
    return 2.0 * macs * hv


def prefill_bytes(T, n_seqs):
    per_tok = 2 * HK * D * 2 + HV * D * 2 + 2 * HV * 4 + HV * D * 2   # q,k,v,a,b,o
    return T * per_tok + 2 * n_seqs * HV * D * D * 4                  # + S in/out


# ----------------------------------------------------------------------------
# The workload on the device
# ----------------------------------------------------------------------------

class Workload:
    def __init__(self, rank: int, device):
        import torch
        from gated_deltanet_linear_build_gb300 import stack as stk, synth
        self.torch = torch
        self.lengths = [int(x) for x in synth.serving_mix_lengths(rank_lengths_seed(rank))]
        self.steps = stk.pack_prefill_steps(self.lengths, STEP_TOKENS)
        seed = 1000 + rank
        self.stack = stk.GdnLayerStack(LAYERS, N_SEQS, hk=HK, hv=HV, d=D,
                                       max_step_tokens=STEP_TOKENS, device=device, seed=seed)
        g = torch.Generator(device=device)
        g.manual_seed(seed + 1)
        self.meta = []
        for st in self.steps:
            cu, has, first = self.stack.step_meta(st)
            self.meta.append((torch.tensor(cu, dtype=torch.int32, device=device),
                              torch.tensor(has, dtype=torch.uint8, device=device), first,
                              len(has), int(st.tokens)))
        bf16 = torch.bfloat16

        def gates(T):
            # raw gate logits z_a, z_b ~ N(0, 1): the delta-rule kernels compute
            # a = exp(-softplus(z_a)) and b = sigmoid(z_b) themselves
            return (torch.randn((T, HV), generator=g, device=device).contiguous(),
                    torch.randn((T, HV), generator=g, device=device).contiguous())

        self.px = [[torch.randn((m[4], C), generator=g, device=device, dtype=bf16)
                    for _ in range(LAYERS)] for m in self.meta]
        self.pg = [[gates(m[4]) for _ in range(LAYERS)] for m in self.meta]
        self.dx = [[torch.randn((N_SEQS, C), generator=g, device=device, dtype=bf16)
                    for _ in range(LAYERS)] for _ in range(DECODE_STEPS)]
        self.dg = [[gates(N_SEQS) for _ in range(LAYERS)] for _ in range(DECODE_STEPS)]
        self.py = [torch.empty((STEP_TOKENS, C), dtype=bf16, device=device) for _ in range(LAYERS)]
        self.po = [torch.empty((STEP_TOKENS, HV, D), dtype=bf16, device=device)
                   for _ in range(LAYERS)]
        self.dy = [torch.empty((N_SEQS, C), dtype=bf16, device=device) for _ in range(LAYERS)]
        self.do = [torch.empty((N_SEQS, HV, D), dtype=bf16, device=device) for _ in range(LAYERS)]
        self.prefill_tokens = sum(self.lengths)
        self.decode_tokens = DECODE_STEPS * N_SEQS
        self.tokens = self.prefill_tokens + self.decode_tokens
        # Each step's conv descriptors, built once here for the per-kind timing
        # (the sweep itself rebuilds them into the stack's buffer every step).
        from gated_deltanet_linear_build_gb300 import gdn
        self.step_chunks = []
        for (cu, has, first, n, T) in self.meta:
            ch = torch.empty((T // 8 + n, 4), dtype=torch.int32, device=device)
            cnt = torch.empty((1,), dtype=torch.int32, device=device)
            gdn.build_conv_chunks(cu, ch, cnt, chunk_tokens=8)
            self.step_chunks.append((ch, cnt))

    def chunk_lengths(self):
        return [min(CHUNK, s.length - CHUNK * j) for st in self.steps for s in st.segments
                for j in range(-(-s.length // CHUNK))]

    def sweep(self):
        """Enqueue one full sweep (all prefill steps, then all decode steps)."""
        for i, (cu, has, first, n, T) in enumerate(self.meta):
            ys = [y[:T] for y in self.py]
            os_ = [o[:T] for o in self.po]
            self.stack.prefill_step(cu, has, first, n, self.px[i], self.pg[i], ys, os_)
        for j in range(DECODE_STEPS):
            self.stack.decode_step(self.dx[j], self.dg[j], self.dy, self.do)

    def kind_launches(self, kind):
        """Library calls of one kind in a sweep."""
        return {"build_chunks": len(self.meta), "conv_prefill": LAYERS * len(self.meta),
                "delta_prefill": LAYERS * len(self.meta), "conv_update": LAYERS * DECODE_STEPS,
                "delta_decode": LAYERS * DECODE_STEPS}[kind]

    def kind_sweep(self, kind):
        """Every call of one kind that a sweep makes, on the same buffers and
        shapes, back to back (for per-kind launch durations). The chunked
        prefill calls run on the step's plan, remade before each step's calls
        (so delta_prefill's time per call includes 1/24 of a plan)."""
        from gated_deltanet_linear_build_gb300 import gdn
        st = self.stack
        for i, (cu, has, first, n, T) in enumerate(self.meta):
            if kind == "build_chunks":
                st.build_chunks(cu, T)
            elif kind == "delta_prefill":
                # the step's plan, as the sweep makes it once per step
                gdn.delta_rule_prefill_plan(cu, T, HV, D, D, st.workspace)
            for l in range(LAYERS):
                if kind == "conv_prefill":
                    ch, cnt = self.step_chunks[i]
                    st.conv_prefill_layer(l, cu, has, first, n, self.px[i][l], self.py[l][:T],
                                          chunks=ch, num_chunks=cnt)
                elif kind == "delta_prefill":
                    a, b = self.pg[i][l]
                    st.delta_prefill_layer(l, cu, has, first, n, self.py[l][:T], a, b,
                                           self.po[l][:T])
        for j in range(DECODE_STEPS):
            for l in range(LAYERS):
                if kind == "conv_update":
                    st.conv_update_layer(l, self.dx[j][l], self.dy[l])
                elif kind == "delta_decode":
                    a, b = self.dg[j][l]
                    st.delta_decode_layer(l, self.dy[l], a, b, self.do[l])


E2E_BYTES_PER_TOKEN = C * 2 + 2 * HV * 4      # x (BF16) | z_a | z_b (float32)


def compact(obj, digits=6):
    """The JSON line's numbers to `digits` significant digits (floats only), so
    that the whole line stays short enough to survive a log tail."""
    if isinstance(obj, float):
        return float(f"{obj:.{digits}g}")
    if isinstance(obj, dict):
        return {k: compact(v, digits) for k, v in obj.items()}
    if isinstance(obj, (list, tuple)):
        return [compact(v, digits) for v in obj]
    return obj


def packed_layer_inputs(buf, n, base=0):
    """Views of one layer's inputs for n tokens packed back to back in the byte
    tensor ``buf`` from byte ``base``: x BF16 [n, C], then z_a and z_b float32
    [n, HV]; together they cover n * E2E_BYTES_PER_TOKEN bytes."""
    import torch
    x = buf[base:base + n * C * 2].view(torch.bfloat16).view(n, C)
    o = base + n * C * 2
    za = buf[o:o + n * HV * 4].view(torch.float32).view(n, HV)
    zb = buf[o + n * HV * 4:o + 2 * n * HV * 4].view(torch.float32).view(n, HV)
    return x, za, zb


class E2EWorkload:
    """The same sweep fed from pinned host memory: every layer's inputs (x and
    the gate logits z_a, z_b) and every step's cu_seqlens / flags are copied
    host->device, and every layer's output o is copied device->host.

    The link to the host, not the copy engines, bounds these copies (a single
    cudaMemcpyAsync already reaches it), so each copy is as large as the data
    allows: a prefill layer's x | z_a | z_b sit back to back in one device
    buffer and arrive in one copy; a decode step's inputs for all 24 layers
    arrive in one copy, and its 24 outputs, back to back in one device buffer,
    leave in one copy.

    The prefill inputs are double-buffered across sweeps, as an engine
    prefetches its next batch: each sweep's graph copies the NEXT sweep's
    prefill inputs into the other buffer set, a slice after each decode step's
    inputs on the same input stream, which runs ahead of the kernels; so they
    cross the link while this sweep's kernels run (sweep() with ``own=True``
    also copies its own prefill inputs first, layer by layer, as the first
    timed sweep must). A stream of their own for the prefetch measured slower:
    the decode steps' inputs then queued behind 34 MB copies. Outputs leave on
    a second side stream as soon as their layer (prefill) or engine step
    (decode) is done; decode outputs alternate between two buffers."""

    def __init__(self, wl: Workload):
        torch = wl.torch
        self.wl = wl
        dev = wl.meta[0][0].device
        u8, bf16 = torch.uint8, torch.bfloat16
        per_tok = E2E_BYTES_PER_TOKEN

        def host_bytes(nbytes):
            # random BF16 values, so that any float32 read of them is finite
            return torch.randn(nbytes // 2, dtype=bf16).view(u8).pin_memory()

        self.hp = [host_bytes(STEP_TOKENS * per_tok) for _ in range(LAYERS)]
        # dp[set][step][layer] -> (buf, x, za, zb); po[step][layer] -> o
        self.dp = [[[(lambda buf: (buf,) + packed_layer_inputs(buf, T))(
                        torch.empty(T * per_tok, dtype=u8, device=dev))
                     for _ in range(LAYERS)] for (_cu, _has, _first, _n, T) in wl.meta]
                   for _ in range(2)]
        self.po = [[torch.empty((T, HV, D), dtype=bf16, device=dev) for _ in range(LAYERS)]
                   for (_cu, _has, _first, _n, T) in wl.meta]
        self.hpo = [torch.empty((STEP_TOKENS, HV, D), dtype=bf16).pin_memory()
                    for _ in range(LAYERS)]
        per_layer = N_SEQS * per_tok
        self.hd = host_bytes(LAYERS * per_layer)
        self.dd = []                               # [decode step] -> (buf, xs, gates)
        for _ in range(DECODE_STEPS):
            buf = torch.empty(LAYERS * per_layer, dtype=u8, device=dev)
            xs, gs = [], []
            for l in range(LAYERS):
                x, za, zb = packed_layer_inputs(buf, N_SEQS, l * per_layer)
                xs.append(x)
                gs.append((za, zb))
            self.dd.append((buf, xs, gs))
        self.dout = [torch.empty((LAYERS, N_SEQS, HV, D), dtype=bf16, device=dev)
                     for _ in range(2)]
        self.hdo = torch.empty((LAYERS, N_SEQS, HV, D), dtype=bf16).pin_memory()
        self.hcu = [m[0].cpu().pin_memory() for m in wl.meta]
        self.hhas = [m[1].cpu().pin_memory() for m in wl.meta]
        self.cin = torch.cuda.Stream(device=dev)
        self.cout = torch.cuda.Stream(device=dev)
        self.h2d = 0
        self.d2h = 0

    def sweep(self, compute, use, prefetch, own):
        """Enqueue one sweep on ``compute`` (the stream being captured): the
        prefill kernels read input set ``use``; the next sweep's prefill inputs
        go to set ``prefetch``; with ``own`` this sweep first copies its own
        prefill inputs into set ``use``. Leaves the sweep's bytes in h2d, d2h."""
        wl, st, torch = self.wl, self.wl.stack, self.wl.torch
        cin, cout = self.cin, self.cout
        for s in (cin, cout):
            s.wait_stream(compute)
        h2d = d2h = 0

        def event(s):
            ev = torch.cuda.Event()
            ev.record(s)
            return ev

        # the next sweep's prefill inputs, a slice per decode step (their
        # buffers were last read by the previous sweep's kernels)
        items = [(i, l) for i in range(len(wl.meta)) for l in range(LAYERS)]
        for i, (cu, has, first, n, T) in enumerate(wl.meta):
            with torch.cuda.stream(cin):
                cu.copy_(self.hcu[i], non_blocking=True)
                has.copy_(self.hhas[i], non_blocking=True)
                h2d += cu.numel() * 4 + has.numel()
                meta_ready = event(cin)
            compute.wait_event(meta_ready)
            with torch.cuda.stream(compute):
                st.build_chunks(cu, T)
            for l in range(LAYERS):
                buf, x, za, zb = self.dp[use][i][l]
                o = self.po[i][l]
                if own:
                    with torch.cuda.stream(cin):
                        buf.copy_(self.hp[l][:buf.numel()], non_blocking=True)
                        h2d += buf.numel()
                        ready = event(cin)
                    compute.wait_event(ready)
                with torch.cuda.stream(compute):
                    st.prefill_layer(l, cu, has, first, n, x, za, zb, wl.py[l][:T], o)
                    done = event(compute)
                with torch.cuda.stream(cout):
                    cout.wait_event(done)
                    self.hpo[l][:T].copy_(o, non_blocking=True)
                    d2h += o.numel() * o.element_size()
        free = [None, None]
        for j in range(DECODE_STEPS):
            buf, xs, gs = self.dd[j]
            with torch.cuda.stream(cin):
                buf.copy_(self.hd, non_blocking=True)
                h2d += buf.numel()
                ready = event(cin)
                lo, hi = len(items) * j // DECODE_STEPS, len(items) * (j + 1) // DECODE_STEPS
                for (pi, pl) in items[lo:hi]:
                    pbuf = self.dp[prefetch][pi][pl][0]
                    pbuf.copy_(self.hp[pl][:pbuf.numel()], non_blocking=True)
                    h2d += pbuf.numel()
            compute.wait_event(ready)
            ob = self.dout[j & 1]
            if free[j & 1] is not None:
                compute.wait_event(free[j & 1])
            with torch.cuda.stream(compute):
                st.decode_step(xs, gs, wl.dy, [ob[l] for l in range(LAYERS)])
                done = event(compute)
            with torch.cuda.stream(cout):
                cout.wait_event(done)
                self.hdo.copy_(ob, non_blocking=True)
                d2h += ob.numel() * ob.element_size()
                free[j & 1] = event(cout)
        for s in (cin, cout):
            compute.wait_stream(s)
        self.h2d, self.d2h = h2d, d2h


# ----------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of the same workload
# ----------------------------------------------------------------------------

CPU_SAMPLE = ("float64 oracle, one layer: 32-seq decode step + 2x128-token prefill slice, "
              "per-token-layer times scaled to the 24-layer mix; 1 thread and 1 process/core")


def cpu_oracle_sample(seconds: float):
    """Oracle seconds per token-layer for decode and for prefill, on a sample
    of one layer of the mix (see CPU_SAMPLE); repeats until `seconds` spent."""
    from oracle import gdn_oracle as O
    from gated_deltanet_linear_build_gb300 import synth

    conv_d = synth.conv_update_case(11, N_SEQS, C)
    dd = synth.delta_case(12, [1] * N_SEQS, HK, HV, D, D, s0_std=0.02, normed_qk=False)
    conv_p = synth.conv_case(13, [128, 128], C, initial_state=False)
    dp = synth.delta_case(14, [128, 128], HK, HV, D, D, normed_qk=False)
    t_dec = t_pre = 0.0
    n_dec = n_pre = 0
    t_end = time.perf_counter() + seconds
    while time.perf_counter() < t_end or n_dec == 0:
        t0 = time.perf_counter()
        O.causal_conv1d_update(conv_d["x"], conv_d["w"], None, conv_d["conv_state"])
        O.delta_rule_decode(dd["q"], dd["k"], dd["v"], dd["a"], dd["b"], dd["S0"], qk_l2norm=True)
        t1 = time.perf_counter()
        O.causal_conv1d_fwd(conv_p["x"], conv_p["w"], None, conv_p["conv_state"],
                            conv_p["has_initial_state"], conv_p["cu_seqlens"])
        O.delta_rule_prefill(dp["q"], dp["k"], dp["v"], dp["a"], dp["b"], dp["cu_seqlens"],
                             dp["S0"], dp["has_initial_state"], qk_l2norm=True)
        t2 = time.perf_counter()
        t_dec += t1 - t0
        t_pre += t2 - t1
        n_dec += N_SEQS
        n_pre += 256
    return t_dec / n_dec, t_pre / n_pre, t_dec + t_pre


def mix_tokens_per_s(per_dec, per_pre, prefill_tokens, decode_tokens):
    t = LAYERS * (prefill_tokens * per_pre + decode_tokens * per_dec)
    return (prefill_tokens + decode_tokens) / t


def _oracle_worker(seconds):
    return cpu_oracle_sample(seconds)


def cpu_oracle_all_cores(seconds: float, prefill_tokens: int, decode_tokens: int):
    """The same sample on every host core at once: one worker process per core
    (started with 'spawn', so none inherits a CUDA context; one BLAS/OpenMP
    thread each), each timing its own share under the full load. Returns
    (tokens/s of the mix summed over the workers, workers, wall seconds)."""
    import multiprocessing as mp
    procs = os.cpu_count() or 1
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                            "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        t0 = time.perf_counter()
        with mp.get_context("spawn").Pool(procs) as pool:
            res = pool.map(_oracle_worker, [seconds] * procs)
        wall = time.perf_counter() - t0
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    total = sum(mix_tokens_per_s(pd, pp, prefill_tokens, decode_tokens) for pd, pp, _ in res)
    return total, procs, wall


def run_reference(args):
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    from gated_deltanet_linear_build_gb300 import synth
    pre = int(sum(int(x) for x in synth.serving_mix_lengths(rank_lengths_seed(0))))
    dec = DECODE_STEPS * N_SEQS
    per_step = max(1.0, min(args.cpu_seconds, 20.0))
    for _ in range(args.warmup):
        cpu_oracle_sample(0.0)
    vals, secs = [], []
    cores = 1
    for _ in range(args.steps):
        t0 = time.perf_counter()
        v, cores, _ = cpu_oracle_all_cores(per_step / 2, pre, dec)
        secs.append(time.perf_counter() - t0)
        vals.append(v)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(secs), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": CPU_SAMPLE},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": CPU_SAMPLE},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(compact(line)), flush=True)
    return 0


# ----------------------------------------------------------------------------
# The GPU arm
# ----------------------------------------------------------------------------

def kernel_report(wl, kind_ms, hbm_peak, bf16_peak):
    """Per kind: launches, average duration, share of the sweep, and achieved
    rate against its roofline (algorithmic work / average duration).
    kind_ms[k] is the device time of all of a sweep's calls of kind k; these
    kernels run inside a seconds-long replay, so bf16_peak should be the
    sustained tensor peak."""
    rep = {}
    total = sum(kind_ms.values())
    n_steps = len(wl.steps)
    chunk_fl = prefill_flops(wl.chunk_lengths()) / n_steps
    work = {
        "delta_decode": ("hbm", decode_delta_bytes()),
        "conv_update": ("hbm", conv_update_bytes()),
        "conv_prefill": ("hbm", sum(conv_prefill_bytes(st.tokens, len(st.segments))
                                    for st in wl.steps) / n_steps),
        "delta_prefill": ("tensor", chunk_fl),
    }
    for k in KINDS:
        n = wl.kind_launches(k)
        avg = kind_ms[k] / n
        r = {"launches": n, "avg_us": avg * 1e3, "share": kind_ms[k] / total if total else None}
        if k in work:
            bound, amount = work[k]
            if bound == "hbm":
                ach = amount / (avg / 1e3) / 1e9
                r.update(bound="hbm", achieved=ach, unit="GB/s", peak=hbm_peak,
                         frac=ach / hbm_peak, algorithmic_per_launch=amount)
            else:
                ach = amount / (avg / 1e3) / 1e12
                r.update(bound="tensor", achieved=ach, unit="TFLOP/s", peak=bf16_peak,
                         frac=ach / bf16_peak, algorithmic_per_launch=amount)
        rep[k] = r
    return rep


def run_gdn(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    from gated_deltanet_linear_build_gb300 import build as B
    B.build_library()
    from gated_deltanet_linear_build_gb300 import gdn
    gdn.load_library()

    hbm_peak, _bf16_burst, bf16_sus, peak_src = load_peaks()
    wl = Workload(rank, dev)
    stream = torch.cuda.Stream(device=dev)

    with torch.cuda.stream(stream):
        wl.sweep()                      # eager warm run (sets kernel attributes)
    torch.cuda.synchronize()
    launches_before = wl.stack.launches
    graph = torch.cuda.CUDAGraph()      # the timed sweep: kernels only
    with torch.cuda.graph(graph, stream=stream):
        wl.sweep()
    launches_per_sweep = wl.stack.launches - launches_before
    kind_graphs = {}                    # the same calls grouped by kind, one graph each
    for k in KINDS:
        with torch.cuda.stream(stream):
            wl.kind_sweep(k)
        torch.cuda.synchronize()
        kind_graphs[k] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(kind_graphs[k], stream=stream):
            wl.kind_sweep(k)

    # Replays go to the stream the events are recorded on.
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
        for k in KINDS:
            kind_graphs[k].replay()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    kev = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for k in KINDS}
    with ClockSampler(local) as clocks, torch.cuda.stream(stream):
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(args.steps - 1):
            graph.replay()
        # The last timed step makes the same calls grouped by kind, with events
        # around each group: per-kind launch durations without per-call events.
        for k in KINDS:
            kev[k][0].record(stream)
            kind_graphs[k].replay()
            kev[k][1].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    ms = start.elapsed_time(end) / args.steps
    ms_max = reduce_over_ranks(ms, "max", dist, dev)
    tokens_all = reduce_over_ranks(float(wl.tokens), "sum", dist, dev)
    value = tokens_all / (ms_max / 1e3)
    kind_ms = {k: kev[k][0].elapsed_time(kev[k][1]) for k in KINDS}

    # in-sweep kernels: the sustained BF16 peak (a seconds-long loop under the
    # power cap), the HBM copy peak
    kernels = kernel_report(wl, kind_ms, hbm_peak, bf16_sus)
    roofline = None
    if kernels:
        dom = max((k for k in kernels if "bound" in kernels[k]),
                  key=lambda k: kernels[k]["share"])
        r = kernels[dom]
        roofline = {"kernel": dom, "bound": r["bound"], "achieved": r["achieved"],
                    "peak": r["peak"], "unit": r["unit"], "frac": r["frac"],
                    "peak_source": peak_src, "share_of_sweep": r["share"],
                    "avg_launch_us": r["avg_us"], "launches_timed": r["launches"],
                    "algorithmic_per_launch": r["algorithmic_per_launch"],
                    "traffic": stored_traffic(dom)}

    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "layers": LAYERS, "seqs_per_gpu": N_SEQS,
                   "prefill_tokens": wl.prefill_tokens, "decode_tokens": wl.decode_tokens,
                   "prefill_steps": len(wl.steps), "step_tokens": STEP_TOKENS,
                   "conv_channels": C, "v_heads": HV, "qk_heads": HK, "head_dim": D,
                   "l2": "inputs > L2 (~11 GB of distinct layer inputs per sweep)",
                   "timing": "sweep graph x (K-1) + per-kind graphs x 1, CUDA events on the "
                             "launch stream around all K",
                   "parallelism": f"dp{world} (independent sequences per GPU)"},
        "roofline": roofline,
        "kernels": kernels,
        "gpu_launches": launches_per_sweep * args.steps,
        "clocks": clocks.summary(),
    }

    if not args.no_e2e:
        e2 = E2EWorkload(wl)
        with torch.cuda.stream(stream):
            e2.sweep(stream, use=0, prefetch=1, own=True)      # eager warm run
        torch.cuda.synchronize()
        # g_first copies its own prefill inputs (set 0) and prefetches set 1;
        # then g_a (reads 1, prefetches 0) and g_b (reads 0, prefetches 1)
        # alternate. Every timed sweep's inputs cross the link inside the
        # timed region: the first sweep's before its kernels, the others'
        # during the sweep before them.
        graphs, moved = {}, {}
        for name, use, pre, own in (("first", 0, 1, True), ("a", 1, 0, False),
                                    ("b", 0, 1, False)):
            graphs[name] = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graphs[name], stream=stream):
                e2.sweep(stream, use=use, prefetch=pre, own=own)
            moved[name] = (e2.h2d, e2.d2h)
        order = ["first"] + ["a" if k % 2 else "b" for k in range(1, args.steps)]
        with torch.cuda.stream(stream):
            for _ in range(max(1, args.warmup)):
                for name in ("first", "a", "b"):
                    graphs[name].replay()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        s2, e2_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            s2.record(stream)
            for name in order:
                graphs[name].replay()
            e2_.record(stream)
        torch.cuda.synchronize()
        ms2 = reduce_over_ranks(s2.elapsed_time(e2_) / args.steps, "max", dist, dev)
        out["e2e"] = {"value": tokens_all / (ms2 / 1e3), "unit": "tokens/s",
                      "h2d_bytes_per_step": sum(moved[n][0] for n in order) // len(order),
                      "d2h_bytes_per_step": sum(moved[n][1] for n in order) // len(order),
                      "ms_per_step": ms2,
                      "path": "C-ABI calls; pinned host <-> device copies in the graph, one per "
                              "prefill layer and per decode step each way; the next sweep's "
                              "prefill inputs are prefetched during this sweep's decode steps "
                              "(double buffered); the first timed sweep copies its own"}

    if rank == 0 and not args.no_cpu_baseline:
        pd, pp, spent = cpu_oracle_sample(args.cpu_seconds / 2)
        one = mix_tokens_per_s(pd, pp, wl.prefill_tokens, wl.decode_tokens)
        allc, cores, wall = cpu_oracle_all_cores(args.cpu_seconds / 2, wl.prefill_tokens,
                                                 wl.decode_tokens)
        out["cpu_baseline"] = {
            "value": allc, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": CPU_SAMPLE, "one_thread_value": one,
            "cpu_seconds": spent + wall * cores}
    if rank == 0:
        print(json.dumps(compact(out)), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_case(args):
    """Time one hot-path call on its own workload shape, cycling through input
    sets whose total exceeds twice the L2 size, CUDA events on the stream."""
    import torch
    from gated_deltanet_linear_build_gb300 import build as B, gdn
    B.build_library()
    gdn.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    hbm_peak, bf16_peak, _, peak_src = load_peaks()
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    bf16 = torch.bfloat16
    L2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def randn(*shape, dtype=torch.float32):
        return torch.randn(shape, generator=g, device=dev, dtype=dtype)

    def gates(T):
        # raw gate logits; the kernels activate them (GDN_FLAG_GATE_LOGITS)
        return randn(T, HV).contiguous(), randn(T, HV).contiguous()

    case = args.case
    if case == "conv_prefill":
        T, n = 2048, 2
        cu = torch.tensor([0, 1024, 2048], dtype=torch.int32, device=dev)
        has = torch.zeros(n, dtype=torch.uint8, device=dev)
        chunks = torch.empty((T // 8 + n, 4), dtype=torch.int32, device=dev)
        cnt = torch.empty(1, dtype=torch.int32, device=dev)
        gdn.build_conv_chunks(cu, chunks, cnt, chunk_tokens=8)
        per = conv_prefill_bytes(T, n)
        sets = [(randn(T, C, dtype=bf16), (randn(C, 4) * 0.5).to(bf16),
                 torch.zeros((n, C, 3), dtype=bf16, device=dev),
                 torch.empty((T, C), dtype=bf16, device=dev))
                for _ in range(max(2, int(2 * L2 // per) + 1))]

        def call(i):
            x, w, st, y = sets[i % len(sets)]
            gdn.causal_conv1d_fwd(x, w, None, st, has, cu, y, chunks=chunks, num_chunks=cnt)
        work, unit, bound = per, "GB/s", "hbm"
    elif case == "conv_update":
        per = conv_update_bytes()
        sets = [(randn(N_SEQS, C, dtype=bf16), (randn(C, 4) * 0.5).to(bf16),
                 randn(N_SEQS, C, 3, dtype=bf16), torch.empty((N_SEQS, C), dtype=bf16, device=dev))
                for _ in range(int(2 * L2 // per) + 1)]

        def call(i):
            x, w, st, y = sets[i % len(sets)]
            gdn.causal_conv1d_update(x, w, None, st, y)
        work, unit, bound = per, "GB/s", "hbm"
    elif case == "decode":
        per = decode_delta_bytes()
        sets = []
        for _ in range(int(2 * L2 // per) + 1):
            y = randn(N_SEQS, C, dtype=bf16)
            a, b = gates(N_SEQS)
            sets.append((y, a, b, randn(N_SEQS, HV, D, D) * 0.02,
                         torch.empty((N_SEQS, HV, D), dtype=bf16, device=dev)))

        def call(i):
            y, a, b, S, o = sets[i % len(sets)]
            q = y[:, :HK * D].view(N_SEQS, HK, D)
            k = y[:, HK * D:2 * HK * D].view(N_SEQS, HK, D)
            v = y[:, 2 * HK * D:].view(N_SEQS, HV, D)
            gdn.delta_rule_decode(q, k, v, a, b, S, o, qk_l2norm=True, gate_logits=True)
        work, unit, bound = per, "GB/s", "hbm"
    else:  # prefill: 2 x 1024 tokens, 32 v-heads over 16 k-heads, d = 128
        T, n = 2048, 2
        cu = torch.tensor([0, 1024, 2048], dtype=torch.int32, device=dev)
        has = torch.zeros(n, dtype=torch.uint8, device=dev)
        ws = torch.empty(gdn.delta_rule_prefill_workspace_size(T, n, HV, D, D), dtype=torch.uint8,
                         device=dev)
        sets = []
        for _ in range(2):
            y = randn(T, C, dtype=bf16)
            a, b = gates(T)
            sets.append((y, a, b, torch.zeros((n, HV, D, D), device=dev),
                         torch.empty((T, HV, D), dtype=bf16, device=dev)))

        def call(i):
            y, a, b, S, o = sets[i % len(sets)]
            q = y[:, :HK * D].view(T, HK, D)
            k = y[:, HK * D:2 * HK * D].view(T, HK, D)
            v = y[:, 2 * HK * D:].view(T, HV, D)
            gdn.delta_rule_prefill_chunked(q, k, v, a, b, cu, S, has, o, ws, qk_l2norm=True,
                                           gate_logits=True)
        work, unit, bound = prefill_flops([64] * 32), "TFLOP/s", "tensor"

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            call(i)
        torch.cuda.synchronize()
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_ev.record(stream)
        for i in range(args.steps):
            call(i)
        e_ev.record(stream)
        torch.cuda.synchronize()
    us = s_ev.elapsed_time(e_ev) * 1e3 / args.steps
    scale = 1e9 if unit == "GB/s" else 1e12
    ach = work / (us / 1e6) / scale
    peak = hbm_peak if bound == "hbm" else bf16_peak
    print(json.dumps({"case": case, "avg_us_per_call": us, "bound": bound, "achieved": ach,
                      "unit": unit, "peak": peak, "frac": ach / peak, "peak_source": peak_src,
                      "algorithmic_per_call": work, "steps": args.steps,
                      "input_sets": len(sets)}), flush=True)
    return 0


def time_graph(torch, stream, enqueue, steps, warmup):
    """Capture ``enqueue()`` once as a CUDA graph on ``stream``; return the
    average replay time in ms (CUDA events on that stream)."""
    with torch.cuda.stream(stream):
        enqueue()                              # eager run (kernel attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        enqueue()
    with torch.cuda.stream(stream):
        for _ in range(max(3, warmup)):
            g.replay()
        torch.cuda.synchronize()
        s_ev = torch.cuda.Event(enable_timing=True)
        e_ev = torch.cuda.Event(enable_timing=True)
        s_ev.record(stream)
        for _ in range(steps):
            g.replay()
        e_ev.record(stream)
        torch.cuda.synchronize()
    return s_ev.elapsed_time(e_ev) / steps


def run_decode_units(args):
    """The decode (d = 128, 32 v-heads over 16 k-heads, gate logits, q/k L2
    norm) at several sequence counts, as graphs of 48 calls cycling over
    states whose total exceeds L2: one JSON line per count with the 64-row
    units per persistent CTA, us per launch and the fraction of the measured
    HBM peak."""
    import torch
    from gated_deltanet_linear_build_gb300 import build as B, gdn
    B.build_library()
    gdn.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    hbm_peak = load_peaks()[0]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    stream = torch.cuda.Stream(device=dev)
    calls = 48
    for n in (16, 19, 24, 32, 38, 48, 57, 64):
        per = decode_delta_bytes(n)
        nsets = max(3, int(400e6 // per) + 1)
        sets = []
        for _ in range(nsets):
            y = torch.randn((n, C), generator=g, device=dev).to(torch.bfloat16)
            sets.append((y, torch.randn((n, HV), generator=g, device=dev),
                         torch.randn((n, HV), generator=g, device=dev),
                         torch.randn((n, HV, D, D), generator=g, device=dev) * 0.02,
                         torch.empty((n, HV, D), dtype=torch.bfloat16, device=dev)))

        def enqueue():
            for i in range(calls):
                y, a, b, S, o = sets[i % nsets]
                gdn.delta_rule_decode(y[:, :HK * D].view(n, HK, D),
                                      y[:, HK * D:2 * HK * D].view(n, HK, D),
                                      y[:, 2 * HK * D:].view(n, HV, D), a, b, S, o,
                                      qk_l2norm=True, gate_logits=True)
        us = time_graph(torch, stream, enqueue, max(1, args.steps // 4), args.warmup) \
            * 1e3 / calls
        units = n * HV * 2
        print(json.dumps(compact({"case": "decode_units", "seqs": n, "units": units,
                                  "units_per_cta": units / sms, "us_per_launch": us,
                                  "achieved_gbs": per / us / 1e3,
                                  "frac": per / us / 1e3 / hbm_peak})), flush=True)
        del sets
        torch.cuda.empty_cache()
    return 0


def run_step_case(args):
    """decode_step: one decode step of 24 layers (N = 32 sequences), as
    gdn_causal_conv1d_update + gdn_delta_rule_decode per layer against
    gdn_decode_step_fused per layer. mixed_step: one 2048-token engine step of
    24 layers carrying two prefill segments (1008 tokens each) and 32 decode
    tokens, as one descriptor build + one conv prefill + one chunked prefill
    per layer (the decode tokens ride the prefill calls as one-token
    sequences) against the same prefill calls on the segments plus a conv
    update + decode per layer for the decode tokens. Each variant is one CUDA
    graph over distinct per-layer weights and states, replayed; inputs are
    raw gate logits, q/k L2-normalised in the kernel."""
    import torch
    from gated_deltanet_linear_build_gb300 import build as B, gdn
    B.build_library()
    gdn.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    bf16 = torch.bfloat16
    stream = torch.cuda.Stream(device=dev)

    def randn(*shape, dtype=torch.float32, std=1.0):
        return (torch.randn(shape, generator=g, device=dev) * std).to(dtype)

    def views(y):
        T = y.shape[0]
        return (y[:, :HK * D].view(T, HK, D), y[:, HK * D:2 * HK * D].view(T, HK, D),
                y[:, 2 * HK * D:].view(T, HV, D))

    W = [randn(C, 4, dtype=bf16, std=0.5) for _ in range(LAYERS)]
    out = {"case": args.case, "layers": LAYERS, "steps": args.steps}
    if args.case == "decode_step":
        N = N_SEQS
        X = [randn(N, C, dtype=bf16) for _ in range(LAYERS)]
        ZA = [randn(N, HV) for _ in range(LAYERS)]
        ZB = [randn(N, HV) for _ in range(LAYERS)]
        S = [randn(N, HV, D, D, std=0.02) for _ in range(LAYERS)]
        ST = [[randn(N, C, 3, dtype=bf16) for _ in range(LAYERS)] for _ in range(2)]
        Y = torch.empty((N, C), dtype=bf16, device=dev)
        O = torch.empty((N, HV, D), dtype=bf16, device=dev)
        par = [0]

        def two_calls():
            for l in range(LAYERS):
                gdn.causal_conv1d_update(X[l], W[l], None, ST[0][l], Y)
                q, k, v = views(Y)
                gdn.delta_rule_decode(q, k, v, ZA[l], ZB[l], S[l], O, qk_l2norm=True,
                                      gate_logits=True)

        def fused():
            # the fused step updates the conv state out of place: alternate buffers
            for rep in range(2):
                for l in range(LAYERS):
                    gdn.decode_step_fused(X[l], W[l], None, ST[rep][l], ST[1 - rep][l], ZA[l],
                                          ZB[l], S[l], O, Hk=HK, qk_l2norm=True,
                                          gate_logits=True)

        t2 = time_graph(torch, stream, two_calls, args.steps, args.warmup) / LAYERS
        tf = time_graph(torch, stream, fused, args.steps, args.warmup) / (2 * LAYERS)
        out.update(unit="us per layer-step (32 sequences)", two_calls=1e3 * t2,
                   fused=1e3 * tf, fused_over_two_calls=tf / t2,
                   delta_bytes_per_layer_step=decode_delta_bytes(),
                   conv_bytes_per_layer_step=conv_update_bytes())
    else:
        seg, nd = 1008, N_SEQS
        T = 2 * seg + nd
        lens = [seg, seg] + [1] * nd
        cu_list = [0]
        for L in lens:
            cu_list.append(cu_list[-1] + L)
        cu_m = torch.tensor(cu_list, dtype=torch.int32, device=dev)
        cu_p = torch.tensor([0, seg, 2 * seg], dtype=torch.int32, device=dev)
        has_m = torch.ones(2 + nd, dtype=torch.uint8, device=dev)
        has_p = torch.ones(2, dtype=torch.uint8, device=dev)
        X = [randn(T, C, dtype=bf16) for _ in range(LAYERS)]
        ZA = [randn(T, HV) for _ in range(LAYERS)]
        ZB = [randn(T, HV) for _ in range(LAYERS)]
        S = [randn(2 + nd, HV, D, D, std=0.02) for _ in range(LAYERS)]
        ST = [randn(2 + nd, C, 3, dtype=bf16) for _ in range(LAYERS)]
        Y = torch.empty((T, C), dtype=bf16, device=dev)
        O = torch.empty((T, HV, D), dtype=bf16, device=dev)
        ch = torch.empty((T // 8 + 2 + nd, 4), dtype=torch.int32, device=dev)
        cnt = torch.empty(1, dtype=torch.int32, device=dev)
        ws = torch.empty(gdn.delta_rule_prefill_workspace_size(T, 2 + nd, HV, D, D),
                         dtype=torch.uint8, device=dev)
        P = 2 * seg

        def mixed():
            gdn.build_conv_chunks(cu_m, ch, cnt, chunk_tokens=8)
            for l in range(LAYERS):
                gdn.causal_conv1d_fwd(X[l], W[l], None, ST[l], has_m, cu_m, Y, chunks=ch,
                                      num_chunks=cnt)
                q, k, v = views(Y)
                gdn.delta_rule_prefill_chunked(q, k, v, ZA[l], ZB[l], cu_m, S[l], has_m, O, ws,
                                               qk_l2norm=True, gate_logits=True)

        def separate():
            gdn.build_conv_chunks(cu_p, ch, cnt, chunk_tokens=8)
            for l in range(LAYERS):
                gdn.causal_conv1d_fwd(X[l][:P], W[l], None, ST[l][:2], has_p, cu_p, Y[:P],
                                      chunks=ch, num_chunks=cnt)
                q, k, v = views(Y[:P])
                gdn.delta_rule_prefill_chunked(q, k, v, ZA[l][:P], ZB[l][:P], cu_p, S[l][:2],
                                               has_p, O[:P], ws, qk_l2norm=True,
                                               gate_logits=True)
                gdn.causal_conv1d_update(X[l][P:], W[l], None, ST[l][2:], Y[P:])
                qd, kd, vd = views(Y[P:])
                gdn.delta_rule_decode(qd, kd, vd, ZA[l][P:], ZB[l][P:], S[l][2:], O[P:],
                                      qk_l2norm=True, gate_logits=True)

        tm = time_graph(torch, stream, mixed, args.steps, args.warmup)
        ts = time_graph(torch, stream, separate, args.steps, args.warmup)
        out.update(unit="ms per 24-layer engine step", tokens=T, prefill_tokens=P,
                   decode_tokens=nd, mixed=tm, separate=ts, mixed_over_separate=tm / ts,
                   mixed_us_per_token_layer=1e3 * tm / (T * LAYERS),
                   separate_us_per_token_layer=1e3 * ts / (T * LAYERS))
    print(json.dumps(out), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.case in ("decode_step", "mixed_step"):
        return run_step_case(args)
    if args.case == "decode_units":
        return run_decode_units(args)
    if args.case != "mix":
        return run_case(args)
    return run_gdn(args)


if __name__ == "__main__":
    sys.exit(main())
