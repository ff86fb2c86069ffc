"""Benchmark: effective weight bandwidth of the skinny decode linears on GB300.

One step = one decode round of the 27B-shaped model's linear layers, at M
tokens (default 8, the k=7 speculative verify round; --m 1 for plain decode):

    64 x { qkv (FP8, K=5120 N=7168), o_proj (FP8, K=6144 N=5120),
           gate_up (NVFP4, K=5120 N=34816), down (NVFP4, K=17408 N=5120) }
    + lm_head (NVFP4, K=5120 N=151936) with the fused greedy argmax and, at
      M > 1, the greedy verification of the M - 1 drafted tokens

i.e. 257 calls of the C ABI, captured once into a CUDA graph and replayed.
Weights (14.43 GB per step) are synthetic, generated on the device with the
same distributions the tests use, and far larger than L2, so every replay
streams them from HBM.  Metric: weight bytes (codes + scales + tensor scale)
per second.

Also measured: the same step at the other token count over the same weights
(M = 1 next to the verify round: `stack_m1`), the dominant kernel alone (the
NVFP4 gate_up launch, rotating over 8 weight copies = 802 MB so L2 is cold) for
the roofline, the small NVFP4 GEMV (K=512, N=256, L2-resident: `c0`), a
per-layer table with cold L2 at M = 1 and 8 (full and 4-way tensor-parallel
per-rank shapes), the quantizers and the sampled lm_head, and the end-to-end
rate through the C ABI with the activations (and drafted tokens) copied from
pinned host memory and the picks (and the round's verdict) read back every
step.  The CPU oracle is timed on a bounded sample with all host threads and
with one.  --impl reference times the CPU oracle on a bounded sample.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# (name, format, K, N) of one decoder layer, then the vocabulary projection.
LAYER = [("qkv", "fp8", 5120, 7168), ("o_proj", "fp8", 6144, 5120),
         ("gate_up", "nvfp4", 5120, 34816), ("down", "nvfp4", 17408, 5120)]
LM_HEAD = ("lm_head", "nvfp4", 5120, 151936)
N_LAYERS = 64
# The pages quote their kernels at the per-rank shapes of 4-way tensor
# parallelism: qkv, gate_up and the lm_head split over N, o_proj and down over K.
TP_WORLD = 4
TP_AXIS = {"qkv": "n", "o_proj": "k", "gate_up": "n", "down": "k", "lm_head": "n"}


def tp_shape(name, K, N, world=TP_WORLD):
    return (K, N // world) if TP_AXIS[name] == "n" else (K // world, N)


def weight_bytes(fmt: str, K: int, N: int) -> int:
    if fmt == "nvfp4":
        return N * K // 2 + N * K // 16 + 4
    return N * K + 4 * ((N + 127) // 128) * ((K + 127) // 128)


STEP_BYTES = N_LAYERS * sum(weight_bytes(f, K, N) for _, f, K, N in LAYER) + weight_bytes(*LM_HEAD[1:])


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------- clocks ---

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- workload ---

def make_weights(fmt, K, N, gen, dev):
    """Synthetic weights on the device (same recipes as the tests' generator)."""
    import torch

    if fmt == "nvfp4":
        codes = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=dev, generator=gen)
        scales = torch.randint(0x18, 0x59, (N, K // 16), dtype=torch.uint8, device=dev, generator=gen)
        return codes, scales, 0.01
    # FP8: N(0, 0.02) -> absmax/448 per 128x128 block -> E4M3 (RNE, saturated)
    w = torch.randn((N, K), dtype=torch.float32, device=dev, generator=gen) * 0.02
    nb, kb = (N + 127) // 128, (K + 127) // 128
    wp = torch.zeros((nb * 128, kb * 128), dtype=torch.float32, device=dev)
    wp[:N, :K] = w
    del w
    blk = wp.view(nb, 128, kb, 128)
    amax = blk.abs().amax(dim=(1, 3))
    scales = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).contiguous()
    q = (blk / scales[:, None, :, None]).clamp_(-448.0, 448.0).view(nb * 128, kb * 128)[:N, :K]
    codes = q.contiguous().to(torch.float8_e4m3fn).view(torch.uint8)
    del wp, blk, q
    return codes, scales, None


class Linear:
    def __init__(self, name, fmt, K, N, M, gen, dev, out_f16=True):
        import torch

        self.name, self.fmt, self.K, self.N, self.M = name, fmt, K, N, M
        self.codes, self.scales, self.g = make_weights(fmt, K, N, gen, dev)
        self.x = torch.randn((M, K), generator=gen, device=dev).to(torch.float16)
        self.y = torch.empty((M, N), dtype=torch.float16 if out_f16 else torch.float32, device=dev)
        self.bytes = weight_bytes(fmt, K, N)

    def at_m(self, M, gen, dev):
        """The same weights with M activation rows of its own (another step
        shape over the weights already in device memory)."""
        import copy

        import torch

        o = copy.copy(self)
        o.M = M
        o.x = torch.randn((M, self.K), generator=gen, device=dev).to(torch.float16)
        o.y = torch.empty((M, self.N), dtype=self.y.dtype, device=dev)
        return o

    def call(self, sk, x=None):
        x = self.x if x is None else x
        if self.fmt == "nvfp4":
            sk.nvfp4_gemm(x, self.codes, self.scales, self.g, y=self.y, f16_out=self.y.dtype.itemsize == 2)
        else:
            sk.fp8_gemm(x, self.codes, self.scales, y=self.y, f16_out=self.y.dtype.itemsize == 2)


class LMHead(Linear):
    """The vocabulary projection with its fused greedy pick; at M > 1 (the
    speculative verify round) it also verifies M - 1 drafted tokens."""

    def __init__(self, M, gen, dev):
        import torch

        super().__init__(*LM_HEAD, M, gen, dev, out_f16=False)
        self.am = torch.empty((M,), dtype=torch.int32, device=dev)
        self.draft = torch.randint(0, LM_HEAD[3], (max(M - 1, 1),), generator=gen, device=dev,
                                   dtype=torch.int32)
        self.accept = torch.empty((2,), dtype=torch.int32, device=dev)

    def at_m(self, M, gen, dev):
        import torch

        o = super().at_m(M, gen, dev)
        o.am = torch.empty((M,), dtype=torch.int32, device=dev)
        o.draft = torch.randint(0, LM_HEAD[3], (max(M - 1, 1),), generator=gen, device=dev, dtype=torch.int32)
        o.accept = torch.empty((2,), dtype=torch.int32, device=dev)
        return o

    def call(self, sk, x=None):
        x = self.x if x is None else x
        if self.M > 1:
            sk.lm_head_verify(x, self.codes, self.scales, self.g, self.draft, logits=self.y, argmax=self.am,
                              accept=self.accept)
        else:
            sk.lm_head_argmax(x, self.codes, self.scales, self.g, logits=self.y, argmax=self.am)


def time_graph(graph, stream, reps, warmup, barrier=None):
    import torch

    with torch.cuda.stream(stream):          # replay() launches on the current stream
        for _ in range(warmup):
            graph.replay()
        stream.synchronize()
        if barrier:
            barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
        e1.synchronize()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps        # ms per replay


def capture(fn, stream):
    import torch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()                                  # warm-up outside the capture (attributes, maps)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn()
    return g


def layer_table(sk, gen, dev, stream, peak, tp=False):
    """Per-layer cold-L2 rates, both formats (the lm_head in NVFP4): at the full
    shapes for M = 1, 2, 4 and 8, at the per-rank shapes of 4-way tensor
    parallelism for M = 1 and 8."""
    rows = []
    for mm in ((1, 8) if tp else (1, 2, 4, 8)):
        for name, f, K, N in LAYER + [LM_HEAD]:
            Ks, Ns = tp_shape(name, K, N) if tp else (K, N)
            for fmt in ((f,) if name == "lm_head" else ("nvfp4", "fp8")):
                t_ms, b = cold_layer_rate(sk, fmt, Ks, Ns, mm, gen, dev, stream)
                gbs = b / (t_ms * 1e-3) / 1e9
                rows.append({"layer": name, "fmt": fmt, "M": mm, "K": Ks, "N": Ns, "us": round(t_ms * 1e3, 2),
                             "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 3)})
    return rows


def quant_rates(sk, gen, dev, stream, peak, K=5120, N=34816, reps=10):
    """The GPU quantizers on one FP16 weight of the gate_up shape (356 MB, far
    above L2).  Algorithmic bytes: the FP16 weight read (twice for NVFP4, whose
    codes need the tensor maximum first) plus the codes and scales written."""
    import torch

    w = (torch.randn((N, K), generator=gen, device=dev) * 0.02).to(torch.float16)
    fp8_bytes = 2 * N * K + N * K + 4 * ((N + 127) // 128) * ((K + 127) // 128)
    nv_bytes = 2 * 2 * N * K + N * K // 2 + N * K // 16 + 4
    rows = []
    for name, fn, b in (("fp8_quantize", lambda: sk.fp8_quantize(w), fp8_bytes),
                        ("nvfp4_quantize", lambda: sk.nvfp4_quantize(w), nv_bytes)):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            e1.synchronize()
        us = e0.elapsed_time(e1) / reps * 1e3
        gbs = b / (us * 1e-6) / 1e9
        rows.append({"op": name, "K": K, "N": N, "us": round(us, 2), "bytes": b, "GB/s": round(gbs, 1),
                     "frac_of_peak": round(gbs / peak, 3)})
    del w
    torch.cuda.empty_cache()
    return rows


def sampler_cost(sk, gen, dev, stream, M=8, reps=10, T=0.6, top_k=50, top_p=0.9):
    """The full-vocabulary lm_head with the sampled pick (temperature 0.6,
    top-k 50, top-p 0.9) against the same projection with the greedy pick, at
    M rows, per call (the weights are far above L2)."""
    import torch

    K, N = LM_HEAD[2], LM_HEAD[3]
    head = LMHead(M, gen, dev)
    u = torch.rand((M,), generator=gen, device=dev)
    tok = torch.empty((M,), dtype=torch.int32, device=dev)
    out = {}
    for name, fn in (("argmax", lambda: sk.lm_head_argmax(head.x, head.codes, head.scales, head.g, logits=head.y,
                                                          argmax=head.am)),
                     ("sample", lambda: sk.lm_head_sample(head.x, head.codes, head.scales, head.g, u, T, top_k,
                                                          top_p, logits=head.y, token=tok))):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            e1.synchronize()
        out[name + "_us"] = round(e0.elapsed_time(e1) / reps * 1e3, 2)
    del head
    torch.cuda.empty_cache()
    return {"M": M, "K": K, "N": N, "temperature": T, "top_k": top_k, "top_p": top_p, **out}


def cold_layer_rate(sk, fmt, K, N, M, gen, dev, stream, copies=None):
    """Per-launch time of one layer with a cold L2: a graph of back-to-back
    launches over enough distinct weight copies (>= 4x L2 in total)."""
    import torch

    b = weight_bytes(fmt, K, N)
    if copies is None:
        copies = max(4, min(32, int(-(-4 * 130e6 // b))))
    lins = [Linear("l", fmt, K, N, M, gen, dev) for _ in range(copies)]
    g = capture(lambda: [ln.call(sk) for ln in lins], stream)
    ms = time_graph(g, stream, reps=10, warmup=3) / copies
    del g, lins
    torch.cuda.empty_cache()
    return ms, b


# ------------------------------------------------------------------- arms ---

def oracle_sample_inputs(M, cols):
    """Synthetic inputs for `cols` output columns of every linear type at full K."""
    import synth

    out = []
    for i, (_, f, K, N) in enumerate([*LAYER, LM_HEAD]):
        x = synth.x_f16(M, K, seed=1000 + i)
        if f == "nvfp4":
            c, s, g = synth.nvfp4_weights(cols, K, seed=2000 + i)
            out.append((f, x, (c, s, g), cols * weight_bytes(f, K, 1)))
        else:
            c, s = synth.fp8_weights(cols, K, seed=2000 + i)
            out.append((f, x, (c, s), cols * (K + 4 * ((K + 127) // 128))))
    return out


def oracle_pass(sample):
    """One pass of the CPU oracle over a sample; returns (weight bytes, seconds)."""
    import oracle

    nbytes, t0 = 0, time.perf_counter()
    for f, x, w, b in sample:
        if f == "nvfp4":
            oracle.nvfp4_linear(x, *w)
        else:
            oracle.fp8_linear(x, *w)
        nbytes += b
    return nbytes, time.perf_counter() - t0


def size_oracle_sample(M, budget_s):
    """Grow the sampled columns until one oracle pass takes >= budget_s (at most
    one extrapolated jump after a small timing pass; capped at 32768 columns)."""
    cols = 64
    while True:
        sample = oracle_sample_inputs(M, cols)
        nbytes, dt = oracle_pass(sample)
        if dt >= budget_s or cols >= 32768:
            return sample, cols, nbytes, dt
        want = int(cols * budget_s / max(dt, 1e-3) * 1.1) + 1
        cols = min(32768, max(cols * 2, want))


def cpu_oracle_sample(M, budget_s=10.0):
    """The CPU oracle on a bounded sample of the step (see size_oracle_sample),
    passed over again until budget_s of CPU work is timed (the column cap keeps
    the host-side weights of the sample near 1 GB).
    Returns (GB/s, cols, passes, seconds, threads)."""
    import oracle

    sample, cols, nbytes, dt = size_oracle_sample(M, budget_s)
    passes = 1
    while dt < budget_s:
        b, t = oracle_pass(sample)
        nbytes, dt, passes = nbytes + b, dt + t, passes + 1
    return nbytes / dt / 1e9, cols, passes, dt, oracle.threads()


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    M = args.m
    per_step = max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    sample, cols, _, _ = size_oracle_sample(M, per_step)
    for _ in range(args.warmup):
        oracle_pass(sample)
    tot_b, tot_t = 0, 0.0
    for _ in range(args.steps):
        b, t = oracle_pass(sample)
        tot_b += b
        tot_t += t
    gbs = tot_b / tot_t / 1e9
    line = {
        "impl": "reference", "metric": "effective weight GB/s (decode-round linears, NVFP4+FP8)",
        "value": round(gbs, 6), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(tot_t / max(1, args.steps) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config(M),
        "cpu_baseline": {"value": round(gbs, 6), "unit": "GB/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": f"each step: {cols} output columns of each of qkv, o_proj, gate_up, "
                                   f"down, lm_head at full K, M={M}"},
        "e2e": {"value": round(gbs, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def aggregate(ms_local, bytes_per_rank, dist=None):
    """Whole-job throughput over all ranks: every rank processes bytes_per_rank
    per step (replicas, weak scaling); the step time is the slowest rank's.
    Returns (GB/s, max ms)."""
    import torch

    ms = float(ms_local)
    world = 1
    if dist is not None and dist.is_initialized():
        world = dist.get_world_size()
        t = torch.tensor([ms], dtype=torch.float64)
        if dist.get_backend() == "nccl":
            t = t.cuda()
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return world * bytes_per_rank / (ms * 1e-3) / 1e9, ms


def config(M):
    return {"workload": f"decode round: {N_LAYERS} x (qkv FP8 5120x7168, o_proj FP8 6144x5120, "
                        f"gate_up NVFP4 5120x34816, down NVFP4 17408x5120) + NVFP4 lm_head 5120x151936 "
                        f"with fused argmax{' and greedy verify of the M-1 drafts' if M > 1 else ''}, M={M}",
            "M": M, "layers": N_LAYERS, "weight_bytes_per_step": STEP_BYTES,
            "l2": "inputs larger than L2 (14.4 GB of weights streamed per step), no flush needed",
            "parallelism": "replicas"}


def time_stack(sk, calls, head, M, stream, steps, warmup, barrier=None, dist=None, clocks_index=None):
    """The decode-round step: `calls` (64 layers x 4 linears + the lm_head)
    captured once into a CUDA graph and replayed `steps` times, CUDA events on
    the capture stream.  Then the same step end to end through the C ABI: the
    activations (and the verify round's drafted tokens) copied from pinned host
    memory and the picks (and the round's verdict) read back every step, all
    inside the timed graph.  Returns a dict of the rates and the clock record."""
    import torch

    dev = head.x.device
    graph = capture(lambda: [c.call(sk) for c in calls], stream)
    with torch.cuda.stream(stream):          # replay() launches on the current stream
        for _ in range(max(3, warmup)):
            graph.replay()
        stream.synchronize()
        if barrier:
            barrier()
        with ClockSampler(clocks_index if clocks_index is not None else dev.index) as clk:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                graph.replay()
            e1.record(stream)
            e1.synchronize()
            torch.cuda.synchronize()
            if barrier:
                barrier()
    value, ms = aggregate(e0.elapsed_time(e1) / steps, STEP_BYTES, dist)
    del graph
    st = sk.last_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error {st}")

    x_dev = torch.empty(sum(c.x.numel() for c in calls), dtype=torch.float16, device=dev)
    views, off = [], 0
    for c in calls:
        views.append(x_dev[off:off + c.x.numel()].view(c.x.shape))
        off += c.x.numel()
    x_host = torch.randn(x_dev.numel(), generator=torch.Generator().manual_seed(7)).to(torch.float16).pin_memory()
    am_host = torch.empty((M,), dtype=torch.int32).pin_memory()
    draft_host = head.draft.cpu().pin_memory()
    accept_host = torch.empty((2,), dtype=torch.int32).pin_memory()
    h2d_bytes = x_dev.numel() * 2 + (draft_host.numel() * 4 if M > 1 else 0)
    d2h_bytes = M * 4 + (8 if M > 1 else 0)

    # The copies run on a side stream in three growing pieces (the first
    # layer, the next seven, the rest with the lm_head's inputs), and each
    # group of calls waits only for its own piece: the first layer starts
    # after ~0.5 MB instead of the whole step's inputs, and the rest of the
    # copy overlaps with compute.
    side = torch.cuda.Stream(device=dev)
    n_lin = len(LAYER)
    cuts = [0, n_lin, 8 * n_lin, len(calls)]
    starts = [0]
    for c in calls:
        starts.append(starts[-1] + c.x.numel())

    def e2e_step():
        cur = torch.cuda.current_stream()
        side.wait_stream(cur)
        evs = []
        with torch.cuda.stream(side):
            for a, b in zip(cuts[:-1], cuts[1:]):
                x_dev[starts[a]:starts[b]].copy_(x_host[starts[a]:starts[b]], non_blocking=True)
                if b == len(calls) and M > 1:
                    head.draft.copy_(draft_host, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(side)
                evs.append(ev)
        for (a, b), ev in zip(zip(cuts[:-1], cuts[1:]), evs):
            cur.wait_event(ev)
            for c, v in zip(calls[a:b], views[a:b]):
                c.call(sk, v)
        am_host.copy_(head.am, non_blocking=True)
        if M > 1:
            accept_host.copy_(head.accept, non_blocking=True)
        cur.wait_stream(side)

    g2 = capture(e2e_step, stream)
    e2e_value, e2e_ms = aggregate(time_graph(g2, stream, reps=steps, warmup=3, barrier=barrier), STEP_BYTES, dist)
    del g2, x_dev
    return {"value": value, "ms": ms, "clocks": clk.summary(),
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": int(h2d_bytes),
                    "d2h_bytes_per_step": int(d2h_bytes), "ms_per_step": round(e2e_ms, 4)}}


def c0_rate(sk, gen, dev, stream, peak, reps=64):
    """The small GEMV case (NVFP4, M=1, K=512, N=256: 73,732 weight bytes).
    Its weights stay in L2, so this is a latency figure, not a bandwidth one:
    a graph of `reps` back-to-back launches on the same weights."""
    K, N = 512, 256
    lin = Linear("c0", "nvfp4", K, N, 1, gen, dev, out_f16=False)
    g = capture(lambda: [lin.call(sk) for _ in range(reps)], stream)
    ms = time_graph(g, stream, reps=10, warmup=3) / reps
    b = weight_bytes("nvfp4", K, N)
    gbs = b / (ms * 1e-3) / 1e9
    return {"K": K, "N": N, "M": 1, "bytes": b, "us": round(ms * 1e3, 2), "GB/s": round(gbs, 1),
            "frac_of_peak": round(gbs / peak, 4), "l2": "weights L2-resident (same weights every launch)"}


def run_ours(args):
    import torch

    import fp8_weight_only_skinny_gb300 as sk

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    barrier = (lambda: dist.barrier()) if dist else None
    sk.init()
    M = args.m
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    stream = torch.cuda.Stream(device=dev)
    if args.layers_only:
        peak, _ = peaks()
        for tp in (False, True):
            for r in layer_table(sk, gen, dev, stream, peak, tp=tp):
                print(f"{'tp4 ' if tp else ''}{r['layer']:8s} {r['fmt']:5s} M={r['M']}  K={r['K']:6d} N={r['N']:6d} "
                      f"{r['us']:8.2f} us  {r['GB/s']:8.1f} GB/s  {r['frac_of_peak'] * 100:5.1f}% of peak", flush=True)
        for r in quant_rates(sk, gen, dev, stream, peak):
            print(f"{r['op']:15s} K={r['K']} N={r['N']}  {r['us']:8.2f} us  {r['GB/s']:8.1f} GB/s  "
                  f"{r['frac_of_peak'] * 100:5.1f}% of peak", flush=True)
        print("lm_head greedy vs sampled:", sampler_cost(sk, gen, dev, stream), flush=True)
        return

    # ---- the decode-round stack, and the same step end to end
    lins = []
    for _ in range(N_LAYERS):
        for name, f, K, N in LAYER:
            lins.append(Linear(name, f, K, N, M, gen, dev))
    head = LMHead(M, gen, dev)
    calls = lins + [head]
    assert sum(c.bytes for c in calls) == STEP_BYTES
    launches_per_step = len(calls)
    main = time_stack(sk, calls, head, M, stream, args.steps, args.warmup, barrier, dist, clocks_index=local)

    # ---- the other step shape over the same weights (single-GPU runs): the
    # plain decode step at M = 1 next to the verify round, or the reverse
    other = None
    if world == 1 and not args.no_other_m:
        Mo = 1 if M != 1 else 8
        ocalls = [c.at_m(Mo, gen, dev) for c in calls]
        r = time_stack(sk, ocalls, ocalls[-1], Mo, stream, args.steps, args.warmup, clocks_index=local)
        other = {"M": Mo, "value": round(r["value"], 1), "unit": "GB/s", "ms_per_step": round(r["ms"], 4),
                 "frac_of_peak": None, "e2e": r["e2e"], "clocks": r["clocks"]}
        del ocalls

    # ---- dominant kernel alone (NVFP4 gate_up launch at this M), cold L2
    peak, peak_kind = peaks()
    if other:
        other["frac_of_peak"] = round(other["value"] / peak, 4)
    gu_ms, gu_bytes = cold_layer_rate(sk, "nvfp4", 5120, 34816, M, gen, dev, stream, copies=8)
    achieved = gu_bytes / (gu_ms * 1e-3) / 1e9
    traffic = read_traffic(M)

    # ---- per-layer tables, cold L2, M = 1 and 8: the full shapes, and the
    # per-rank shapes of 4-way tensor parallelism (the pages' own workload);
    # single-GPU runs only (every replica would measure the same)
    layers, tp_layers, quant, sampler, c0 = [], [], [], None, None
    del calls, lins, head
    torch.cuda.empty_cache()
    if world == 1:
        c0 = c0_rate(sk, gen, dev, stream, peak)
    if not args.no_layers and world == 1:
        layers = layer_table(sk, gen, dev, stream, peak)
        tp_layers = layer_table(sk, gen, dev, stream, peak, tp=True)
        quant = quant_rates(sk, gen, dev, stream, peak)
        sampler = sampler_cost(sk, gen, dev, stream)

    if rank == 0:
        line = {
            "metric": "effective weight GB/s (decode-round linears, NVFP4+FP8)",
            "value": round(main["value"], 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(main["ms"], 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16 x {e2m1,e4m3} -> f32 accumulate",
            "data": "synthetic (device-generated weights, seeded)", "config": config(M),
            "roofline": {"bound": "hbm", "kernel": f"nvfp4 gate_up 5120x34816 M={M}, cold L2",
                         "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "peak_kind": f"{peak_kind} (MEASURED_PEAKS hbm_gbs)" if peak_kind == "measured"
                         else "fallback 6.8 TB/s"},
            "e2e": main["e2e"],
            "gpu_launches": launches_per_step * args.steps,
            "clocks": main["clocks"],
            "frac_of_peak": round(main["value"] / world / peak, 4),
            f"stack_m{other['M']}" if other else "stack_other_m": other,
            "c0": c0,
            "layers": layers,
            "tp4_layers": tp_layers,
            "quantizers": quant,
            "lm_head_sampler": sampler,
        }
        if not args.no_cpu and world == 1:
            import oracle

            gbs, cols, passes, dt, cores = cpu_oracle_sample(M)
            line["cpu_baseline"] = {
                "value": round(gbs, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                "sample": f"{passes} pass(es) over {cols} output columns of each of qkv, o_proj, gate_up, "
                          f"down, lm_head at full K, M={M}, synthetic weights; {dt:.1f} s"}
            oracle.set_threads(1)
            try:
                gbs1, cols1, passes1, dt1, _ = cpu_oracle_sample(M, budget_s=5.0)
            finally:
                oracle.set_threads(cores)
            line["cpu_baseline_1thread"] = {
                "value": round(gbs1, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": f"{passes1} pass(es) over {cols1} output columns of each of qkv, o_proj, gate_up, "
                          f"down, lm_head at full K, M={M}, one thread; {dt1:.1f} s"}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_profile_case(args):
    """A small, bounded workload for ncu: one layer shape at --m over --copies
    weight copies (each launch reads a different copy, so L2 is cold when the
    copies total more than L2), run twice.  Launch order: copies x 2.

    "stack:S" instead runs a shortened decode stack -- S layer sets (qkv,
    o_proj FP8; gate_up, down NVFP4) and the lm_head -- three times in the
    stack's order, eagerly with programmatic dependent launch: the DRAM
    traffic of each kernel inside a stack whose weights L2 cannot hold."""
    import torch

    import fp8_weight_only_skinny_gb300 as sk

    name, fmt = args.profile.split(":")
    if name == "stack":
        torch.cuda.set_device(0)
        dev = torch.device("cuda", 0)
        sk.init()
        gen = torch.Generator(device=dev)
        gen.manual_seed(5)
        calls = [Linear(n, f, K, N, args.m, gen, dev) for _ in range(int(fmt)) for n, f, K, N in LAYER]
        calls.append(LMHead(args.m, gen, dev))
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for _ in range(3):
                for c in calls:
                    c.call(sk)
        s.synchronize()
        st = sk.last_device_error()
        if st != 0:
            raise RuntimeError(f"device error {st}")
        print(f"profile case stack of {fmt} layer sets + lm_head, M={args.m}: {len(calls)} calls x 3: ok")
        return
    if name == "sample":
        # The sampled lm_head (temperature 0.6, top-k 50, top-p 0.9) at --m rows,
        # three calls: the projection kernel, then the cluster sampler.
        torch.cuda.set_device(0)
        dev = torch.device("cuda", 0)
        sk.init()
        gen = torch.Generator(device=dev)
        gen.manual_seed(99)
        head = LMHead(args.m, gen, dev)
        u = torch.rand((args.m,), generator=gen, device=dev)
        tok = torch.empty((args.m,), dtype=torch.int32, device=dev)
        for _ in range(3):
            sk.lm_head_sample(head.x, head.codes, head.scales, head.g, u, 0.6, 50, 0.9, logits=head.y, token=tok)
        torch.cuda.synchronize()
        st = sk.last_device_error()
        if st != 0:
            raise RuntimeError(f"device error {st}")
        print(f"profile case sample M={args.m} x 3: ok")
        return
    if name == "quant":
        # One FP16 weight of the gate_up shape (356 MB), quantized three times.
        K, N = 5120, 34816
        torch.cuda.set_device(0)
        dev = torch.device("cuda", 0)
        sk.init()
        gen = torch.Generator(device=dev)
        gen.manual_seed(99)
        w = (torch.randn((N, K), generator=gen, device=dev) * 0.02).to(torch.float16)
        fn = {"fp8": sk.fp8_quantize, "nvfp4": sk.nvfp4_quantize}[fmt]
        for _ in range(3):
            fn(w)
        torch.cuda.synchronize()
        st = sk.last_device_error()
        if st != 0:
            raise RuntimeError(f"device error {st}")
        print(f"profile case quant:{fmt} K={K} N={N} x 3: ok")
        return
    shapes = {n: (K, N) for n, _, K, N in [*LAYER, LM_HEAD]}
    K, N = shapes[name]
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    sk.init()
    gen = torch.Generator(device=dev)
    gen.manual_seed(99)
    if name == "lm_head":
        lins = [LMHead(args.m, gen, dev) for _ in range(args.copies)]
    else:
        lins = [Linear(name, fmt, K, N, args.m, gen, dev) for _ in range(args.copies)]
    torch.cuda.synchronize()
    for _ in range(2):
        for ln in lins:
            ln.call(sk)
    torch.cuda.synchronize()
    st = sk.last_device_error()
    if st != 0:
        raise RuntimeError(f"device error {st}")
    print(f"profile case {name}:{fmt} M={args.m} K={K} N={N} copies={args.copies}: ok")


# The sources that decide the dominant kernel's code and launch: the linear-layer
# kernel, its PTX helpers, its instantiation and the host code that picks its
# grid and variant.
KERNEL_SOURCES = ("api.cu", "internal.h", "k_nvfp4.cu", "kernel.cuh", "launch.cuh", "ptx.cuh")


def kernel_digest():
    """sha256[:16] over KERNEL_SOURCES, in that order."""
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_weight_only_skinny_gb300", "csrc")
    for n in KERNEL_SOURCES:
        h.update(open(os.path.join(csrc, n), "rb").read())
    return h.hexdigest()[:16]


def read_traffic(M):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source (else None)."""
    f = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(f):
        return None
    digest = kernel_digest()
    for ln in open(f):
        p = ln.split()
        if len(p) == 3 and p[0] == f"M{M}" and p[1] == digest:
            return int(p[2])
    return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--m", type=int, default=8, choices=range(1, 9))
    ap.add_argument("--no-layers", action="store_true", help="skip the per-layer table")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-other-m", action="store_true",
                    help="skip the second stack at the other step shape (M = 1 next to M > 1, or M = 8 next to M = 1)")
    ap.add_argument("--layers-only", action="store_true",
                    help="only print the per-layer cold-L2 table (development A/B runs)")
    ap.add_argument("--profile", metavar="LAYER:FMT",
                    help="small profiling case: run one layer (e.g. gate_up:nvfp4, lm_head:nvfp4) "
                         "over --copies distinct weight copies, twice, and exit; stack:S runs S layer "
                         "sets and the lm_head three times; quant:FMT quantizes one FP16 gate_up "
                         "weight three times; sample:lm_head runs the sampled lm_head three times")
    ap.add_argument("--copies", type=int, default=4)
    args = ap.parse_args()
    if args.profile:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
