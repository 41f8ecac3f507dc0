#!/usr/bin/env python3
"""Benchmark of the NVFP4 W4A4 routed-MoE layer forward (tokens/s per layer on one GB300).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config prefill16k|decode|prefill4k|stack48|tiny]
                    [--impl ours|reference] [--no-graph] [--no-cpu-baseline] [--no-extra]

A step is one whole layer forward (router, W4A4 quantisation, permutation, gate/up GEMM with fused
SwiGLU + requantisation, down GEMM, combine) over one batch of synthetic tokens whose inputs are
resident in HBM. The headline workload (default) is the long prefill chunk: hidden 2048, 512
experts, top-10 + 1 shared, intermediate 768, 16,384 tokens with 10 % of the experts taking half of
the assignments -- the largest single-layer configuration. Unless --no-extra is given, the same
JSON line also carries the 4-token decode call (an MTP K=3 verify window), the same decode call
through a 48-layer stack captured in one graph (per-layer start-up and tail overlap across layer
boundaries), and the 48-layer stack at 2,048 tokens (residual add between layers), under the keys
"decode", "decode_stack48" and "stack48", each measured the same way with its own steps, roofline
and clock record.

L2 is flushed before every timed step, outside the timed interval: a 256 MiB write, then a 256 MiB
read of a second buffer, so the write-back of the flushed lines also happens before the step. Each
step is timed with CUDA events on the launching stream. The end-to-end figure ("e2e") goes through
the library's host-buffer call (moe_layer_forward_host: pinned host input, the copy in, the layer
and the copy out inside the interval; for the layer stack one copy in and one copy out around the
layers). Under torchrun every rank runs an independent replica (weak scaling: per-GPU work fixed);
rank 0 prints one JSON line.

Roofline (per workload): the algorithmic bytes are the routed experts the batch touches plus the
shared expert (3 H I x 0.5625 + 12 bytes each: E2M1 codes, UE4M3 scales, FP32 scales), the router
matrix, x in and the output out (and the residual in the stack); the FP4 work is
2 T (k+1) 3 H I FLOP. Intermediates (x codes, h, y) are reported separately as overhead bytes. The
bound is whichever of the two times at the measured peaks is longer (HBM copy bandwidth; FP4 dense
rate = measured bf16 burst x 6, the nominal FP4:BF16 ratio).

--impl reference times the CPU oracle (the plain FP64 reference of the same layer) on the host
cores, one bounded sample of the workload per step.
"""
import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from nvfp4_w4a4_mixture_gb300 import workloads as wl  # noqa: E402

METRIC = "MoE-layer tokens/s (NVFP4 W4A4) at 1 GB300; % of FP4-TC / HBM roofline"
DEFAULT_CONFIG = "prefill16k"
EXTRA_CONFIGS = ("decode", "decode_stack48", "stack48")
DEFAULT_STEPS = {"tiny": 2000, "decode": 5000, "prefill4k": 600, "prefill16k": 400, "stack48": 30,
                 "decode_stack48": 200, "wide_router": 300, "max_hidden": 500, "max_inter": 500,
                 "max_experts_k": 500}
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 : BF16 tensor-core ratio
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(wl.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-graph", action="store_true", help="launch the layer directly instead of a CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="measure only --config (no decode / stack48 keys)")
    a = ap.parse_args()
    a.steps_given = a.steps is not None
    if a.steps is None:
        a.steps = DEFAULT_STEPS[a.config]
    a.warmup = max(a.warmup, 3)
    return a


def workload_name(c, name):
    s = "%s: MoE layer H%d E%d top-%d + 1 shared, I%d, %d tokens" % (name, c["H"], c["E"], c["k"], c["I"], c["T"])
    if c["router"] == "zipf":
        s += ", Zipf(1.1) expert prior"
    elif c["router"] == "hot":
        s += ", 10% of experts take 50% of assignments"
    if c["layers"] > 1:
        s += ", %d layers + residual" % c["layers"]
    return s


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ------------------------------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ------------------------------------------------------------------------------------------------

class Dist:
    def __init__(self):
        import torch
        import torch.distributed as dist

        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.dist = dist if self.world > 1 else None
        if torch.cuda.is_available():
            torch.cuda.set_device(self.local)
        if self.dist:
            dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    def barrier(self):
        if self.dist:
            self.dist.barrier()

    def max(self, v):
        if not self.dist:
            return v
        import torch

        t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist:
            self.dist.destroy_process_group()


# ------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        import torch

        self.proc = None
        sel = []
        try:
            p = torch.cuda.get_device_properties(device)
            bus = "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
            sel = ["-i", bus]
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-lms", "50"] + sel, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        out = self.proc.communicate(timeout=10)[0]
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# synthetic layer on the device
# ------------------------------------------------------------------------------------------------

def make_device_layer(m, c, seed, layer_idx, s_mid):
    """Weights drawn on the device (seeded torch RNG, the workload's distributions), expert matrices
    quantised to NVFP4 with the library's quantizer (one FP32 scale per expert matrix), prepacked."""
    import torch

    H, E, I = c["H"], c["E"], c["I"]
    g = torch.Generator(device="cuda")
    g.manual_seed(1_000_003 * seed + 7919 * layer_idx + 1)
    w_r = (torch.randn(E + 1, H, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    gu_codes = torch.empty(E + 1, 2 * I, H // 2, dtype=torch.uint8, device="cuda")
    gu_sf = torch.empty(E + 1, 2 * I, H // 16, dtype=torch.uint8, device="cuda")
    gu_scale = torch.empty(E + 1, 2, dtype=torch.float32, device="cuda")
    dn_codes = torch.empty(E + 1, H, I // 2, dtype=torch.uint8, device="cuda")
    dn_sf = torch.empty(E + 1, H, I // 16, dtype=torch.uint8, device="cuda")
    dn_scale = torch.empty(E + 1, dtype=torch.float32, device="cuda")
    ws = m.Workspace(4096)
    for e in range(E + 1):
        w = torch.randn(2 * I, H, generator=g, device="cuda") * 0.02
        for h in range(2):
            m.moe_quantize_nvfp4(w[h * I:(h + 1) * I], ws=ws,
                                 out=(gu_codes[e, h * I:(h + 1) * I], gu_sf[e, h * I:(h + 1) * I], gu_scale[e, h:h + 1]))
        wd = torch.randn(H, I, generator=g, device="cuda") * 0.02
        m.moe_quantize_nvfp4(wd, ws=ws, out=(dn_codes[e], dn_sf[e], dn_scale[e:e + 1]))
    bias = wl.router_bias(c["router"], E)
    bias_t = None if bias is None else torch.tensor(bias.astype("float32"), device="cuda")
    s_mid_t = torch.full((E + 1,), s_mid, dtype=torch.float32, device="cuda")
    layer = m.MoeLayer(H, E, c["k"], I, w_r, (gu_codes, gu_sf, gu_scale), (dn_codes, dn_sf, dn_scale), s_mid_t,
                       logit_bias=bias_t)
    del gu_codes, gu_sf, dn_codes, dn_sf
    return layer


def one_launch_front(c):
    """Small batches run quantisation, routing and permutation as one launch (see csrc/api.cu)."""
    return c["T"] <= 64 and c["T"] * c["k"] <= 512 and c["E"] <= 1024


def fused_route(c):
    """Large batches with 512 experts route first, in one launch that also takes x's maximum, and the
    quantizer's encoding pass follows (see csrc/api.cu)."""
    return (not one_launch_front(c) and c["E"] == 512 and c["k"] <= 16 and c["T"] >= 12288 and c["H"] % 64 == 0
            and c["H"] <= 8192)


def launches_per_layer(c):
    """Kernels of the library launched by one layer forward (see csrc/api.cu)."""
    T, H, k = c["T"], c["H"], c["k"]
    if one_launch_front(c):
        return 3  # front half (quantize + route + permute), expert GEMMs, combine
    if fused_route(c):
        return 1 + 1 + 3 + 1 + 1  # router + top-k + max |x|, encoder, permute, expert GEMMs, combine
    quant = 1 if T * H // 16 <= 4096 else 2
    perm = 1 if T * k <= 512 else 3
    # quantize (its first launch also zeroes the layer's counters), logits + top-k, permute, expert GEMMs
    # (one launch), combine
    return quant + 2 + perm + 1 + 1


def distinct_experts(m, layer, x):
    ids, _, _, _ = m.moe_route_topk(x, layer)
    return int(ids.unique().numel())


GEMM_SOURCES = ("grouped_gemm.cu", "ptx.cuh", "common.cuh", "kernels.cuh")


def gemm_sources_hash(csrc=os.path.join(ROOT, "nvfp4_w4a4_mixture_gb300", "csrc")):
    """Hash of the expert GEMM's sources with comments and blank space removed: a traffic record stays
    valid across edits that do not change the code."""
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(key):
    """DRAM bytes per launch from a committed ncu summary, only while the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    e = rec.get(key)
    if not e or e.get("source_hash") != gemm_sources_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ------------------------------------------------------------------------------------------------

class OracleSample:
    """The oracle layer forward on a few tokens of the workload (inputs from the workload generator;
    the expert weights the sample routes to are quantised by the oracle itself, untimed)."""

    def __init__(self, c, seed, n_tokens):
        import numpy as np

        import oracle

        self.oracle = oracle
        H, E, k, I = c["H"], c["E"], c["k"], c["I"]
        self.k = k
        self.x = wl.gen_x(seed, n_tokens, H)
        self.w_r = wl.gen_router(seed, E, H)
        b = wl.router_bias(c["router"], E)
        self.bias = None if b is None else b.astype(np.float32).astype(np.float64)
        ids, _, _, _ = oracle.router(self.x, self.w_r, k, bias=self.bias)
        experts = sorted(set(ids.ravel().tolist()) | {E})
        self.gu = [np.zeros((E + 1, 2 * I, H // 2), np.uint8), np.zeros((E + 1, 2 * I, H // 16), np.uint8),
                   np.ones((E + 1, 2), np.float32)]
        self.dn = [np.zeros((E + 1, H, I // 2), np.uint8), np.zeros((E + 1, H, I // 16), np.uint8),
                   np.ones(E + 1, np.float32)]
        for e in experts:
            g, u, d = wl.gen_expert(seed, e, H, I)
            for h, w in enumerate((g, u)):
                cc, s, S = oracle.quantize_nvfp4(w)
                self.gu[0][e, h * I:(h + 1) * I], self.gu[1][e, h * I:(h + 1) * I], self.gu[2][e, h] = cc, s, S
            cc, s, S = oracle.quantize_nvfp4(d)
            self.dn[0][e], self.dn[1][e], self.dn[2][e] = cc, s, S
        self.s_mid = np.full(E + 1, s_mid_value(c), np.float32)
        self.n_tokens = n_tokens
        self.cores = oracle.num_threads()

    def run(self, rows=None):
        x = self.x if rows is None else self.x[rows]
        self.oracle.layer_forward(x, self.w_r, self.k, self.gu, self.dn, self.s_mid, bias=self.bias)
        return x.shape[0]


def s_mid_value(c):
    cfg = "tiny" if c["H"] == 256 else "decode"
    return wl.s_mid_for(cfg)


def cpu_baseline(c, seed, budget_s=12.0):
    n = min(c["T"], 4)
    smp = OracleSample(c, seed, n)
    done, t0 = 0, time.perf_counter()
    while True:
        done += smp.run()
        el = time.perf_counter() - t0
        if el >= budget_s or done >= 64 * n:
            break
    return {"value": done / el, "unit": "tokens/s", "cores": smp.cores, "kind": "oracle",
            "sample": "%d tokens of the workload per oracle call (their %d-expert weights prepared untimed), "
                      "%d tokens timed over %.1f s" % (n, c["k"] + 1, done, el)}


def run_reference(args, c, d):
    if d.rank != 0:
        return
    smp = OracleSample(c, args.seed, min(c["T"], 4))
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        smp.run(rows=[i % smp.n_tokens])
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1000.0 * statistics.mean(times)
    value = 1000.0 / ms
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(c, args.config), "sample_per_step": "1 token (its k routed + 1 shared experts)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": smp.cores, "kind": "oracle",
                             "sample": "1 token per step through the FP64 CPU oracle"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------------
# roofline arithmetic (algorithmic work of one layer call)
# ------------------------------------------------------------------------------------------------

def expert_bytes(H, I):
    """Bytes of one expert: gate, up and down matrices as E2M1 codes + UE4M3 block scales, 3 FP32 scales."""
    return 3 * H * I * 9 // 16 + 12


def algorithmic_work(c, U):
    """Per layer call: bytes the method must move (touched routed experts + the shared one, router,
    x, out, residual in a stack) split into weights / activations, FP4 FLOPs of the expert GEMMs,
    bf16 FLOPs of the router, and the intermediates' traffic reported as overhead."""
    H, E, k, I, T = c["H"], c["E"], c["k"], c["I"], c["T"]
    P = T * (k + 1)
    weights = (U + 1) * expert_bytes(H, I)
    router = (E + 1) * H * 2
    io = T * H * 2 * (3 if c["layers"] > 1 else 2)  # x, out (+ residual)
    overhead = {"x_codes_written_read": 2 * T * H * 9 // 16, "h_written_read": 2 * P * I * 9 // 16,
                "y_written_read": 2 * P * H * 2}
    return {"weights": weights, "router": router, "io": io, "layer_bytes": weights + router + io,
            "kernel_bytes": weights + io, "flops_fp4": 2.0 * P * 3 * H * I, "flops_bf16": 2.0 * T * H * (E + 1),
            "overhead_bytes": overhead}


def roofline(bytes_, flops, seconds, hbm_gbs, fp4_tflops):
    """Bound = the longer of the two times at the peaks; achieved and frac against that peak."""
    t_hbm = bytes_ / (hbm_gbs * 1e9)
    t_fp4 = flops / (fp4_tflops * 1e12)
    hbm_ach = bytes_ / seconds / 1e9
    fp4_ach = flops / seconds / 1e12
    if t_fp4 > t_hbm:
        return {"bound": "tensor", "achieved": fp4_ach, "peak": fp4_tflops, "unit": "TFLOP/s",
                "frac": fp4_ach / fp4_tflops, "hbm_frac": hbm_ach / hbm_gbs, "fp4_tc_frac": fp4_ach / fp4_tflops}
    return {"bound": "hbm", "achieved": hbm_ach, "peak": hbm_gbs, "unit": "GB/s", "frac": hbm_ach / hbm_gbs,
            "hbm_frac": hbm_ach / hbm_gbs, "fp4_tc_frac": fp4_ach / fp4_tflops}


# ------------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------------

def measure(m, name, K, W, args, d):
    """One workload: timed steps (CUDA graph replay, L2 flushed before each), per-stage stream events,
    the end-to-end host-buffer call, roofline. Frees its device memory before returning."""
    import torch

    c = wl.CONFIGS[name]
    H, E, k, I, T, L = c["H"], c["E"], c["k"], c["I"], c["T"], c["layers"]
    s_mid = s_mid_value(c)
    layers = [make_device_layer(m, c, args.seed + 1000 * d.rank, li, s_mid) for li in range(L)]
    g = torch.Generator(device="cuda")
    g.manual_seed(12345 + d.rank)
    x = torch.randn(T, H, generator=g, device="cuda").to(torch.bfloat16)
    bufs = [torch.empty(T, H, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    ws = m.Workspace(layers[0].workspace_bytes(T))
    flush_w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    flush_sum = torch.empty((), dtype=torch.float32, device="cuda")

    def flush_l2():
        # evict everything the previous step left in L2: write a buffer larger than L2, then read
        # another one, which also writes the dirty flush lines back before the step starts
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_sum)

    def forward():
        cur = x
        for li, lay in enumerate(layers):
            o = bufs[li % 2]
            m.moe_layer_forward(lay, cur, residual=cur if L > 1 else None, out=o, ws=ws)
            cur = o
        return cur

    use_graph = not args.no_graph
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        forward()
        forward()
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    m.moe_read_device_status(ws)
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            forward()
        run = graph.replay
    else:
        run = forward

    # ---- timed region: K steps, L2 flushed before each, CUDA events on the launching stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with torch.cuda.stream(stream):
        for _ in range(W):
            flush_l2()
            run()
    torch.cuda.synchronize()
    d.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(d.local)
    torch.cuda.nvtx.range_push("timed " + name)
    with torch.cuda.stream(stream):
        for i in range(K):
            flush_l2()
            ev[i][0].record(stream)
            run()
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    d.barrier()
    torch.cuda.synchronize()
    clk = clocks.stop()
    m.moe_read_device_status(ws)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = d.max(statistics.mean(step_ms))
    value = d.world * T / (ms / 1000.0)

    # ---- per-stage durations of the same launch sequence (CUDA events at the stage boundaries). A
    # spin kernel (~0.5 ms) ahead of each step lets the host queue the whole step first, so an
    # interval holds its kernel's device time (with the launch gap in front of it), not the host's
    # launch latency.
    Kp = min(K, 500)
    st_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(m.LAYER_STAGES) + 1)] for _ in range(Kp)]
    with torch.cuda.stream(stream):
        for i in range(Kp):
            flush_l2()
            torch.cuda._sleep(1_000_000)
            m.moe_layer_forward_profiled(layers[0], x, st_ev[i], residual=x if L > 1 else None, out=bufs[0], ws=ws)
    torch.cuda.synchronize()
    durs = [[e[j].elapsed_time(e[j + 1]) for e in st_ev] for j in range(len(m.LAYER_STAGES))]
    stage_us = {sn: 1000.0 * statistics.mean(durs[j]) for j, sn in enumerate(m.LAYER_STAGES)}
    if one_launch_front(c):
        # one launch covers the first three stages: events 1..3 follow it back to back
        stage_us = {"front": sum(stage_us.pop(n) for n in ("quantize", "route", "permute")), **stage_us}
    elif fused_route(c):
        # routing ran first: the first interval is the router's, the second the encoder's
        first, second = stage_us.pop("quantize"), stage_us.pop("route")
        stage_us = {"route (with max |x|)": first, "quantize (encode)": second, **stage_us}

    # ---- end to end through the public calls: pinned host input -> layer -> pinned host output.
    # Small batches and the stack: one step at a time on one stream, L2 flushed before each step
    # (outside its interval): moe_layer_forward_host (the library enqueues both copies and the layer)
    # for one layer; the input copied in once, the layers, the last output copied back for a stack.
    # Large batches (one layer, T >= 1024): two steps in flight on two streams, each with its own
    # device buffers and workspace, as a serving loop runs them: a step's input copy and the previous
    # step's output copy overlap the other step's kernels, and each step's layer waits for the
    # previous step's layer (so the kernels of two steps never share the GPU); the interval covers all
    # Ke steps, every one of which copies its input in and its output out inside it (no L2 flush: a
    # step's expert weights, 0.4 GB and more at these sizes, exceed the 126 MB L2 by themselves).
    x_h = x.cpu().pin_memory()
    n_str = 2 if (L == 1 and T >= 1024) else 1
    out_h = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(n_str)]
    Ke = min(K, 1000)
    x_dev = [torch.empty_like(x) for _ in range(n_str)]
    streams = [stream] + [torch.cuda.Stream() for _ in range(n_str - 1)]
    if n_str == 1:
        e2e_call = "moe_layer_forward_host" if L == 1 else "copy in + %d x moe_layer_forward + copy out" % L
        ws_h = m.Workspace(m.moe_workspace_bytes_host(H, E, k, I, T)) if L == 1 else None
        ee = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Ke)]
        with torch.cuda.stream(stream):
            for i in range(Ke):
                flush_l2()
                ee[i][0].record(stream)
                if L == 1:
                    m.moe_layer_forward_host(layers[0], x_h, out=out_h[0], ws=ws_h)
                else:
                    x_dev[0].copy_(x_h, non_blocking=True)
                    cur = x_dev[0]
                    for li, lay in enumerate(layers):
                        o = bufs[li % 2]
                        m.moe_layer_forward(lay, cur, residual=cur, out=o, ws=ws)
                        cur = o
                    out_h[0].copy_(cur, non_blocking=True)
                ee[i][1].record(stream)
        torch.cuda.synchronize()
        e2e_ms = d.max(statistics.mean(a.elapsed_time(b) for a, b in ee))
        e2e_ws = [ws_h or ws]
    else:
        e2e_call = "copy in + moe_layer_forward + copy out, two steps in flight on two streams"
        e2e_ws = [ws] + [m.Workspace(layers[0].workspace_bytes(T)) for _ in range(n_str - 1)]
        out_dev = [torch.empty_like(x) for _ in range(n_str)]
        layer_done = [torch.cuda.Event() for _ in range(n_str)]

        def e2e_step(i):
            j, jp = i % n_str, (i - 1) % n_str
            sj = streams[j]
            with torch.cuda.stream(sj):
                x_dev[j].copy_(x_h, non_blocking=True)
                if i > 0:
                    sj.wait_event(layer_done[jp])  # the previous step's layer has finished
                m.moe_layer_forward(layers[0], x_dev[j], out=out_dev[j], ws=e2e_ws[j])
                layer_done[j].record(sj)
                out_h[j].copy_(out_dev[j], non_blocking=True)

        for i in range(W):
            e2e_step(i)
        torch.cuda.synchronize()
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_side = [torch.cuda.Event() for _ in streams[1:]]
        e_start.record(streams[0])
        for sd in streams[1:]:
            sd.wait_event(e_start)
        for i in range(Ke):
            e2e_step(i)
        for sd, ev in zip(streams[1:], e_side):
            ev.record(sd)
            streams[0].wait_event(ev)
        e_end.record(streams[0])
        torch.cuda.synchronize()
        e2e_ms = d.max(e_start.elapsed_time(e_end) / Ke)
    for w in e2e_ws:
        m.moe_read_device_status(w)

    # ---- roofline of the dominant kernel (the expert GEMMs, one launch) and of the whole step
    hbm, bf16_burst, bf16_sus, peak_src = measured_peaks()
    fp4_peak = bf16_burst * FP4_OVER_BF16
    U = distinct_experts(m, layers[0], x)  # routed experts touched by this batch (first layer)
    work = algorithmic_work(c, U)
    exp_us = stage_us["experts"]
    kern = roofline(work["kernel_bytes"], work["flops_fp4"], exp_us * 1e-6, hbm, fp4_peak)
    kern.update({
        "traffic": recorded_traffic("experts/" + name),
        "kernel": "k_grouped_gemm_nvf4 (gate/up + SwiGLU + NVFP4 requant + down, one launch)",
        "algorithmic_bytes_per_launch": work["kernel_bytes"],
        "algorithmic_bytes": "touched routed experts + shared expert (%d x %d B) + x + out%s" % (
            U + 1, expert_bytes(H, I), " + residual" if L > 1 else ""),
        "flops_fp4_per_launch": work["flops_fp4"], "overhead_bytes_per_launch": work["overhead_bytes"],
        "avg_launch_us": exp_us, "timed_by": "stream events around the launch (includes its launch gap)",
        "peak_source": "%s hbm_gbs; FP4 = %s bf16 burst x %.0f (nominal FP4:BF16)" % (peak_src, peak_src, FP4_OVER_BF16)})
    t_s = ms / 1000.0  # per-replica step time
    step_roof = roofline(L * work["layer_bytes"], L * work["flops_fp4"], t_s, hbm, fp4_peak)
    step_roof.update({"bytes": L * work["layer_bytes"], "flops_fp4": L * work["flops_fp4"],
                      "overhead_bytes": {kk: L * v for kk, v in work["overhead_bytes"].items()},
                      "fp4_peak_tflops": fp4_peak, "hbm_peak_gbs": hbm})
    res = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": d.world, "steps": K, "warmup": W,
        "ms_per_step": ms, "per_layer_us": 1000.0 * ms / L,
        "config": {"workload": workload_name(c, name), "tokens": T, "layers": L,
                   "distinct_routed_experts": U, "cuda_graph": use_graph,
                   "l2": "flushed before every timed step (256 MiB write, then 256 MiB read of another "
                         "buffer; outside the timed interval)",
                   "parallelism": "replicas" if d.world > 1 else "single GPU"},
        "roofline": kern,
        "layer_roofline": step_roof,
        "stages_us": stage_us,
        "stages_timed_by": "stream events at the stage boundaries, each step queued behind a spin kernel",
        "step_ms_median": statistics.median(step_ms),
        "e2e": {"value": d.world * T / (e2e_ms / 1000.0), "unit": "tokens/s", "h2d_bytes_per_step": T * H * 2,
                "d2h_bytes_per_step": T * H * 2, "ms_per_step": e2e_ms, "cuda_graph": False, "call": e2e_call,
                "streams": n_str},
        "gpu_launches": K * L * launches_per_layer(c),
        "clocks": clk,
    }
    del layers, run
    if use_graph:
        del graph
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_ours(args, c, d):
    import nvfp4_w4a4_mixture_gb300 as m
    from nvfp4_w4a4_mixture_gb300 import build

    if d.local == 0 or not os.path.exists(m.LIB_PATH):
        build.build()
    d.barrier()
    m.lib()
    head = measure(m, args.config, args.steps, args.warmup, args, d)
    line = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": d.world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "nvfp4",
            "data": "synthetic: seeded torch RNG on the device; x ~ N(0,1) bf16, router N(0,0.02) bf16, experts "
                    "N(0,0.02) fp32 quantised to NVFP4 by the library"}
    line.update({kk: v for kk, v in head.items() if kk not in line and kk != "metric"})
    if not args.no_extra:
        for name in EXTRA_CONFIGS:
            if name != args.config:
                line[name] = measure(m, name, DEFAULT_STEPS[name], args.warmup, args, d)
    return line


def main():
    args = parse_args()
    c = wl.CONFIGS[args.config]
    d = Dist()
    try:
        if args.impl == "reference":
            run_reference(args, c, d)
            return
        line = run_ours(args, c, d)
        if d.rank == 0:
            if not args.no_cpu_baseline and d.world == 1:
                line["cpu_baseline"] = cpu_baseline(c, args.seed)
            print(json.dumps(line), flush=True)
    finally:
        d.close()


if __name__ == "__main__":
    main()
