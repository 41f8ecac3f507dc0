"""Seeded synthetic workloads for the routed-MoE layer (shapes of Qwen3.8-Flash-Next's MoE layer).

This module only draws inputs: it holds none of the layer's arithmetic. Every tensor is drawn
from numpy's PCG64 generator seeded by (seed, tensor id, layer, expert), so any single tensor (an
expert's weights, a layer's router) can be regenerated on its own.

Distributions (the capy-flash pages give the layer's shape, not its weights; see "What shipped"
in the richland.au article: 512 experts, 10 routed + 1 shared, 48 layers):
  hidden states x      bf16 values of N(0, 1)
  router / shared gate bf16 values of N(0, 0.02)          [E + 1][H], last row = shared gate
  expert weights       fp32 N(0, 0.02) before NVFP4 quantisation
  router bias          none | Zipf(s=1.1) prior over expert ids | hot set of 10 % of the experts
"""
import json
import math
import os

import numpy as np

# tensor ids of the seeding scheme
TID_X, TID_ROUTER, TID_GATE, TID_UP, TID_DOWN, TID_RESIDUAL = 1, 2, 3, 4, 5, 6

CONFIGS = {
    # parity-size layer: every kernel spans several tiles and a ragged tail
    "tiny": dict(H=256, E=16, k=2, I=128, T=64, router="uniform", layers=1),
    # 4 tokens per call: an MTP K=3 verify window; weight-streaming bound
    "decode": dict(H=2048, E=512, k=10, I=768, T=4, router="uniform", layers=1),
    # prefill chunk with a Zipf(1.1) popularity prior
    "prefill4k": dict(H=2048, E=512, k=10, I=768, T=4096, router="zipf", layers=1),
    # long prefill chunk: 10 % of the experts receive 50 % of the assignments
    "prefill16k": dict(H=2048, E=512, k=10, I=768, T=16384, router="hot", layers=1),
    # 48 MoE-only layers with a residual add between them
    "stack48": dict(H=2048, E=512, k=10, I=768, T=2048, router="uniform", layers=48),
    # the decode call through the same 48-layer stack: 4 tokens per layer, one graph for all layers
    "decode_stack48": dict(H=2048, E=512, k=10, I=768, T=4, router="uniform", layers=48),
    # parity-size layer with the routed-expert count of the full layer and a batch that takes the
    # fused router (12,288 tokens and more), ragged in its last 128-token block
    "wide_router": dict(H=256, E=512, k=10, I=128, T=12365, router="uniform", layers=1),
    # parity cases at the shape limits: hidden size 8192, intermediate size 8192, 1024 experts with top-32
    "max_hidden": dict(H=8192, E=16, k=2, I=128, T=70, router="uniform", layers=1),
    "max_inter": dict(H=256, E=16, k=2, I=8192, T=70, router="uniform", layers=1),
    "max_experts_k": dict(H=256, E=1024, k=32, I=128, T=70, router="uniform", layers=1),
}

CALIBRATION_FILE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                                "tests", "golden", "workload_calibration.json")


def _rng(seed, tid, layer=0, expert=0):
    return np.random.default_rng([int(seed), int(tid), int(layer), int(expert)])


def bf16_round(a):
    """Round float32 values to the nearest bf16 (ties to even); returns float32 holding them."""
    a = np.ascontiguousarray(a, np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def bf16_bits(a):
    """float32 array holding bf16 values -> uint16 bit patterns."""
    a = np.ascontiguousarray(a, np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def gen_x(seed, T, H, layer=0, row0=0):
    """Hidden states: bf16 values of N(0,1), [T][H]. Rows are drawn in blocks of one row so a row
    can be redrawn (row0 selects the counter block)."""
    out = np.empty((T, H), np.float32)
    for t in range(T):
        out[t] = _rng(seed, TID_X, layer, row0 + t).standard_normal(H, dtype=np.float32)
    return bf16_round(out)


def gen_router(seed, E, H, layer=0):
    """Router rows [E][H] and the shared-expert gate row, stacked as [E+1][H], bf16 values."""
    w = _rng(seed, TID_ROUTER, layer).standard_normal((E + 1, H), dtype=np.float32) * np.float32(0.02)
    return bf16_round(w)


def gen_expert(seed, e, H, I, layer=0):
    """FP32 weights of expert e (e == E is the shared expert): gate [I][H], up [I][H], down [H][I]."""
    g = _rng(seed, TID_GATE, layer, e).standard_normal((I, H), dtype=np.float32) * np.float32(0.02)
    u = _rng(seed, TID_UP, layer, e).standard_normal((I, H), dtype=np.float32) * np.float32(0.02)
    d = _rng(seed, TID_DOWN, layer, e).standard_normal((H, I), dtype=np.float32) * np.float32(0.02)
    return g, u, d


def load_calibration():
    if not os.path.exists(CALIBRATION_FILE):
        return {}
    with open(CALIBRATION_FILE) as f:
        return json.load(f)


def router_bias(kind, E, beta=None):
    """Additive router-logit bias that sets the expert-popularity mix of a workload.

    zipf: bias[e] = -1.1 ln(e+1), so the softmax prior is proportional to (e+1)^-1.1.
    hot:  bias[e] = beta for the first floor(0.1 E) experts, 0 elsewhere; beta is calibrated so
          that the hot set receives 50 % of the top-k assignments (stored calibration)."""
    if kind == "uniform":
        return None
    if kind == "zipf":
        return np.array([-1.1 * math.log(e + 1) for e in range(E)], np.float64)
    if kind == "hot":
        if beta is None:
            beta = load_calibration().get("hot_beta")
            if beta is None:
                raise RuntimeError("hot-set router bias is not calibrated")
        b = np.zeros(E, np.float64)
        b[: int(0.1 * E)] = beta
        return b
    raise ValueError(kind)


def s_mid_for(config):
    """Static FP32 scale of the intermediate h (one value for every expert of a layer)."""
    cal = load_calibration()
    key = "s_mid_tiny" if CONFIGS[config]["H"] == 256 else "s_mid_flash"
    if key not in cal:
        raise RuntimeError("intermediate scale for %s is not calibrated" % config)
    return float(cal[key])
