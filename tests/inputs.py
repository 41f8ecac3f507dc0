"""Seeded layer inputs for the parity tests (test infrastructure: may call the oracle).

The raw tensors come from nvfp4_w4a4_mixture_gb300.workloads; this module adds what needs the
oracle: the router-gap rule (no two of a token's top k+1 logits closer than 1e-4, so the
routing decision cannot depend on the accumulation order) and the oracle's NVFP4 quantisation
of the expert weights.
"""
import functools

import numpy as np

import oracle
from nvfp4_w4a4_mixture_gb300 import workloads as wl

GAP = 1e-4


def gap_ok_rows(logits, k, gap=GAP):
    s = -np.sort(-logits, axis=1)[:, : k + 1]
    return np.min(s[:, :-1] - s[:, 1:], axis=1) >= gap


def draw_x(seed, T, H, w_r, k, bias=None, layer=0):
    """x [T][H] (bf16 values), rows redrawn from fresh counter blocks until the gap rule holds."""
    x = wl.gen_x(seed, T, H, layer)
    redrawn = 0
    for attempt in range(1, 64):
        _, _, _, lg = oracle.router(x, w_r, k, bias=bias, want_logits=True)
        bad = np.where(~gap_ok_rows(lg, k))[0]
        if bad.size == 0:
            return x, redrawn
        for t in bad:
            x[t] = wl.gen_x(seed, 1, H, layer, row0=attempt * 10_000_000 + int(t))[0]
        redrawn += bad.size
    raise RuntimeError("gap rule not met after 63 redraws")


def bias_for(config):
    kind = wl.CONFIGS[config]["router"]
    b = wl.router_bias(kind, wl.CONFIGS[config]["E"])
    # the device takes an FP32 bias: both sides use the FP32 values
    return None if b is None else b.astype(np.float32)


def quantized_experts(seed, E, H, I, experts, layer=0):
    """Oracle NVFP4 (row-major) of the listed experts; the others are all-zero filler (never routed to
    in a test that uses them: routing is compared bit-exactly first)."""
    gu = [np.zeros((E + 1, 2 * I, H // 2), np.uint8), np.zeros((E + 1, 2 * I, H // 16), np.uint8),
          np.ones((E + 1, 2), np.float32)]
    dn = [np.zeros((E + 1, H, I // 2), np.uint8), np.zeros((E + 1, H, I // 16), np.uint8),
          np.ones(E + 1, np.float32)]
    for e in experts:
        g, u, d = wl.gen_expert(seed, e, H, I, layer)
        for h, w in enumerate((g, u)):
            c, s, S = oracle.quantize_nvfp4(w)
            gu[0][e, h * I:(h + 1) * I], gu[1][e, h * I:(h + 1) * I], gu[2][e, h] = c, s, S
        c, s, S = oracle.quantize_nvfp4(d)
        dn[0][e], dn[1][e], dn[2][e] = c, s, S
    return gu, dn


@functools.lru_cache(maxsize=4)
def layer_case(config, seed=0, sample=None, T=None):
    """Inputs of one layer call. sample: number of tokens whose experts get real weights (None: all
    tokens); T: token count other than the configuration's. Returns a dict of numpy arrays."""
    c = wl.CONFIGS[config]
    H, E, k, I = c["H"], c["E"], c["k"], c["I"]
    T = c["T"] if T is None else int(T)
    w_r = wl.gen_router(seed, E, H)
    bias = bias_for(config)
    x, redrawn = draw_x(seed, T, H, w_r, k, bias=None if bias is None else bias.astype(np.float64))
    ids, _, _, _ = oracle.router(x, w_r, k, bias=None if bias is None else bias.astype(np.float64))
    if sample is None:
        rows = np.arange(T)
    else:
        rows = np.unique(np.random.default_rng(seed + 99).choice(T, size=min(sample, T), replace=False))
    experts = sorted(set(ids[rows].ravel().tolist()) | {E})
    gu, dn = quantized_experts(seed, E, H, I, experts)
    s_mid = np.full(E + 1, wl.s_mid_for(config), np.float32)
    return dict(H=H, E=E, k=k, I=I, T=T, x=x, w_r=w_r, bias=bias, gu=gu, dn=dn, s_mid=s_mid, rows=rows,
                redrawn=redrawn)


def rel_frobenius(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))
