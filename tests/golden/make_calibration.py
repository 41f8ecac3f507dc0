"""Write tests/golden/workload_calibration.json: workload constants computed by the CPU oracle only.

  s_mid_tiny, s_mid_flash  static FP32 scale of the intermediate h for the tiny layer (H 256,
                           E 16, k 2, I 128) and the Flash-Next-shaped layer (H 2048, E 512,
                           k 10, I 768): max over experts and over a calibration batch (seed 1,
                           256 tokens, uniform router) of amax(h) / (6 * 448), so the largest h of
                           the batch maps to the top of the NVFP4 range.
  hot_beta                 router bias of the hot set (the first 10 % of the 512 experts) that
                           gives that set 50 % of the top-10 assignments (FP64 bisection on a
                           batch of 1024 tokens, seed 1).

Run:  python tests/golden/make_calibration.py [--skip-flash]
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from nvfp4_w4a4_mixture_gb300 import workloads as wl  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "workload_calibration.json")


def quantized_experts(seed, E, H, I, experts, layer=0):
    """Oracle NVFP4 of the FP32 expert weights, row-major, for the listed experts (others zero)."""
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


def s_mid_for_shape(H, E, k, I, T=256, seed=0, cal_seed=1):
    x = wl.gen_x(cal_seed, T, H)
    w_r = wl.gen_router(seed, E, H)
    ids, tw, g, _ = oracle.router(x, w_r, k)
    experts = sorted(set(ids.ravel().tolist()) | {E})
    gu, dn = quantized_experts(seed, E, H, I, experts)
    xc, xs, Sx = oracle.quantize_nvfp4(x)
    offsets, perm_src, src_perm = oracle.permute(ids, E)
    row_token = np.concatenate([perm_src // k, np.arange(T, dtype=np.int32)]).astype(np.int32)
    gu_out = oracle.grouped_gemm(xc, xs, Sx, offsets, gu[0], gu[1], gu[2], a_row=row_token)
    h = oracle.swiglu(gu_out)
    return float(np.float32(np.abs(h).max()) / np.float32(2688.0))


def hot_beta(H=2048, E=512, k=10, T=1024, seed=0, cal_seed=1):
    x = wl.gen_x(cal_seed, T, H)
    w_r = wl.gen_router(seed, E, H)
    n_hot = int(0.1 * E)

    def share(beta):
        b = wl.router_bias("hot", E, beta=beta).astype(np.float32).astype(np.float64)
        ids, _, _, _ = oracle.router(x, w_r, k, bias=b)
        return float(np.mean(ids < n_hot))

    lo, hi = 0.0, 8.0
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        if share(mid) < 0.5:
            lo = mid
        else:
            hi = mid
    beta = float(np.float32(0.5 * (lo + hi)))
    return beta, share(beta)


def main():
    cal = wl.load_calibration()
    cal["s_mid_tiny"] = s_mid_for_shape(256, 16, 2, 128)
    print("s_mid_tiny", cal["s_mid_tiny"])
    if "--skip-flash" not in sys.argv:
        cal["s_mid_flash"] = s_mid_for_shape(2048, 512, 10, 768)
        print("s_mid_flash", cal["s_mid_flash"])
        beta, sh = hot_beta()
        cal["hot_beta"] = beta
        cal["hot_share_at_beta"] = sh
        print("hot_beta", beta, "share", sh)
    cal["note"] = "written by tests/golden/make_calibration.py (CPU oracle only)"
    with open(OUT, "w") as f:
        json.dump(cal, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main()
