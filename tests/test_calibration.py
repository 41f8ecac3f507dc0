"""The stored workload constants are reproduced by their generator, which calls only the oracle."""
import importlib.util
import json
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def _gen():
    spec = importlib.util.spec_from_file_location("make_calibration", os.path.join(HERE, "golden", "make_calibration.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _stored():
    with open(os.path.join(HERE, "golden", "workload_calibration.json")) as f:
        return json.load(f)


def test_s_mid_tiny_reproduces(orc):
    assert _gen().s_mid_for_shape(256, 16, 2, 128) == _stored()["s_mid_tiny"]


def test_s_mid_flash_reproduces(orc):
    # the Flash-shaped layer's intermediate scale (H 2048, E 512, k 10, I 768; about a minute of
    # oracle work: the touched experts' weights quantised, the gate/up GEMM and SwiGLU of 256 tokens)
    assert _gen().s_mid_for_shape(2048, 512, 10, 768) == _stored()["s_mid_flash"]


def test_hot_beta_gives_half_the_assignments(orc):
    # the stored bias gives the first 10 % of the 512 experts 50 % of the top-10 assignments of the
    # calibration batch (1024 tokens), and a slightly smaller bias gives them less
    from nvfp4_w4a4_mixture_gb300 import workloads as wl

    beta = _stored()["hot_beta"]
    x = wl.gen_x(1, 1024, 2048)
    w_r = wl.gen_router(0, 512, 2048)

    def share(b):
        bias = wl.router_bias("hot", 512, beta=b).astype(np.float32).astype(np.float64)
        ids, _, _, _ = orc.router(x, w_r, 10, bias=bias)
        return float(np.mean(ids < 51))

    assert share(beta) >= 0.5
    assert share(beta * 0.99) < 0.5
