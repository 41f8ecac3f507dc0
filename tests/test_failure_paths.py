"""Failure detection on the GPU without a fault: a device-side wait that runs out.

Every wait in the library is bounded. The test hook of the workspace header makes the expert GEMMs'
wait for a token block's intermediate need more completions than will ever come, with a 20 ms limit:
every down tile then gives up, the launch stops its roles, drains the tensor pipe, frees its tensor
memory and returns; moe_read_device_status reports MOE_ERR_DEVICE_TIMEOUT (one failed call, not a
dead process: capy-flash README v0.7.7, "What's new"). The next call on the same workspace, hook
cleared, must match the oracle -- which also shows the tensor memory was given back (an allocation
that never returns would leave the next launch's CTAs waiting).

The product's environment switches (MOE_NVFP4_GEMM_PERMUTE=0: the front half builds the permutation
for small batches instead of the expert GEMMs; MOE_NVFP4_PDL=0: plain stream order instead of
programmatic dependent launch) are run through the layer parity tests in child processes, since the
library reads them once per process.
"""
import os
import subprocess
import sys

import pytest
import torch

from tests import inputs as I_
from tests.test_gpu_parity import _check_layer, bf16_dev, gpu_layer

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_w4a4_mixture_gb300 as m
    from nvfp4_w4a4_mixture_gb300 import build

    build.build()
    m.lib()
    return m


@pytest.mark.parametrize("name,T", [("tiny", 64), ("decode", 4), ("tiny", 300)])
def test_expert_gemm_wait_runs_out_then_recovers(moe, name, T):
    # 64 tokens: wide tiles; 4: wide-narrow tiles with the shared-memory epilogue and the GEMMs'
    # own permutation; 300: separate front kernels
    case = I_.layer_case(name, seed=31, sample=4, T=T) if name == "decode" else I_.layer_case(name, seed=31, T=T)
    layer = gpu_layer(moe, case)
    ws = moe.Workspace(layer.workspace_bytes(T))
    x = bf16_dev(case["x"])
    moe.moe_set_wait_test_hook(ws, 20_000, 1 << 20)
    moe.moe_layer_forward(layer, x, ws=ws)
    with pytest.raises(moe.MoeError, match="timed out"):
        moe.moe_read_device_status(ws=ws)
    moe.moe_read_device_status(ws=ws)  # reading cleared it
    moe.moe_set_wait_test_hook(ws, 0, 0)
    # the same process and workspace go on: a normal call is correct
    import oracle
    import numpy as np

    out = moe.moe_layer_forward(layer, x, ws=ws)
    moe.moe_read_device_status(ws=ws)
    rows = case["rows"]
    b64 = None if case["bias"] is None else case["bias"].astype(np.float64)
    ref = oracle.layer_forward(case["x"][rows], case["w_r"], case["k"], case["gu"], case["dn"], case["s_mid"],
                               bias=b64, x_scale=oracle.tensor_scale(case["x"]))
    assert I_.rel_frobenius(out.float().cpu().numpy()[rows], ref["out_f64"]) <= 2e-2


def test_wait_hook_rejects_bad_arguments(moe):
    with pytest.raises(moe.MoeError):
        moe.moe_set_wait_test_hook(moe.Workspace(4096), 0, -1)


@pytest.mark.parametrize("env", ["MOE_NVFP4_GEMM_PERMUTE=0", "MOE_NVFP4_PDL=0"])
def test_layer_parity_under_environment_switch(env):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    key, val = env.split("=")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_gpu_parity.py", "tests/test_layer_intermediates.py",
                        "-k", "layer_tiny or layer_decode_full_size or intermediates_tiny or intermediates_decode"
                              " or intermediates_fused_router"],
                       cwd=ROOT, env={**os.environ, key: val}, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
