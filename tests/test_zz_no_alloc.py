"""moe_route_topk_noalloc: the router call for callers that cannot give the library scratch memory
(their device memory belongs to another allocator, or their decode loop cannot afford the device
synchronisation of a cudaMalloc). It keeps its logits scratch in a fixed array inside the library.

Checked through the C ABI against moe_route_topk (the workspace-based call) and against the CPU
oracle's router on calls in a row: 4, then 64, then 7 tokens, so later calls run on the array the
earlier ones left behind (the last one on an array holding 64 tokens' stale rows); an empty batch
returns before anything is read; and the size limit (64 tokens) is refused with a clear error.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from nvfp4_w4a4_mixture_gb300 import workloads as wl
from tests import inputs as I_

pytestmark = pytest.mark.gpu

W_TOL = 1e-6
MOE_ERR_UNSUPPORTED_SHAPE = 2


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_w4a4_mixture_gb300 as m
    from nvfp4_w4a4_mixture_gb300 import build

    build.build()
    m.lib()
    return m


def _layer(m, H, E, k, seed):
    w_r = torch.from_numpy(wl.gen_router(seed, E, H)).to(torch.bfloat16).cuda()
    dummy = (torch.zeros(1, 1, 8, dtype=torch.uint8, device="cuda"),) * 2 + (torch.ones(1, 2, device="cuda"),)
    return m.MoeLayer(H, E, k, 128, w_r, dummy, dummy, torch.ones(E + 1, device="cuda"), prepacked=True)


def _noalloc(m, layer, x):
    T = x.shape[0]
    ids = torch.full((T, layer.k), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros(T, layer.k, dtype=torch.float32, device="cuda")
    g = torch.zeros(T, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = m.lib().moe_route_topk_noalloc(ctypes.c_void_p(x.data_ptr()), T, ctypes.byref(layer.desc),
                                        ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                        ctypes.c_void_p(g.data_ptr()), None, stream)
    assert rc == 0, m.lib().moe_last_error_detail().decode()
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), g.cpu().numpy()


def test_noalloc_router_matches_workspace_router_and_oracle(moe):
    H, E, k = 2048, 512, 10
    layer = _layer(moe, H, E, k, seed=0)
    w_r = wl.gen_router(0, E, H)
    for call, T in enumerate((4, 64, 7)):  # calls in a row on the shared scratch array
        x_np, _ = I_.draw_x(100 + call, T, H, w_r, k)  # gap rule: no near-ties at the top-k edge
        x = torch.from_numpy(x_np).to(torch.bfloat16).cuda()
        ids_ref, w_ref, g_ref, _ = moe.moe_route_topk(x, layer)
        ids, w, g = _noalloc(moe, layer, x)
        np.testing.assert_array_equal(ids, ids_ref.cpu().numpy())
        assert np.max(np.abs(w - w_ref.cpu().numpy())) <= W_TOL
        assert np.max(np.abs(g - g_ref.cpu().numpy())) <= W_TOL
        ids_orc, _, _, _ = oracle.router(x_np, w_r, k)
        np.testing.assert_array_equal(ids, ids_orc)


def test_noalloc_router_empty_batch(moe):
    # T = 0: the shape is checked, then nothing is read or written (NULL buffers accepted)
    layer = _layer(moe, 256, 16, 2, seed=2)
    rc = moe.lib().moe_route_topk_noalloc(None, 0, ctypes.byref(layer.desc), None, None, None, None, None)
    assert rc == 0


def test_noalloc_router_refuses_more_than_64_tokens(moe):
    layer = _layer(moe, 256, 16, 2, seed=1)
    x = torch.zeros(65, 256, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(65, 2, dtype=torch.int32, device="cuda")
    rc = moe.lib().moe_route_topk_noalloc(ctypes.c_void_p(x.data_ptr()), 65, ctypes.byref(layer.desc),
                                          ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(out.data_ptr()), None,
                                          None, None)
    assert rc == MOE_ERR_UNSUPPORTED_SHAPE
    assert b"64 tokens" in moe.lib().moe_last_error_detail()
