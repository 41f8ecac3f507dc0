"""The C ABI without a GPU: the library builds, loads and exports every symbol the header
declares; host-side validation returns the documented error codes before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_nvfp4.h")


@pytest.fixture(scope="module")
def L():
    from nvfp4_w4a4_mixture_gb300 import build

    build.build()
    import nvfp4_w4a4_mixture_gb300 as m

    return m.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s+(moe_[a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("moe_quantize_nvfp4", "moe_route_topk", "moe_permute", "moe_grouped_gemm_nvfp4",
                     "moe_combine", "moe_layer_forward"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_binding_lists_every_declared_symbol():
    import nvfp4_w4a4_mixture_gb300 as m

    assert set(declared_functions()) <= set(m.ENTRY_POINTS)


def test_status_strings(L):
    for s in range(8):
        assert L.moe_status_string(s).decode().startswith("MOE_")
    assert L.moe_status_string(99) == b"unknown moe_status_t"


def test_workspace_bytes_grows_with_tokens(L):
    a = L.moe_workspace_bytes(2048, 512, 10, 768, 4)
    b = L.moe_workspace_bytes(2048, 512, 10, 768, 4096)
    assert 0 < a < b
    assert a % 256 == 0 and b % 256 == 0
    assert L.moe_workspace_bytes(-1, 512, 10, 768, 4) == 0


def test_workspace_bytes_host_adds_three_staging_buffers(L):
    # the host-buffer layer call stages x, the residual and the output (T x H bf16 each, 256-byte
    # aligned) behind the layer's own workspace
    for H, T in ((2048, 4), (2048, 4096), (256, 3)):
        base = L.moe_workspace_bytes(H, 512, 10, 768, T)
        stage = (T * H * 2 + 255) // 256 * 256
        assert L.moe_workspace_bytes_host(H, 512, 10, 768, T) == base + 3 * stage
    assert L.moe_workspace_bytes_host(2048, 512, 10, 768, -1) == 0


MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED_SHAPE, MOE_ERR_WORKSPACE_TOO_SMALL, MOE_ERR_MISALIGNED = 1, 2, 3, 4


def _fake(addr):
    # host-side validation never dereferences device pointers
    return ctypes.c_void_p(addr)


def test_quantize_validation(L):
    ws = _fake(0x10000)
    p = _fake(0x20000)
    assert L.moe_quantize_nvfp4(p, 4, 24, None, p, p, p, ws, 4096, None) == MOE_ERR_UNSUPPORTED_SHAPE
    assert b"K=24" in L.moe_last_error_detail()
    assert L.moe_quantize_nvfp4(None, 4, 32, None, p, p, p, ws, 4096, None) == MOE_ERR_INVALID_ARG
    assert L.moe_quantize_nvfp4(_fake(0x20008), 4, 32, None, p, p, p, ws, 4096, None) == MOE_ERR_MISALIGNED
    assert L.moe_quantize_nvfp4(p, 4, 32, None, p, p, p, ws, 16, None) == MOE_ERR_WORKSPACE_TOO_SMALL
    assert L.moe_quantize_nvfp4(p, 4, 32, None, p, p, p, _fake(0x10010), 4096, None) == MOE_ERR_MISALIGNED
    assert b"not 256-byte aligned" in L.moe_last_error_detail()


def test_layer_validation(L):
    import nvfp4_w4a4_mixture_gb300 as m

    p = 0x40000
    bank = m.NvFp4Bank(p, p, p)
    good = m.LayerDesc(2048, 512, 10, 768, p, None, bank, bank, p)
    ws = _fake(0x100000)
    need = L.moe_workspace_bytes(2048, 512, 10, 768, 4)
    f = L.moe_layer_forward
    assert f(None, _fake(p), 4, None, _fake(p + 4096), ws, need, None) == MOE_ERR_INVALID_ARG
    bad = m.LayerDesc(2050, 512, 10, 768, p, None, bank, bank, p)
    assert f(ctypes.byref(bad), _fake(p), 4, None, _fake(p + 4096), ws, need, None) == MOE_ERR_UNSUPPORTED_SHAPE
    assert b"H=2050" in L.moe_last_error_detail()
    bad = m.LayerDesc(2048, 512, 33, 768, p, None, bank, bank, p)
    assert f(ctypes.byref(bad), _fake(p), 4, None, _fake(p + 4096), ws, need, None) == MOE_ERR_UNSUPPORTED_SHAPE
    bad = m.LayerDesc(2048, 2048, 10, 768, p, None, bank, bank, p)
    assert f(ctypes.byref(bad), _fake(p), 4, None, _fake(p + 4096), ws, need, None) == MOE_ERR_UNSUPPORTED_SHAPE
    assert f(ctypes.byref(good), _fake(p), 4, None, _fake(p + 4096), ws, need - 256, None) == MOE_ERR_WORKSPACE_TOO_SMALL
    assert f(ctypes.byref(good), _fake(p + 8), 4, None, _fake(p + 4096), ws, need, None) == MOE_ERR_MISALIGNED
    biased = m.LayerDesc(2048, 512, 10, 768, p, p + 4, bank, bank, p)  # the logit bias is read 16 bytes at a time
    assert f(ctypes.byref(biased), _fake(p), 4, None, _fake(p + 4096), ws, need, None) == MOE_ERR_MISALIGNED
    assert b"logit_bias" in L.moe_last_error_detail()
    assert f(ctypes.byref(good), _fake(p), 4, None, _fake(p), ws, need, None) == MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(good), _fake(p), -1, None, _fake(p + 4096), ws, need, None) == MOE_ERR_UNSUPPORTED_SHAPE
    nullbank = m.NvFp4Bank(p, None, p)
    bad = m.LayerDesc(2048, 512, 10, 768, p, None, nullbank, bank, p)
    assert f(ctypes.byref(bad), _fake(p), 4, None, _fake(p + 4096), ws, need, None) == MOE_ERR_INVALID_ARG


def test_layer_host_validation(L):
    # host-side checks of the host-buffer layer call, made before any device is touched
    import nvfp4_w4a4_mixture_gb300 as m

    p = 0x40000
    bank = m.NvFp4Bank(p, p, p)
    good = m.LayerDesc(2048, 512, 10, 768, p, None, bank, bank, p)
    ws = _fake(0x100000)
    need = L.moe_workspace_bytes_host(2048, 512, 10, 768, 4)
    f = L.moe_layer_forward_host
    x, out = _fake(0x7000000), _fake(0x7100000)
    assert f(None, x, 4, None, out, ws, need, None) == MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(good), None, 4, None, out, ws, need, None) == MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(good), x, -1, None, out, ws, need, None) == MOE_ERR_UNSUPPORTED_SHAPE
    # out overlapping x (4 tokens x 4 KB) or the residual
    assert f(ctypes.byref(good), x, 4, None, _fake(0x7000000 + 4096), ws, need, None) == MOE_ERR_INVALID_ARG
    assert b"overlaps" in L.moe_last_error_detail()
    assert f(ctypes.byref(good), x, 4, _fake(0x7100000 + 8192), out, ws, need, None) == MOE_ERR_INVALID_ARG
    # the layer's workspace alone is not enough: the three staging buffers come on top of it
    small = L.moe_workspace_bytes(2048, 512, 10, 768, 4)
    assert f(ctypes.byref(good), x, 4, None, out, ws, small, None) == MOE_ERR_WORKSPACE_TOO_SMALL


def test_gemm_and_permute_validation(L):
    import nvfp4_w4a4_mixture_gb300 as m

    p = 0x40000
    bank = m.NvFp4Bank(p, p, p)
    ws = _fake(0x100000)
    g = L.moe_grouped_gemm_nvfp4
    args = lambda N, K, G=4, epi=0, gu=1, epi_scale=None, out_sf=None: (
        _fake(p), _fake(p), _fake(p), 0, None, _fake(p), G, 100, ctypes.byref(bank), N, K, gu, epi,
        epi_scale, _fake(p), out_sf, ws, 1 << 20, None)
    assert g(*args(200, 256)) == MOE_ERR_UNSUPPORTED_SHAPE
    assert g(*args(256, 96)) == MOE_ERR_UNSUPPORTED_SHAPE
    assert g(*args(256, 256, G=0)) == MOE_ERR_UNSUPPORTED_SHAPE
    assert g(*args(256, 256, epi=7)) == MOE_ERR_INVALID_ARG
    assert g(*args(256, 256, epi=2, gu=0)) == MOE_ERR_INVALID_ARG
    pm = L.moe_permute
    assert pm(_fake(p), 4, 11, 10, 1, _fake(p), _fake(p), _fake(p), None, ws, 1 << 20, None) == MOE_ERR_UNSUPPORTED_SHAPE
    assert pm(_fake(p), 4, 2, 10, 1, _fake(p), _fake(p), _fake(p), None, ws, 16, None) == MOE_ERR_WORKSPACE_TOO_SMALL
    assert pm(None, 4, 2, 10, 1, _fake(p), _fake(p), _fake(p), None, ws, 1 << 20, None) == MOE_ERR_INVALID_ARG


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import nvfp4_w4a4_mixture_gb300 as m

    monkeypatch.setattr(m, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(m, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        m.lib()


def test_empty_batch_is_a_no_op(L):
    # T = 0: the shape is checked, nothing is read, written or launched, so NULL buffers are accepted;
    # a bad shape is still refused
    import nvfp4_w4a4_mixture_gb300 as m

    p = 0x40000
    bank = m.NvFp4Bank(p, p, p)
    good = m.LayerDesc(2048, 512, 10, 768, p, None, bank, bank, p)
    assert L.moe_layer_forward(ctypes.byref(good), None, 0, None, None, None, 0, None) == 0
    assert L.moe_layer_forward_host(ctypes.byref(good), None, 0, None, None, None, 0, None) == 0
    assert L.moe_route_topk(None, 0, ctypes.byref(good), None, None, None, None, None, 0, None) == 0
    assert L.moe_combine(None, None, None, None, 0, 10, 2048, None, None, None) == 0
    bad = m.LayerDesc(2050, 512, 10, 768, p, None, bank, bank, p)
    assert L.moe_layer_forward(ctypes.byref(bad), None, 0, None, None, None, 0, None) == MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_combine(None, None, None, None, 0, 33, 2048, None, None, None) == MOE_ERR_UNSUPPORTED_SHAPE
