"""Python binding of libmoe_nvfp4 (include/moe_nvfp4.h): NVFP4 W4A4 routed-MoE layer forward on sm_103a.

Argument marshalling only: every step of the layer runs in the library's CUDA kernels. PyTorch
provides device memory and the current stream. There is no CPU fallback: every call raises if
the shared library is missing or returns an error.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmoe_nvfp4.so")

EPI_F32, EPI_BF16, EPI_SWIGLU_NVFP4 = 0, 1, 2
SCHED_AUTO, SCHED_ACT_ON_M, SCHED_WEIGHTS_ON_M, SCHED_WIDE, SCHED_WIDE_ROWS = 0, 0x100, 0x200, 0x400, 0x800
SCHED_WEIGHTS_RESIDENT = 0x1000

ENTRY_POINTS = (
    "moe_quantize_nvfp4", "moe_quantize_nvfp4_f32", "moe_route_topk", "moe_permute", "moe_prepack_nvfp4",
    "moe_grouped_gemm_nvfp4", "moe_combine", "moe_layer_forward", "moe_layer_forward_profiled", "moe_workspace_bytes",
    "moe_read_device_status", "moe_status_string", "moe_last_error_detail", "moe_route_topk_noalloc",
    "moe_layer_forward_host", "moe_workspace_bytes_host", "moe_layer_workspace_view",
    "moe_set_wait_test_hook",
)


class MoeError(RuntimeError):
    def __init__(self, status, detail):
        super().__init__("%s (%s)" % (detail, status))
        self.status = status


class NvFp4Bank(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("sf", ctypes.c_void_p), ("gscale", ctypes.c_void_p)]


class LayerDesc(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int), ("I", ctypes.c_int),
                ("w_router", ctypes.c_void_p), ("logit_bias", ctypes.c_void_p),
                ("w_gate_up", NvFp4Bank), ("w_down", NvFp4Bank), ("s_mid", ctypes.c_void_p)]


class LayerView(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "bytes", "x_scale", "x_codes", "x_sf", "logits", "logits_ld", "topk_ids", "topk_w", "shared_g",
        "permutation_in_workspace", "expert_offsets", "perm_src", "src_perm", "row_token", "h_codes", "h_sf",
        "h_block_rows", "y", "route_first")]


_lib = None


def lib():
    """Load the shared library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmoe_nvfp4.so is not built (%s); run nvfp4_w4a4_mixture_gb300.build.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [i32]
        L.moe_last_error_detail.restype = ctypes.c_char_p
        L.moe_last_error_detail.argtypes = []
        L.moe_workspace_bytes.restype = sz
        L.moe_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
        L.moe_workspace_bytes_host.restype = sz
        L.moe_workspace_bytes_host.argtypes = [i32, i32, i32, i32, i32]
        L.moe_read_device_status.restype = i32
        L.moe_read_device_status.argtypes = [vp, vp]
        for name in ("moe_quantize_nvfp4", "moe_quantize_nvfp4_f32"):
            f = getattr(L, name)
            f.restype = i32
            f.argtypes = [vp, i64, i64, vp, vp, vp, vp, vp, sz, vp]
        L.moe_route_topk.restype = i32
        L.moe_route_topk.argtypes = [vp, i32, ctypes.POINTER(LayerDesc), vp, vp, vp, vp, vp, sz, vp]
        L.moe_route_topk_noalloc.restype = i32
        L.moe_route_topk_noalloc.argtypes = [vp, i32, ctypes.POINTER(LayerDesc), vp, vp, vp, vp, vp]
        L.moe_permute.restype = i32
        L.moe_permute.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
        L.moe_prepack_nvfp4.restype = i32
        L.moe_prepack_nvfp4.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp]
        L.moe_grouped_gemm_nvfp4.restype = i32
        L.moe_grouped_gemm_nvfp4.argtypes = [vp, vp, vp, i32, vp, vp, i32, i64, ctypes.POINTER(NvFp4Bank), i32, i32,
                                             i32, i32, vp, vp, vp, vp, sz, vp]
        L.moe_combine.restype = i32
        L.moe_combine.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, vp, vp]
        L.moe_layer_forward.restype = i32
        L.moe_layer_forward.argtypes = [ctypes.POINTER(LayerDesc), vp, i32, vp, vp, vp, sz, vp]
        L.moe_layer_forward_host.restype = i32
        L.moe_layer_forward_host.argtypes = [ctypes.POINTER(LayerDesc), vp, i32, vp, vp, vp, sz, vp]
        L.moe_set_wait_test_hook.restype = i32
        L.moe_set_wait_test_hook.argtypes = [vp, ctypes.c_uint, i32, vp]
        L.moe_layer_workspace_view.restype = i32
        L.moe_layer_workspace_view.argtypes = [ctypes.POINTER(LayerDesc), i32, ctypes.POINTER(LayerView)]
        L.moe_layer_forward_profiled.restype = i32
        L.moe_layer_forward_profiled.argtypes = [ctypes.POINTER(LayerDesc), vp, i32, vp, vp, vp, sz, vp,
                                                 ctypes.POINTER(vp), i32]
        _lib = L
    return _lib


def _check(status):
    if status != 0:
        L = lib()
        raise MoeError(L.moe_status_string(status).decode(), L.moe_last_error_detail().decode())


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def moe_workspace_bytes(H, E, k, I, T):
    return int(lib().moe_workspace_bytes(H, E, k, I, T))


def moe_workspace_bytes_host(H, E, k, I, T):
    return int(lib().moe_workspace_bytes_host(H, E, k, I, T))


class Workspace:
    """Device scratch for the library calls (header zeroed once)."""

    def __init__(self, nbytes, device="cuda"):
        self.nbytes = int(max(nbytes, 4096))
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device)
        off = (-self.buf.data_ptr()) % 256
        self.tensor = self.buf[off: off + self.nbytes]
        self.tensor[:256].zero_()

    @property
    def ptr(self):
        return ctypes.c_void_p(self.tensor.data_ptr())


_default_ws = {}


def _ws(nbytes):
    dev = torch.cuda.current_device()
    w = _default_ws.get(dev)
    if w is None or w.nbytes < nbytes:
        w = Workspace(nbytes)
        _default_ws[dev] = w
    return w


def moe_set_wait_test_hook(ws, wait_limit_us, ready_extra):
    """Test hook: the expert GEMMs' wait for a token block's intermediate gives up after
    wait_limit_us (0: default) and needs ready_extra more completions (0: none); (0, 0) restores."""
    _check(lib().moe_set_wait_test_hook(ws.ptr, int(wait_limit_us), int(ready_extra), _stream()))


def moe_read_device_status(ws=None):
    ws = ws or _ws(4096)
    _check(lib().moe_read_device_status(ws.ptr, _stream()))


def _bf16_bits(t):
    assert t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous()
    return t


def moe_quantize_nvfp4(x, s_in=None, ws=None, out=None):
    """x: bf16 or fp32 [rows, K] CUDA tensor -> (codes u8 [rows, K/2], sf u8 [rows, K/16], S f32 [1]).
    out: optional preallocated (codes, sf, s) contiguous views to write into."""
    assert x.is_cuda and x.is_contiguous() and x.dim() == 2
    rows, K = x.shape
    if out is None:
        codes = torch.empty(rows, K // 2, dtype=torch.uint8, device=x.device)
        sf = torch.empty(rows, K // 16, dtype=torch.uint8, device=x.device)
        s_out = torch.empty(1, dtype=torch.float32, device=x.device)
    else:
        codes, sf, s_out = out
        assert codes.is_contiguous() and sf.is_contiguous() and codes.numel() == rows * K // 2
        assert sf.numel() == rows * K // 16
    ws = ws or _ws(4096)
    f = lib().moe_quantize_nvfp4 if x.dtype == torch.bfloat16 else lib().moe_quantize_nvfp4_f32
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("x must be bf16 or fp32")
    _check(f(_p(x), rows, K, _p(s_in), _p(codes), _p(sf), _p(s_out), ws.ptr, ws.nbytes, _stream()))
    return codes, sf, s_out


def moe_prepack_nvfp4(codes, sf, gate_up_interleave):
    """codes u8 [G, N, K/2], sf u8 [G, N, K/16] (row-major) -> prepacked (codes [G, ceil(K/256), N, 128]
    K-slabs, sf tiles)."""
    G, N, Kh = codes.shape
    K = Kh * 2
    codes_out = torch.empty(G, (K + 255) // 256, N, 128, dtype=torch.uint8, device=codes.device)
    sf_out = torch.empty(G * (N // 128) * (K // 64) * 512, dtype=torch.uint8, device=codes.device)
    _check(lib().moe_prepack_nvfp4(_p(codes), _p(sf), G, N, K, int(gate_up_interleave), _p(codes_out), _p(sf_out),
                                   _stream()))
    return codes_out, sf_out


class MoeLayer:
    """Device tensors of one MoE layer plus its C descriptor.

    w_router: bf16 [E+1, H] (row E = shared gate); gate_up: (codes [E+1, 2I, H/2], sf [E+1, 2I, H/16],
    gscale f32 [E+1, 2]) row-major; down: (codes [E+1, H, I/2], sf [E+1, H, I/16], gscale [E+1]);
    s_mid f32 [E+1]; logit_bias nullable f32 [E]. The expert banks are prepacked on the device."""

    def __init__(self, H, E, k, I, w_router, gate_up, down, s_mid, logit_bias=None, prepacked=False):
        self.H, self.E, self.k, self.I = H, E, k, I
        self.w_router = _bf16_bits(w_router)
        if prepacked:
            self.gu_codes, self.gu_sf, self.gu_scale = gate_up
            self.dn_codes, self.dn_sf, self.dn_scale = down
        else:
            self.gu_codes, self.gu_sf = moe_prepack_nvfp4(gate_up[0], gate_up[1], True)
            self.gu_scale = gate_up[2].contiguous()
            self.dn_codes, self.dn_sf = moe_prepack_nvfp4(down[0], down[1], False)
            self.dn_scale = down[2].contiguous()
        self.s_mid = s_mid.contiguous()
        self.logit_bias = logit_bias.contiguous() if logit_bias is not None else None
        self.desc = LayerDesc(H, E, k, I, self.w_router.data_ptr(),
                              self.logit_bias.data_ptr() if self.logit_bias is not None else None,
                              NvFp4Bank(self.gu_codes.data_ptr(), self.gu_sf.data_ptr(), self.gu_scale.data_ptr()),
                              NvFp4Bank(self.dn_codes.data_ptr(), self.dn_sf.data_ptr(), self.dn_scale.data_ptr()),
                              self.s_mid.data_ptr())

    def workspace_bytes(self, T):
        return moe_workspace_bytes(self.H, self.E, self.k, self.I, T)


def moe_route_topk(x, layer, want_logits=False, ws=None):
    T = x.shape[0]
    dev = x.device
    ids = torch.empty(T, layer.k, dtype=torch.int32, device=dev)
    w = torch.empty(T, layer.k, dtype=torch.float32, device=dev)
    g = torch.empty(T, dtype=torch.float32, device=dev)
    lg = torch.empty(T, layer.E, dtype=torch.float32, device=dev) if want_logits else None
    ws = ws or _ws(layer.workspace_bytes(T))
    _check(lib().moe_route_topk(_p(_bf16_bits(x)), T, ctypes.byref(layer.desc), _p(ids), _p(w), _p(g), _p(lg), ws.ptr,
                                ws.nbytes, _stream()))
    return ids, w, g, lg


def moe_permute(topk_ids, E, with_shared=True, ws=None):
    T, k = topk_ids.shape
    dev = topk_ids.device
    offsets = torch.empty(E + 2, dtype=torch.int32, device=dev)
    perm_src = torch.empty(T * k, dtype=torch.int32, device=dev)
    src_perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    row_token = torch.empty(T * k + (T if with_shared else 0), dtype=torch.int32, device=dev)
    ws = ws or _ws(moe_workspace_bytes(128, E, k, 128, T))
    _check(lib().moe_permute(_p(topk_ids.contiguous()), T, k, E, int(with_shared), _p(offsets), _p(perm_src),
                             _p(src_perm), _p(row_token), ws.ptr, ws.nbytes, _stream()))
    return offsets, perm_src, src_perm, row_token


def moe_grouped_gemm_nvfp4(a_codes, a_sf, a_scale, group_offsets, p_max, b_codes, b_sf, b_scale, N, K, gate_up,
                           epilogue, a_row_index=None, epi_scale=None, ws=None, schedule=SCHED_AUTO):
    """Grouped GEMM over a prepacked bank. Returns out (and out_sf for the SwiGLU epilogue)."""
    G = group_offsets.numel() - 1
    dev = a_codes.device
    P = int(p_max)
    out_sf = None
    if epilogue == EPI_F32:
        out = torch.empty(P, N, dtype=torch.float32, device=dev)
    elif epilogue == EPI_BF16:
        out = torch.empty(P, N, dtype=torch.bfloat16, device=dev)
    else:
        out = torch.empty(P, N // 4, dtype=torch.uint8, device=dev)
        out_sf = torch.empty(P, N // 32, dtype=torch.uint8, device=dev)
    bank = NvFp4Bank(b_codes.data_ptr(), b_sf.data_ptr(), b_scale.data_ptr())
    ws = ws or _ws(256 + 4 * (G + 1) + 4096)
    per_group = int(a_scale.numel() > 1)
    _check(lib().moe_grouped_gemm_nvfp4(_p(a_codes), _p(a_sf), _p(a_scale), per_group, _p(a_row_index),
                                        _p(group_offsets), G, P, ctypes.byref(bank), N, K, int(gate_up),
                                        epilogue | schedule,
                                        _p(epi_scale), _p(out), _p(out_sf), ws.ptr, ws.nbytes, _stream()))
    return (out, out_sf) if epilogue == EPI_SWIGLU_NVFP4 else out


def moe_combine(y, topk_w, src_perm, shared_g=None, residual=None):
    T, k = topk_w.shape
    H = y.shape[1]
    out = torch.empty(T, H, dtype=torch.bfloat16, device=y.device)
    _check(lib().moe_combine(_p(_bf16_bits(y)), _p(topk_w), _p(shared_g), _p(src_perm), T, k, H,
                             _p(residual), _p(out), _stream()))
    return out


def moe_layer_forward(layer, x, residual=None, out=None, ws=None):
    T = x.shape[0]
    if out is None:
        out = torch.empty(T, layer.H, dtype=torch.bfloat16, device=x.device)
    ws = ws or _ws(layer.workspace_bytes(T))
    _check(lib().moe_layer_forward(ctypes.byref(layer.desc), _p(_bf16_bits(x)), T, _p(residual), _p(out), ws.ptr,
                                   ws.nbytes, _stream()))
    return out


def moe_layer_forward_host(layer, x, residual=None, out=None, ws=None):
    """The layer on host tensors (bf16 [T][H] on the CPU; page-locked keeps the call asynchronous):
    the copies in and out and the layer are enqueued on the current stream. `out` holds the result
    once that stream has passed this call."""
    T = x.shape[0]
    for t in (x, residual, out):
        assert t is None or (t.dtype == torch.bfloat16 and not t.is_cuda and t.is_contiguous())
    if out is None:
        out = torch.empty(T, layer.H, dtype=torch.bfloat16).pin_memory()
    ws = ws or _ws(moe_workspace_bytes_host(layer.H, layer.E, layer.k, layer.I, T))
    _check(lib().moe_layer_forward_host(ctypes.byref(layer.desc), _p(x), T, _p(residual), _p(out), ws.ptr, ws.nbytes,
                                        _stream()))
    return out


def moe_layer_workspace_view(layer, T):
    """The byte offsets of the layer's intermediate results in a forward's workspace (LayerView)."""
    v = LayerView()
    _check(lib().moe_layer_workspace_view(ctypes.byref(layer.desc), T, ctypes.byref(v)))
    return v


def layer_intermediates(layer, T, ws):
    """Views (no copies, no arithmetic) of the intermediate results that the last moe_layer_forward of
    T tokens left in workspace `ws`, at the offsets moe_layer_workspace_view reports. Read them once
    the forward's stream has passed it. Keys: x_scale, x_codes, x_sf, logits [T][E+1] (column E: the
    shared-gate logit), topk_ids, topk_w, shared_g, h_codes, h_sf (tiles), y, route_first (the fused
    router ran before the encoder); with the permutation in the workspace also expert_offsets,
    perm_src, src_perm, row_token."""
    v = moe_layer_workspace_view(layer, T)
    H, E, k, I = layer.H, layer.E, layer.k, layer.I
    buf = ws.tensor
    assert buf.numel() >= v.bytes

    def at(off, nbytes, dtype, shape):
        return buf[off: off + nbytes].view(dtype).reshape(shape)

    P = T * k + T
    n_blocks_max = (P + v.h_block_rows - 1) // v.h_block_rows + E + 1
    out = dict(
        x_scale=at(v.x_scale, 4, torch.float32, (1,)),
        x_codes=at(v.x_codes, T * H // 2, torch.uint8, (T, H // 2)),
        x_sf=at(v.x_sf, T * H // 16, torch.uint8, (T, H // 16)),
        logits=at(v.logits, T * v.logits_ld * 4, torch.float32, (T, v.logits_ld))[:, : E + 1],
        topk_ids=at(v.topk_ids, T * k * 4, torch.int32, (T, k)),
        topk_w=at(v.topk_w, T * k * 4, torch.float32, (T, k)),
        shared_g=at(v.shared_g, T * 4, torch.float32, (T,)),
        h_codes=at(v.h_codes, P * I // 2, torch.uint8, (P, I // 2)),
        h_sf=at(v.h_sf, n_blocks_max * (I // 64) * 512, torch.uint8, (n_blocks_max, I // 64, 512)),
        h_block_rows=int(v.h_block_rows),
        y=at(v.y, P * H * 2, torch.bfloat16, (P, H)),
        permutation_in_workspace=bool(v.permutation_in_workspace),
        route_first=bool(v.route_first),
    )
    if v.permutation_in_workspace:
        out.update(expert_offsets=at(v.expert_offsets, (E + 2) * 4, torch.int32, (E + 2,)),
                   perm_src=at(v.perm_src, T * k * 4, torch.int32, (T * k,)),
                   src_perm=at(v.src_perm, T * k * 4, torch.int32, (T * k,)),
                   row_token=at(v.row_token, P * 4, torch.int32, (P,)))
    return out


LAYER_STAGES = ("quantize", "route", "permute", "experts", "combine")


def moe_layer_forward_profiled(layer, x, events, residual=None, out=None, ws=None):
    """moe_layer_forward recording 6 torch.cuda.Event objects (already created, enable_timing) at the
    stage boundaries of LAYER_STAGES."""
    T = x.shape[0]
    if out is None:
        out = torch.empty(T, layer.H, dtype=torch.bfloat16, device=x.device)
    ws = ws or _ws(layer.workspace_bytes(T))
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event on its first record
            e.record()
    handles = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(lib().moe_layer_forward_profiled(ctypes.byref(layer.desc), _p(_bf16_bits(x)), T, _p(residual), _p(out),
                                            ws.ptr, ws.nbytes, _stream(), handles, len(events)))
    return out
