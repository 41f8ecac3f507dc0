"""CPU oracle of the NVFP4 (W4A4) routed-MoE layer forward -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline and reference legs of ``bench.py`` may import
this package. It is a plain, slow, FP64-accumulating restatement of the layer (see
``moe_oracle.c`` for the definition of every step and the readings taken where the capy-flash
pages are silent). It shares no code with the GPU library and never calls it.

Parity status of each function (how it is pinned, in ``tests/test_oracle_pins.py``):
  formats / encode  -- exhaustive closed-form tables, hand-worked blocks (tests/golden), round trips
  router            -- brute-force sort, sum of weights, crafted exact ties, bias invariance
  route_from_logits -- closed-form softmax weights on crafted logits, ties, the router's own logits
  permute           -- bijection, stability, offsets = scan(histogram), brute force
  grouped_gemm      -- numpy float64 matmul of the dequantized operands; all-ones closed form
  swiglu / combine  -- closed forms on crafted inputs
  layer_forward     -- an independent per-token nested-loop layer; k = E and E = 1 special cases;
                       with the Zipf logit bias and a residual
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        d, f, i32, i64, u8 = (ctypes.c_double, ctypes.c_float, ctypes.c_int32, ctypes.c_int64,
                              ctypes.c_uint8)
        p = ctypes.c_void_p
        L.orc_e2m1_value.restype = d
        L.orc_e2m1_value.argtypes = [ctypes.c_int]
        L.orc_ue4m3_value.restype = d
        L.orc_ue4m3_value.argtypes = [ctypes.c_int]
        L.orc_e2m1_encode.restype = u8
        L.orc_e2m1_encode.argtypes = [f]
        L.orc_ue4m3_encode.restype = u8
        L.orc_ue4m3_encode.argtypes = [f]
        L.orc_round_bf16.restype = d
        L.orc_round_bf16.argtypes = [d]
        L.orc_tensor_scale.restype = f
        L.orc_tensor_scale.argtypes = [p, i64]
        L.orc_quantize_nvfp4.restype = ctypes.c_int
        L.orc_quantize_nvfp4.argtypes = [p, i64, i64, f, p, p, p]
        L.orc_dequantize_nvfp4.restype = None
        L.orc_dequantize_nvfp4.argtypes = [p, p, f, i64, i64, p]
        L.orc_router.restype = None
        L.orc_router.argtypes = [p, p, p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_int, p, p, p, p]
        L.orc_route_from_logits.restype = None
        L.orc_route_from_logits.argtypes = [p, p, ctypes.c_int, ctypes.c_int, ctypes.c_int, p, p, p]
        L.orc_permute.restype = ctypes.c_int
        L.orc_permute.argtypes = [p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, p, p, p]
        L.orc_grouped_gemm.restype = None
        L.orc_grouped_gemm.argtypes = [p, p, p, ctypes.c_int, p, p, ctypes.c_int, p, p, p,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, p]
        L.orc_swiglu.restype = None
        L.orc_swiglu.argtypes = [p, i64, i64, p]
        L.orc_combine.restype = None
        L.orc_combine.argtypes = [p, ctypes.c_int, ctypes.c_int, i64, p, p, i64, p, p, p, p]
        L.orc_num_threads.restype = ctypes.c_int
        L.orc_num_threads.argtypes = []
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return lib().orc_num_threads()


# ---------------------------------------------------------------------------------------------
# formats
# ---------------------------------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(int(code))


def ue4m3_value(code: int) -> float:
    return lib().orc_ue4m3_value(int(code))


def e2m1_encode(v: float) -> int:
    return int(lib().orc_e2m1_encode(float(np.float32(v))))


def ue4m3_encode(q: float) -> int:
    return int(lib().orc_ue4m3_encode(float(np.float32(q))))


def round_bf16(v: float) -> float:
    return lib().orc_round_bf16(float(v))


def tensor_scale(x) -> float:
    x = _c(x, np.float32)
    return float(lib().orc_tensor_scale(_ptr(x), x.size))


def quantize_nvfp4(x, s_in=None):
    """x: float32 [rows][K] -> (codes uint8 [rows][K/2], sf uint8 [rows][K/16], S float32)."""
    x = _c(x, np.float32)
    rows, K = x.shape
    codes = np.zeros((rows, K // 2), np.uint8)
    sf = np.zeros((rows, K // 16), np.uint8)
    s_out = np.zeros(1, np.float32)
    rc = lib().orc_quantize_nvfp4(_ptr(x), rows, K, float(s_in) if s_in is not None else 0.0,
                                  _ptr(codes), _ptr(sf), _ptr(s_out))
    if rc != 0:
        raise ValueError("oracle quantize: bad shape %r" % (x.shape,))
    return codes, sf, np.float32(s_out[0])


def dequantize_nvfp4(codes, sf, S):
    codes = _c(codes, np.uint8)
    sf = _c(sf, np.uint8)
    rows, K = codes.shape[0], codes.shape[1] * 2
    out = np.zeros((rows, K), np.float64)
    lib().orc_dequantize_nvfp4(_ptr(codes), _ptr(sf), float(S), rows, K, _ptr(out))
    return out


# ---------------------------------------------------------------------------------------------
# layer steps
# ---------------------------------------------------------------------------------------------

def router(x, w_router, k, has_shared=True, bias=None, want_logits=False):
    """x: [T][H] float32 (bf16 values), w_router: [E + has_shared][H] float32.
    Returns (topk_ids int32 [T][k], topk_w float64 [T][k], shared_g float64 [T] or None,
    logits float64 [T][E] or None)."""
    x = _c(x, np.float32)
    w = _c(w_router, np.float32)
    T, H = x.shape
    E = w.shape[0] - (1 if has_shared else 0)
    ids = np.zeros((T, k), np.int32)
    tw = np.zeros((T, k), np.float64)
    g = np.zeros(T, np.float64) if has_shared else None
    lg = np.zeros((T, E), np.float64) if want_logits else None
    b = _c(bias, np.float64) if bias is not None else None
    lib().orc_router(_ptr(x), _ptr(w), _ptr(b), T, H, E, k, int(has_shared), _ptr(ids), _ptr(tw),
                     _ptr(g), _ptr(lg))
    return ids, tw, g, lg


def route_from_logits(logits, k, gate_logit=None):
    """The routing decision on given logits [T][E] (any float dtype, taken as FP64): FP64 softmax
    over all E, top k by (logit desc, index asc), weights renormalised over the k.
    Returns (topk_ids int32 [T][k], topk_w float64 [T][k], shared_g float64 [T] or None)."""
    lg = _c(logits, np.float64)
    T, E = lg.shape
    ids = np.zeros((T, k), np.int32)
    tw = np.zeros((T, k), np.float64)
    gl = _c(gate_logit, np.float64) if gate_logit is not None else None
    g = np.zeros(T, np.float64) if gl is not None else None
    lib().orc_route_from_logits(_ptr(lg), _ptr(gl), T, E, k, _ptr(ids), _ptr(tw), _ptr(g))
    return ids, tw, g


def permute(topk_ids, E, with_shared=True):
    ids = _c(topk_ids, np.int32)
    T, k = ids.shape
    offsets = np.zeros(E + 2, np.int32)
    perm_src = np.zeros(T * k, np.int32)
    src_perm = np.zeros(T * k, np.int32)
    rc = lib().orc_permute(_ptr(ids), T, k, E, int(with_shared), _ptr(offsets), _ptr(perm_src),
                           _ptr(src_perm))
    if rc != 0:
        raise ValueError("oracle permute: expert id out of range")
    return offsets, perm_src, src_perm


def grouped_gemm(a_codes, a_sf, a_scale, offsets, b_codes, b_sf, b_scale, a_row=None):
    """FP64 grouped GEMM of dequantized NVFP4 operands. a_scale: scalar or [G];
    b_codes [G][N][K/2], b_sf [G][N][K/16], b_scale [G] or [G][2] (gate | up column halves).
    Returns out float64 [offsets[-1]][N]."""
    a_codes = _c(a_codes, np.uint8)
    a_sf = _c(a_sf, np.uint8)
    b_codes = _c(b_codes, np.uint8)
    b_sf = _c(b_sf, np.uint8)
    offsets = _c(offsets, np.int32)
    G, N, Kh = b_codes.shape
    K = Kh * 2
    a_scale = np.atleast_1d(np.asarray(a_scale, np.float32))
    per_group = 1 if a_scale.size > 1 else 0
    b_scale = np.asarray(b_scale, np.float32).reshape(G, -1).copy()
    nscale = b_scale.shape[1]
    P = int(offsets[G])
    out = np.zeros((P, N), np.float64)
    row = _c(a_row, np.int32) if a_row is not None else None
    lib().orc_grouped_gemm(_ptr(a_codes), _ptr(a_sf), _ptr(a_scale), per_group, _ptr(row),
                           _ptr(offsets), G, _ptr(b_codes), _ptr(b_sf), _ptr(b_scale), nscale, N, K,
                           _ptr(out))
    return out


def swiglu(gu):
    gu = _c(gu, np.float64)
    P, N2 = gu.shape
    I = N2 // 2
    h = np.zeros((P, I), np.float32)
    lib().orc_swiglu(_ptr(gu), P, I, _ptr(h))
    return h


def combine(y, topk_w, src_perm, shared_g=None, shared_row0=0, residual=None):
    """Weighted un-permute. Returns (out_f64 [T][H], out_bf16 [T][H] as float64)."""
    y = _c(y, np.float64)
    tw = _c(topk_w, np.float64)
    T, k = tw.shape
    H = y.shape[1]
    sp = _c(src_perm, np.int32)
    g = _c(shared_g, np.float64) if shared_g is not None else None
    res = _c(residual, np.float32) if residual is not None else None
    o64 = np.zeros((T, H), np.float64)
    o16 = np.zeros((T, H), np.float64)
    lib().orc_combine(_ptr(y), T, k, H, _ptr(tw), _ptr(g), int(shared_row0), _ptr(sp), _ptr(res),
                      _ptr(o64), _ptr(o16))
    return o64, o16


def requantize_groups(h, offsets, s_mid):
    """Encode the FP32 intermediate h [P][I] group by group with the static scale s_mid[g]."""
    P, I = h.shape
    codes = np.zeros((P, I // 2), np.uint8)
    sf = np.zeros((P, I // 16), np.uint8)
    G = len(offsets) - 1
    for g in range(G):
        p0, p1 = int(offsets[g]), int(offsets[g + 1])
        if p1 > p0:
            c, s, _ = quantize_nvfp4(h[p0:p1], s_in=float(s_mid[g]))
            codes[p0:p1] = c
            sf[p0:p1] = s
    return codes, sf


def layer_forward(x, w_router, k, wgu, wd, s_mid, bias=None, residual=None, x_scale=None):
    """The whole layer, step by step, in the order the layer is defined.

    x: [T][H] float32 (bf16 values); w_router: [E+1][H] (last row = shared gate);
    wgu = (codes [E+1][2I][H/2], sf [E+1][2I][H/16], scale [E+1][2]);
    wd  = (codes [E+1][H][I/2],  sf [E+1][H][I/16],  scale [E+1]);
    s_mid: [E+1] static scales of the intermediate; x_scale: tensor scale of x when the rows
    given are a sample of a larger call (default: computed from x).
    Returns a dict with every intermediate result."""
    x = _c(x, np.float32)
    T, H = x.shape
    E = w_router.shape[0] - 1
    ids, tw, g, logits = router(x, w_router, k, True, bias, want_logits=True)
    xc, xs, Sx = quantize_nvfp4(x, s_in=x_scale)
    offsets, perm_src, src_perm = permute(ids, E, True)
    row_token = np.concatenate([perm_src // k, np.arange(T, dtype=np.int32)]).astype(np.int32)
    gu = grouped_gemm(xc, xs, Sx, offsets, wgu[0], wgu[1], wgu[2], a_row=row_token)
    h = swiglu(gu)
    hc, hs = requantize_groups(h, offsets, s_mid)
    y = grouped_gemm(hc, hs, np.asarray(s_mid, np.float32), offsets, wd[0], wd[1], wd[2])
    o64, o16 = combine(y, tw, src_perm, shared_g=g, shared_row0=T * k, residual=residual)
    return dict(topk_ids=ids, topk_w=tw, shared_g=g, logits=logits, x_codes=xc, x_sf=xs, x_scale=Sx,
                offsets=offsets, perm_src=perm_src, src_perm=src_perm, row_token=row_token, gu=gu,
                h=h, h_codes=hc, h_sf=hs, y=y, out_f64=o64, out=o16)
