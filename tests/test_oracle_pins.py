"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks one oracle function against a closed form, a library routine (torch's float8
decoding, numpy's float64 matmul / argsort), brute force on tiny inputs, or the hand-worked
examples in tests/golden. A plausible slip in the oracle (a dropped term, a wrong sign, a swapped
operand, a wrong tie rule) fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------------------------------------
# formats
# ------------------------------------------------------------------------------------------------

def e2m1_from_bits(code):
    """E2M1 from its bit fields: sign | 2 exponent bits (bias 1) | 1 mantissa bit."""
    s = -1.0 if code & 8 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        return s * 0.5 * m
    return s * 2.0 ** (e - 1) * (1 + m / 2)


def test_e2m1_decode_table(orc):
    for c in range(16):
        assert orc.e2m1_value(c) == e2m1_from_bits(c), c
    assert sorted({abs(orc.e2m1_value(c)) for c in range(16)}) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_ue4m3_decode_matches_torch_float8(orc):
    codes = torch.arange(0, 0x7F, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().tolist()
    for c in range(0x7F):
        assert orc.ue4m3_value(c) == ref[c], c
    assert orc.ue4m3_value(0x7E) == 448.0
    assert orc.ue4m3_value(0x01) == 2.0 ** -9
    assert math.isnan(orc.ue4m3_value(0x7F))


def test_ue4m3_encode_matches_torch_on_random_and_ties(orc):
    rng = np.random.default_rng(7)
    vals = list(np.exp(rng.uniform(np.log(2.0 ** -12), np.log(440.0), 3000)).astype(np.float32))
    # every midpoint between neighbouring finite codes is an exact tie
    finite = [orc.ue4m3_value(c) for c in range(0x7F)]
    for a, b in zip(finite[:-1], finite[1:]):
        vals.append(np.float32((a + b) / 2))
    ref = torch.tensor(np.array(vals, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    for v, r in zip(vals, ref):
        assert orc.ue4m3_encode(float(v)) == r, float(v)


def test_ue4m3_encode_saturates_and_zero(orc):
    assert orc.ue4m3_encode(448.0) == 0x7E
    assert orc.ue4m3_encode(463.9) == 0x7E
    assert orc.ue4m3_encode(1e6) == 0x7E
    assert orc.ue4m3_encode(0.0) == 0
    assert orc.ue4m3_encode(2.0 ** -10) == 0  # tie between 0 and 2^-9: even code 0
    assert orc.ue4m3_encode(2.0 ** -10 * 1.0001) == 1


def test_e2m1_encode_ties_and_saturation(orc):
    mags = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    # exact midpoints go to the even code (even mantissa bit)
    expect_tie = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for v, c in expect_tie.items():
        assert orc.e2m1_encode(v) == c, v
        assert orc.e2m1_encode(-v) == c | 8, -v
    # brute force nearest away from ties
    rng = np.random.default_rng(3)
    for v in rng.uniform(-8, 8, 4000).astype(np.float32):
        a = abs(float(v))
        d = [abs(a - m) for m in mags]
        best = int(np.argmin(d))
        if sorted(d)[0] == sorted(d)[1]:
            continue
        assert orc.e2m1_encode(v) == (best | (8 if v < 0 else 0)), float(v)
    assert orc.e2m1_encode(100.0) == 7 and orc.e2m1_encode(-100.0) == 15
    assert orc.e2m1_encode(-0.1) == 8  # sign kept on a value that rounds to zero


def test_round_bf16_matches_torch(orc):
    rng = np.random.default_rng(11)
    v = rng.standard_normal(2000) * 10.0 ** rng.uniform(-3, 3, 2000)
    # doubles that round through float32 may differ from a direct rounding; torch converts the
    # float32 value, so only compare where the float32 value is exact
    v32 = v.astype(np.float32).astype(np.float64)
    ref = torch.tensor(v32, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    for a, r in zip(v32, ref):
        assert orc.round_bf16(a) == r


def _load_golden():
    ex, cur = [], None
    with open(os.path.join(GOLDEN, "nvfp4_worked_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            if key == "example":
                cur = {"name": rest[0]}
                ex.append(cur)
            elif key == "scale":
                cur["scale"] = None if rest[0] == "dynamic" else float(rest[0])
            elif key == "row":
                cur["row"] = np.array([float(v) for v in rest], np.float32)
            elif key == "expect_S":
                cur["S"] = float(rest[0])
            elif key == "expect_sf":
                cur["sf"] = [int(v, 16) for v in rest]
            elif key == "expect_codes":
                cur["codes"] = [int(v, 16) for v in rest]
    return ex


@pytest.mark.parametrize("ex", _load_golden(), ids=lambda e: e["name"])
def test_worked_examples(orc, ex):
    row = ex["row"]
    assert row.size % 16 == 0 and len(ex["codes"]) == row.size and len(ex["sf"]) == row.size // 16
    codes, sf, S = orc.quantize_nvfp4(row[None, :], s_in=ex["scale"])
    assert float(S) == ex["S"]
    assert list(sf[0]) == ex["sf"]
    nibbles = []
    for b in codes[0]:
        nibbles += [int(b) & 15, int(b) >> 4]
    assert nibbles == ex["codes"]


def test_round_trip_exact(orc):
    """encode(decode(q)) == q for power-of-two S, one +-6 per block and one block at sf = 448."""
    rng = np.random.default_rng(5)
    rows, K = 6, 64
    for j in (-12, -8, -3, 0, 2):
        S = np.float32(2.0 ** j)
        codes = rng.integers(0, 16, (rows, K), dtype=np.uint8)
        sf = rng.integers(0x08, 0x7E, (rows, K // 16), dtype=np.uint8)
        for r in range(rows):
            for b in range(K // 16):
                codes[r, b * 16 + rng.integers(16)] = 7 if rng.integers(2) else 15
        sf[2, 1] = 0x7E
        packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
        xhat = orc.dequantize_nvfp4(packed, sf, S)
        x32 = xhat.astype(np.float32)
        assert np.array_equal(x32.astype(np.float64), xhat)  # exactly representable
        c2, s2, S2 = orc.quantize_nvfp4(x32)
        assert S2 == S
        assert np.array_equal(s2, sf)
        assert np.array_equal(c2, packed)


def test_dequantize_matches_bitfield_decode(orc):
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 256, (3, 16), dtype=np.uint8)
    sf = rng.integers(0, 0x7F, (3, 2), dtype=np.uint8)
    S = np.float32(0.37)
    ref = np.zeros((3, 32))
    f8 = torch.tensor(sf.ravel()).view(torch.float8_e4m3fn).double().numpy().reshape(3, 2)
    for r in range(3):
        for k in range(32):
            c = (codes[r, k // 2] >> (4 * (k & 1))) & 15
            ref[r, k] = e2m1_from_bits(int(c)) * f8[r, k // 16] * float(S)
    assert np.array_equal(orc.dequantize_nvfp4(codes, sf, S), ref)


def test_tensor_scale(orc):
    x = np.array([[1.0, -5376.0, 3.0]], np.float32)
    assert orc.tensor_scale(x) == 2.0
    assert orc.tensor_scale(np.zeros((2, 2), np.float32)) == 1.0


# ------------------------------------------------------------------------------------------------
# router
# ------------------------------------------------------------------------------------------------

def _numpy_router(x, w, k, bias=None):
    lg = x.astype(np.float64) @ w[:-1].astype(np.float64).T
    if bias is not None:
        lg = lg + bias
    ids = np.zeros((x.shape[0], k), np.int32)
    for t in range(x.shape[0]):
        order = sorted(range(lg.shape[1]), key=lambda e: (-lg[t, e], e))
        ids[t] = order[:k]
    p = np.exp(lg - lg.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    tw = np.take_along_axis(p, ids, 1)
    tw /= tw.sum(1, keepdims=True)
    g = 1 / (1 + np.exp(-(x.astype(np.float64) @ w[-1].astype(np.float64))))
    return ids, tw, g


def test_router_matches_brute_force(orc):
    rng = np.random.default_rng(1)
    T, H, E, k = 9, 48, 12, 3
    x = rng.standard_normal((T, H)).astype(np.float32)
    w = (rng.standard_normal((E + 1, H)) * 0.3).astype(np.float32)
    ids, tw, g, lg = orc.router(x, w, k, want_logits=True)
    rids, rtw, rg = _numpy_router(x, w, k)
    assert np.array_equal(ids, rids)
    np.testing.assert_allclose(tw, rtw, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(g, rg, rtol=1e-12)
    np.testing.assert_allclose(tw.sum(1), 1.0, atol=1e-12)
    # weights are in routing order (non-increasing)
    assert np.all(np.diff(tw, axis=1) <= 0)


def test_router_ties_pick_lowest_index(orc):
    rng = np.random.default_rng(2)
    T, H, E, k = 4, 32, 8, 3
    x = rng.standard_normal((T, H)).astype(np.float32)
    w = rng.standard_normal((E + 1, H)).astype(np.float32)
    w[5] = w[2]  # experts 2 and 5 always tie
    w[6] = w[2]
    ids, tw, _, _ = orc.router(x, w, E)  # k = E: full order
    for t in range(T):
        order = list(ids[t])
        assert order.index(2) < order.index(5) < order.index(6)
        assert order.index(6) == order.index(2) + 2
        i2 = order.index(2)
        assert tw[t, i2] == tw[t, i2 + 1] == tw[t, i2 + 2]


def test_router_bias_and_k_equals_e(orc):
    rng = np.random.default_rng(4)
    T, H, E = 5, 16, 6
    x = rng.standard_normal((T, H)).astype(np.float32)
    w = rng.standard_normal((E + 1, H)).astype(np.float32)
    bias = np.zeros(E)
    bias[3] = 1e3  # forces expert 3 first everywhere
    ids, tw, _, _ = orc.router(x, w, 2, bias=bias)
    assert np.all(ids[:, 0] == 3)
    np.testing.assert_allclose(tw[:, 0], 1.0, atol=1e-12)
    # k = E: the renormalised weights are the full softmax
    ids, tw, _, lg = orc.router(x, w, E, want_logits=True)
    p = np.exp(lg - lg.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    np.testing.assert_allclose(tw, np.take_along_axis(p, ids, 1), rtol=1e-12)


def test_router_shared_gate_closed_form(orc):
    H, E = 8, 3
    x = np.zeros((2, H), np.float32)
    x[1, 0] = math.log(3.0)
    w = np.zeros((E + 1, H), np.float32)
    w[E, 0] = 1.0
    _, _, g, _ = orc.router(x, w, 1)
    assert g[0] == 0.5
    assert abs(g[1] - 0.75) < 1e-7  # sigmoid(ln 3) = 3/4 (x rounded to float32)


def test_route_from_logits_closed_forms(orc):
    # logits ln 1 .. ln 4 (+ a far-away fifth): softmax ∝ 1, 2, 3, 4, so the top two are experts 3
    # then 2 with renormalised weights 4/7 and 3/7 whatever the other terms of the denominator
    lg = np.log(np.array([[1.0, 2.0, 3.0, 4.0, 1e-9]]))
    ids, tw, g = orc.route_from_logits(lg, 2, gate_logit=np.array([math.log(3.0)]))
    assert ids.tolist() == [[3, 2]]
    np.testing.assert_allclose(tw[0], [4 / 7, 3 / 7], rtol=1e-14)
    assert abs(g[0] - 0.75) < 1e-15
    # k = 1: the single weight is exactly 1; exact ties go to the lowest id, in id order
    ids, tw, g = orc.route_from_logits(np.array([[0.5, 2.0, 2.0, -1.0, 2.0]]), 3)
    assert ids.tolist() == [[1, 2, 4]] and g is None
    np.testing.assert_allclose(tw[0], [1 / 3] * 3, rtol=1e-14)
    ids, tw, _ = orc.route_from_logits(np.array([[7.0, -3.0]]), 1)
    assert ids.tolist() == [[0]] and tw[0, 0] == 1.0


def test_route_from_logits_is_the_routers_decision(orc):
    # the router's selection and weights are route_from_logits applied to its own logits (a
    # logit shift by a constant leaves both unchanged: the softmax is shift-invariant)
    rng = np.random.default_rng(12)
    T, H, E, k = 6, 40, 9, 4
    x = rng.standard_normal((T, H)).astype(np.float32)
    w = (rng.standard_normal((E + 1, H)) * 0.3).astype(np.float32)
    ids, tw, g, lg = orc.router(x, w, k, want_logits=True)
    gate = x.astype(np.float64) @ w[E].astype(np.float64)
    ids2, tw2, g2 = orc.route_from_logits(lg + 5.0, k, gate_logit=gate)
    assert np.array_equal(ids, ids2)
    np.testing.assert_allclose(tw2, tw, rtol=1e-12)
    np.testing.assert_allclose(g2, g, rtol=1e-12)
    rids, rtw, _ = _numpy_router(x, w, k)
    assert np.array_equal(ids2, rids)
    np.testing.assert_allclose(tw2, rtw, rtol=1e-12)


# ------------------------------------------------------------------------------------------------
# permute
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (7, 3, 5), (40, 4, 16), (64, 2, 16)])
def test_permute_brute_force(orc, T, k, E):
    rng = np.random.default_rng(T * 100 + E)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    offsets, perm_src, src_perm = orc.permute(ids, E)
    flat = ids.ravel()
    order = sorted(range(T * k), key=lambda f: (flat[f], f))
    assert list(perm_src) == order
    assert np.array_equal(src_perm[perm_src], np.arange(T * k))
    counts = np.bincount(flat, minlength=E)
    assert list(offsets[: E + 1]) == [0] + list(np.cumsum(counts))
    assert offsets[E + 1] == T * k + T
    for e in range(E):
        seg = perm_src[offsets[e]: offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)


def test_permute_one_expert_takes_all(orc):
    ids = np.zeros((10, 1), np.int32)
    offsets, perm_src, src_perm = orc.permute(ids, 4, with_shared=False)
    assert list(offsets) == [0, 10, 10, 10, 10, 10]
    assert list(perm_src) == list(range(10))


# ------------------------------------------------------------------------------------------------
# grouped GEMM, SwiGLU, combine
# ------------------------------------------------------------------------------------------------

def _np_decode(codes, sf, S):
    rows, K = codes.shape[0], codes.shape[1] * 2
    lut = np.array([e2m1_from_bits(c) for c in range(16)])
    nib = np.zeros((rows, K), np.int64)
    nib[:, 0::2] = codes & 15
    nib[:, 1::2] = codes >> 4
    sfv = torch.tensor(sf.ravel()).view(torch.float8_e4m3fn).double().numpy().reshape(sf.shape)
    return lut[nib] * np.repeat(sfv, 16, axis=1) * float(S)


def test_grouped_gemm_matches_numpy_matmul(orc):
    rng = np.random.default_rng(12)
    G, N, K, P_src = 3, 24, 64, 11
    a = rng.standard_normal((P_src, K)).astype(np.float32)
    ac, asf, sa = orc.quantize_nvfp4(a)
    bw = rng.standard_normal((G, N, K)).astype(np.float32) * 0.1
    bc = np.zeros((G, N, K // 2), np.uint8)
    bsf = np.zeros((G, N, K // 16), np.uint8)
    bs = np.zeros((G, 2), np.float32)
    for g in range(G):
        for h in range(2):
            c, s, S = orc.quantize_nvfp4(bw[g, h * N // 2:(h + 1) * N // 2])
            bc[g, h * N // 2:(h + 1) * N // 2] = c
            bsf[g, h * N // 2:(h + 1) * N // 2] = s
            bs[g, h] = S
    offsets = np.array([0, 4, 4, 9], np.int32)  # an empty group in the middle
    a_row = rng.integers(0, P_src, 9).astype(np.int32)
    out = orc.grouped_gemm(ac, asf, sa, offsets, bc, bsf, bs, a_row=a_row)
    A = _np_decode(ac, asf, sa)
    for g in range(G):
        B = np.concatenate([_np_decode(bc[g, :N // 2], bsf[g, :N // 2], bs[g, 0]),
                            _np_decode(bc[g, N // 2:], bsf[g, N // 2:], bs[g, 1])])
        rows = a_row[offsets[g]:offsets[g + 1]]
        ref = A[rows] @ B.T
        np.testing.assert_allclose(out[offsets[g]:offsets[g + 1]], ref, rtol=1e-13, atol=1e-13)


def test_grouped_gemm_all_ones_closed_form(orc):
    K, N = 128, 8
    ac = np.full((3, K // 2), 0x22, np.uint8)  # code 2 = 1.0 in both nibbles
    asf = np.full((3, K // 16), 0x38, np.uint8)  # UE4M3 0x38 = 1.0
    bc = np.full((2, N, K // 2), 0x22, np.uint8)
    bsf = np.full((2, N, K // 16), 0x38, np.uint8)
    out = orc.grouped_gemm(ac, asf, 1.0, np.array([0, 1, 3], np.int32), bc, bsf,
                           np.ones(2, np.float32))
    assert np.all(out == K)


def test_swiglu_closed_forms(orc):
    I = 3
    gu = np.array([[0.0, math.log(3.0), 50.0, 7.0, 2.0, -1.5]])
    h = orc.swiglu(gu)
    assert h[0, 0] == 0.0
    assert abs(h[0, 1] - np.float32(0.75 * math.log(3.0) * 2.0)) <= 1e-7
    assert abs(h[0, 2] - np.float32(-75.0)) <= 1e-5  # silu(50) = 50 (1 - 2e-22)


def test_combine_one_hot(orc):
    T, k, H = 3, 2, 4
    y = np.zeros((T * k + T, H))
    for p in range(T * k + T):
        y[p] = p + 1
    tw = np.array([[0.75, 0.25], [0.5, 0.5], [1.0, 0.0]])
    src_perm = np.array([5, 0, 1, 2, 3, 4], np.int32)
    g = np.array([0.0, 1.0, 0.5])
    res = np.full((T, H), 2.0, np.float32)
    o64, o16 = orc.combine(y, tw, src_perm, shared_g=g, shared_row0=T * k, residual=res)
    assert np.all(o64[0] == 2 + 0.75 * 6 + 0.25 * 1)
    assert np.all(o64[1] == 2 + 0.5 * 2 + 0.5 * 3 + 1.0 * 8)
    assert np.all(o64[2] == 2 + 1.0 * 4 + 0.5 * 9)
    assert np.array_equal(o16, o64)  # all values are bf16-exact here


# ------------------------------------------------------------------------------------------------
# layer
# ------------------------------------------------------------------------------------------------

def _make_layer(orc, rng, T, H, E, k, I):
    x = rng.standard_normal((T, H)).astype(np.float32)
    w_r = (rng.standard_normal((E + 1, H)) * 0.2).astype(np.float32)
    wgu = [np.zeros((E + 1, 2 * I, H // 2), np.uint8), np.zeros((E + 1, 2 * I, H // 16), np.uint8),
           np.zeros((E + 1, 2), np.float32)]
    wd = [np.zeros((E + 1, H, I // 2), np.uint8), np.zeros((E + 1, H, I // 16), np.uint8),
          np.zeros(E + 1, np.float32)]
    for e in range(E + 1):
        for h in range(2):
            c, s, S = orc.quantize_nvfp4((rng.standard_normal((I, H)) * 0.3).astype(np.float32))
            wgu[0][e, h * I:(h + 1) * I], wgu[1][e, h * I:(h + 1) * I], wgu[2][e, h] = c, s, S
        c, s, S = orc.quantize_nvfp4((rng.standard_normal((H, I)) * 0.3).astype(np.float32))
        wd[0][e], wd[1][e], wd[2][e] = c, s, S
    s_mid = np.full(E + 1, 0.004, np.float32)
    return x, w_r, wgu, wd, s_mid


def _per_token_layer(orc, x, w_r, k, wgu, wd, s_mid, bias=None, residual=None):
    """Independent restatement: loop over tokens and their experts, no permutation."""
    T, H = x.shape
    E = w_r.shape[0] - 1
    I = wd[0].shape[2] * 2
    xc, xs, Sx = orc.quantize_nvfp4(x)
    X = _np_decode(xc, xs, Sx)
    lg = x.astype(np.float64) @ w_r[:E].astype(np.float64).T
    if bias is not None:
        lg = lg + np.asarray(bias, np.float64)[None, :]
    out = np.zeros((T, H)) if residual is None else residual.astype(np.float64).copy()
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-lg[t, e], e))[:k]
        p = np.exp(lg[t] - lg[t].max())
        p /= p.sum()
        wts = p[order] / p[order].sum()
        gate = 1 / (1 + np.exp(-(x[t].astype(np.float64) @ w_r[E].astype(np.float64))))
        for e, wt in list(zip(order, wts)) + [(E, gate)]:
            Wg = _np_decode(wgu[0][e, :I], wgu[1][e, :I], wgu[2][e, 0])
            Wu = _np_decode(wgu[0][e, I:], wgu[1][e, I:], wgu[2][e, 1])
            gg, uu = Wg @ X[t], Wu @ X[t]
            h = (gg / (1 + np.exp(-gg)) * uu).astype(np.float32)
            hc, hs, _ = orc.quantize_nvfp4(h[None, :], s_in=float(s_mid[e]))
            Hq = _np_decode(hc, hs, s_mid[e])[0]
            Wd = _np_decode(wd[0][e], wd[1][e], wd[2][e])
            out[t] += wt * (Wd @ Hq)
    return out


@pytest.mark.parametrize("T,H,E,k,I", [(5, 32, 4, 2, 16), (6, 64, 3, 3, 32), (4, 32, 1, 1, 16)])
def test_layer_equals_per_token_restatement(orc, T, H, E, k, I):
    rng = np.random.default_rng(T * 7 + E)
    x, w_r, wgu, wd, s_mid = _make_layer(orc, rng, T, H, E, k, I)
    r = orc.layer_forward(x, w_r, k, wgu, wd, s_mid)
    ref = _per_token_layer(orc, x, w_r, k, wgu, wd, s_mid)
    np.testing.assert_allclose(r["out_f64"], ref, rtol=1e-12, atol=1e-12)
    # the bf16 output is the nearest bf16 of the FP64 output
    ref16 = torch.tensor(ref).to(torch.float32).to(torch.bfloat16).double().numpy()
    assert np.mean(r["out"] == ref16) > 0.99


def test_layer_sampled_rows_equal_full_call(orc):
    """Computing a subset of tokens with the full call's x scale gives the same rows."""
    rng = np.random.default_rng(21)
    x, w_r, wgu, wd, s_mid = _make_layer(orc, rng, 12, 32, 5, 2, 16)
    full = orc.layer_forward(x, w_r, 2, wgu, wd, s_mid)
    rows = np.array([3, 7, 11])
    sub = orc.layer_forward(x[rows], w_r, 2, wgu, wd, s_mid, x_scale=full["x_scale"])
    np.testing.assert_array_equal(sub["out_f64"], full["out_f64"][rows])


def test_layer_bias_and_residual_equal_per_token_restatement(orc):
    """The workload's logit bias moves selection and weights alike; the residual is added once, in FP64."""
    T, H, E, k, I = 6, 32, 6, 2, 16
    rng = np.random.default_rng(33)
    x, w_r, wgu, wd, s_mid = _make_layer(orc, rng, T, H, E, k, I)
    bias = -1.1 * np.log(np.arange(E) + 1.0)  # the Zipf workload's bias
    res = rng.standard_normal((T, H)).astype(np.float32)
    r = orc.layer_forward(x, w_r, k, wgu, wd, s_mid, bias=bias, residual=res)
    ref = _per_token_layer(orc, x, w_r, k, wgu, wd, s_mid, bias=bias, residual=res)
    np.testing.assert_allclose(r["out_f64"], ref, rtol=1e-12, atol=1e-12)
    # without the bias the selection differs for some token (the bias is not a no-op here)
    plain = orc.layer_forward(x, w_r, k, wgu, wd, s_mid, residual=res)
    assert not np.allclose(plain["out_f64"], r["out_f64"])
    # without the residual the output drops exactly the residual
    nores = orc.layer_forward(x, w_r, k, wgu, wd, s_mid, bias=bias)
    np.testing.assert_allclose(r["out_f64"] - nores["out_f64"], res.astype(np.float64), rtol=0, atol=1e-12)
