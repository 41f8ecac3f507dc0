"""GPU parity: every call of the C ABI against the CPU oracle on the same seeded inputs.

Bars: bit-exact for codes, block scales, tensor scales, expert ids and routing order, offsets and
permutation indices; the gate/up GEMM (FP32 out) within 1e-5 relative Frobenius error (overall and
per expert); the layer output within 2e-2 relative Frobenius error; >= 99.9 % of the requantized
intermediate codes identical; routing weights within 1e-6.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from nvfp4_w4a4_mixture_gb300 import workloads as wl
from tests import inputs as I_

pytestmark = pytest.mark.gpu

GEMM_TOL = 1e-5
LAYER_TOL = 2e-2
CODE_MATCH = 0.999
W_TOL = 1e-6


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_w4a4_mixture_gb300 as m
    from nvfp4_w4a4_mixture_gb300 import build

    build.build()
    m.lib()
    return m


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def bf16_dev(x32):
    return torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16).cuda()


def nibbles(codes):
    c = np.asarray(codes)
    out = np.empty(c.shape[:-1] + (c.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = c & 15
    out[..., 1::2] = c >> 4
    return out


def gpu_layer(m, case):
    E, H, I, k = case["E"], case["H"], case["I"], case["k"]
    gu, dn = case["gu"], case["dn"]
    layer = m.MoeLayer(H, E, k, I, bf16_dev(case["w_r"]),
                       (dev(gu[0]), dev(gu[1]), dev(gu[2])), (dev(dn[0]), dev(dn[1]), dev(dn[2])),
                       dev(case["s_mid"]), logit_bias=None if case["bias"] is None else dev(case["bias"]))
    return layer


# ------------------------------------------------------------------------------------------------
# quantize
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("rows,K", [(64, 256), (1, 16), (3, 48), (1000, 2064), (4, 2048)])
def test_quantize_bf16_bitexact(moe, rows, K):
    x = wl.gen_x(rows * 7 + K, rows, K)
    c_ref, s_ref, S_ref = oracle.quantize_nvfp4(x)
    codes, sf, S = moe.moe_quantize_nvfp4(bf16_dev(x))
    assert np.float32(S.item()) == S_ref
    np.testing.assert_array_equal(sf.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(codes.cpu().numpy(), c_ref)


def test_quantize_fp32_weights_bitexact(moe):
    g, u, d = wl.gen_expert(0, 3, 2048, 768)
    for w in (g, d):
        c_ref, s_ref, S_ref = oracle.quantize_nvfp4(w)
        codes, sf, S = moe.moe_quantize_nvfp4(dev(w))
        assert np.float32(S.item()) == S_ref
        np.testing.assert_array_equal(sf.cpu().numpy(), s_ref)
        np.testing.assert_array_equal(codes.cpu().numpy(), c_ref)


def test_quantize_golden_examples(moe):
    from tests.test_oracle_pins import _load_golden

    for ex in _load_golden():
        row = ex["row"][None, :]
        s_in = None if ex["scale"] is None else dev(np.array([ex["scale"]], np.float32))
        codes, sf, S = moe.moe_quantize_nvfp4(dev(row), s_in=s_in)
        assert S.item() == ex["S"], ex["name"]
        assert list(sf.cpu().numpy()[0]) == ex["sf"], ex["name"]
        assert list(nibbles(codes.cpu().numpy())[0]) == ex["codes"], ex["name"]


def test_quantize_static_scale_edge_values(moe):
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((32, 128)) * np.exp(rng.uniform(-12, 6, (32, 1)))).astype(np.float32)
    x[0] = 0.0
    x[1, :16] = 2.0 ** -20  # underflows to a zero block scale
    x[2] = 1e4              # saturates
    x[3, 5] = -0.0
    for S in (2.0 ** -8, 0.013, 7.5):
        c_ref, s_ref, _ = oracle.quantize_nvfp4(x, s_in=S)
        codes, sf, Sd = moe.moe_quantize_nvfp4(dev(x), s_in=dev(np.array([S], np.float32)))
        np.testing.assert_array_equal(sf.cpu().numpy(), s_ref)
        np.testing.assert_array_equal(codes.cpu().numpy(), c_ref)


def _boundary_blocks(S, n_blocks, seed):
    """FP32 blocks whose quotients v / d lie on and within 3 FP32 ulps of the E2M1 rounding boundaries
    (midpoints and grid values), and whose amax / (6 S) lies on and near UE4M3 midpoints, for a static
    tensor scale S."""
    rng = np.random.default_rng(seed)
    S = np.float32(S)
    six_s = np.float32(np.float32(6.0) * S)
    e2m1_edges = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    e4m3 = [1.0, 1.125, 1.25, 1.375, 1.5, 1.625, 1.75, 1.875, 2.0]

    def step(v, k):
        v = np.float32(v)
        for _ in range(abs(k)):
            v = np.nextafter(v, np.float32(np.inf if k > 0 else -np.inf), dtype=np.float32)
        return v

    out = np.zeros((n_blocks, 16), np.float32)
    for b in range(n_blocks):
        lo = rng.integers(0, len(e4m3) - 1)
        scale = np.float32(2.0 ** rng.integers(-6, 4))
        if b % 2:
            q = np.float32((e4m3[lo] + e4m3[lo + 1]) / 2) * scale  # an UE4M3 midpoint
        else:
            q = np.float32(e4m3[lo]) * scale
        amax = step(np.float32(q * six_s), int(rng.integers(-3, 4)))
        dsf = np.float32(q)  # the scale the block should get, up to the rounding being probed
        d = np.float32(dsf * S)
        out[b, 0] = amax * (1 if rng.random() < 0.5 else -1)
        for i in range(1, 16):
            m = e2m1_edges[rng.integers(0, len(e2m1_edges))]
            v = step(np.float32(np.float32(m) * d), int(rng.integers(-3, 4)))
            v = min(v, np.float32(abs(out[b, 0])))  # amax stays the block's maximum
            out[b, i] = v * (1 if rng.random() < 0.5 else -1)
        rng.shuffle(out[b])
    return out


@pytest.mark.parametrize("S,n_blocks", [(0.1, 3000), (0.013, 6000), (1.0 / 3.0, 300)])
def test_quantize_codes_at_rounding_boundaries(moe, S, n_blocks):
    # the encoder decides codes from products with a correctly rounded reciprocal and divides only
    # when a quotient is within about 2^-20 of a rounding boundary: quotients placed on and a few
    # ulps around every boundary must give the oracle's codes and scales bit for bit (3000 and 6000
    # blocks take the two-launch quantizer, 300 the one-CTA one)
    x = _boundary_blocks(S, n_blocks, seed=n_blocks).reshape(-1, 64)
    c_ref, s_ref, _ = oracle.quantize_nvfp4(x, s_in=S)
    codes, sf, _ = moe.moe_quantize_nvfp4(dev(x), s_in=dev(np.array([S], np.float32)))
    np.testing.assert_array_equal(sf.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(codes.cpu().numpy(), c_ref)


# ------------------------------------------------------------------------------------------------
# router
# ------------------------------------------------------------------------------------------------

def _check_route_values(w, g, lg, w_ref, g_ref, lg_ref, ids=None, k=None):
    # The logits are FP32 sums (their order differs between the CUDA-core and tensor-core routers);
    # the renormalised softmax moves each weight by at most half the largest logit change (its
    # Jacobian rows sum to 2 p (1 - p) <= 1/2 in absolute value) and the sigmoid gate by a quarter
    # of it, so against the oracle's own logits the weights are held to the logits' error plus FP32
    # rounding. The routing arithmetic itself is held to 1e-6: the oracle's FP64 softmax and
    # renormalisation of the kernel's OWN FP32 logits must give the same ids and weights.
    lg = lg.cpu().numpy()
    dl = float(np.max(np.abs(lg - lg_ref)))
    assert dl <= 1e-4, dl
    w = w.cpu().numpy()
    assert np.max(np.abs(w - w_ref)) <= dl + W_TOL
    assert np.max(np.abs(w.sum(1) - 1.0)) <= W_TOL
    assert np.max(np.abs(g.cpu().numpy() - g_ref)) <= 0.5 * dl + W_TOL
    if ids is not None:
        ids2, w2, _ = oracle.route_from_logits(lg.astype(np.float64), k)
        np.testing.assert_array_equal(ids2, ids.cpu().numpy())
        assert np.max(np.abs(w - w2)) <= W_TOL


@pytest.mark.parametrize("config", ["tiny", "decode", "prefill4k"])
def test_route_topk(moe, config):
    c = wl.CONFIGS[config]
    H, E, k, T = c["H"], c["E"], c["k"], c["T"]
    w_r = wl.gen_router(0, E, H)
    bias = I_.bias_for(config)
    b64 = None if bias is None else bias.astype(np.float64)
    x, _ = I_.draw_x(0, T, H, w_r, k, bias=b64)
    ids_ref, w_ref, g_ref, lg_ref = oracle.router(x, w_r, k, bias=b64, want_logits=True)
    dummy = (torch.zeros(1, 1, 8, dtype=torch.uint8, device="cuda"),) * 2 + (torch.ones(1, 2, device="cuda"),)
    layer = moe.MoeLayer(H, E, k, 128, bf16_dev(w_r), dummy, dummy, torch.ones(E + 1, device="cuda"),
                         logit_bias=None if bias is None else dev(bias), prepacked=True)
    ids, w, g, lg = moe.moe_route_topk(bf16_dev(x), layer, want_logits=True)
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    _check_route_values(w, g, lg, w_ref, g_ref, lg_ref, ids=ids, k=k)


@pytest.mark.parametrize("config,T", [("tiny", 65), ("tiny", 130), ("decode", 300), ("decode", 2500), ("decode", 12365),
                                      ("wide_router", 20000)])
def test_route_topk_tensor_core_ragged(moe, config, T):
    # more than 64 tokens take the tensor-core router: token blocks of 128 and router-row tiles with
    # ragged edges (E + 1 = 17 and 513); the tile width follows the token count (64 rows while the
    # CTAs fit one wave, then 96 — 2500 tokens — then 176). From 12288 tokens with E = 512 the fused
    # router holds all 512 logits of a 128-token block per CTA (12365: a ragged last block of 77;
    # 20000: 157 CTAs, more than one per SM)
    c = wl.CONFIGS[config]
    H, E, k = c["H"], c["E"], c["k"]
    w_r = wl.gen_router(T, E, H)
    x, _ = I_.draw_x(T, T, H, w_r, k)
    ids_ref, w_ref, g_ref, lg_ref = oracle.router(x, w_r, k, want_logits=True)
    dummy = (torch.zeros(1, 1, 8, dtype=torch.uint8, device="cuda"),) * 2 + (torch.ones(1, 2, device="cuda"),)
    layer = moe.MoeLayer(H, E, k, 128, bf16_dev(w_r), dummy, dummy, torch.ones(E + 1, device="cuda"), prepacked=True)
    ids, w, g, lg = moe.moe_route_topk(bf16_dev(x), layer, want_logits=True)
    moe.moe_read_device_status()
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    _check_route_values(w, g, lg, w_ref, g_ref, lg_ref, ids=ids, k=k)


@pytest.mark.parametrize("interleave", [0, 1])
def test_prepack_layout(moe, interleave):
    # the documented prepacked layout, restated with numpy: K-slab-major codes (zero past K/2) with
    # the optional 64 gate + 64 up row interleave, and 512-byte scale tiles
    rng = np.random.default_rng(11 + interleave)
    G, N, K = 3, 256, 384
    codes = rng.integers(0, 256, (G, N, K // 2), dtype=np.uint8)
    sf = rng.integers(0, 256, (G, N, K // 16), dtype=np.uint8)
    cp, sp = moe.moe_prepack_nvfp4(dev(codes), dev(sf), bool(interleave))
    src = np.arange(N)
    if interleave:
        blk, w = src // 128, src % 128
        src = np.where(w < 64, blk * 64 + w, N // 2 + blk * 64 + (w - 64))
    slabs = (K + 255) // 256
    padded = np.zeros((G, N, slabs * 128), np.uint8)
    padded[:, :, :K // 2] = codes[:, src, :]
    want_codes = padded.reshape(G, N, slabs, 128).transpose(0, 2, 1, 3)
    np.testing.assert_array_equal(cp.cpu().numpy().reshape(G, slabs, N, 128), want_codes)
    want_sf = np.zeros((G, N // 128, K // 64, 512), np.uint8)
    rs = sf[:, src, :]
    for r in range(N):
        for kb in range(K // 64):
            t = want_sf[:, r // 128, kb]
            rr = r % 128
            t[:, (rr % 32) * 16 + (rr // 32) * 4:(rr % 32) * 16 + (rr // 32) * 4 + 4] = rs[:, r, kb * 4:kb * 4 + 4]
    np.testing.assert_array_equal(sp.cpu().numpy().reshape(G, N // 128, K // 64, 512), want_sf)


def test_route_exact_ties_lowest_index(moe):
    H, E, k, T = 256, 16, 4, 8
    rng = np.random.default_rng(3)
    w_r = wl.bf16_round(rng.standard_normal((E + 1, H)).astype(np.float32) * 0.05)
    w_r[7] = w_r[3]
    w_r[12] = w_r[3]
    bias = np.zeros(E, np.float32)
    bias[3] = bias[7] = bias[12] = 1e3  # the tied trio is always selected first
    x = wl.gen_x(4, T, H)
    ids_ref, _, _, _ = oracle.router(x, w_r, k, bias=bias.astype(np.float64))
    dummy = (torch.zeros(1, 1, 8, dtype=torch.uint8, device="cuda"),) * 2 + (torch.ones(1, 2, device="cuda"),)
    layer = moe.MoeLayer(H, E, k, 128, bf16_dev(w_r), dummy, dummy, torch.ones(E + 1, device="cuda"),
                         logit_bias=dev(bias), prepacked=True)
    ids, w, _, _ = moe.moe_route_topk(bf16_dev(x), layer)
    ids = ids.cpu().numpy()
    np.testing.assert_array_equal(ids, ids_ref)
    assert np.all(ids[:, :3] == [3, 7, 12])
    w = w.cpu().numpy()
    assert np.all(w[:, 0] == w[:, 1]) and np.all(w[:, 1] == w[:, 2])


def _tied_router(seed, E, H, n_tied):
    """Router whose n_tied rows (scattered ids) are one row with a large bias: those experts tie for
    every token, so the lowest ids among them must be selected, in id order."""
    rng = np.random.default_rng(seed)
    w_r = wl.gen_router(seed, E, H)
    tied = np.sort(rng.choice(E, size=n_tied, replace=False))
    w_r[tied] = w_r[tied[0]]
    bias = np.zeros(E, np.float32)
    bias[tied] = 100.0
    return w_r, bias, tied


@pytest.mark.parametrize("E,n_tied,T", [(512, 40, 4), (512, 70, 4), (512, 512, 9), (600, 40, 3), (600, 90, 70)])
def test_route_topk_tied_groups(moe, E, n_tied, T):
    # up to 64 candidates are ranked in shared memory; 70, 90 or 512 equal logits overflow the list
    # and take the round-by-round arg-max; E = 600 uses 19 keys per lane
    H, k = 256, 10
    w_r, bias, tied = _tied_router(E + n_tied, E, H, n_tied)
    if n_tied == E:
        w_r[:E] = 0.0
        bias[:] = 0.0
    x = wl.gen_x(7, T, H)
    ids_ref, w_ref, _, _ = oracle.router(x, w_r, k, bias=bias.astype(np.float64))
    np.testing.assert_array_equal(ids_ref, np.broadcast_to(tied[:k], (T, k)))
    dummy = (torch.zeros(1, 1, 8, dtype=torch.uint8, device="cuda"),) * 2 + (torch.ones(1, 2, device="cuda"),)
    layer = moe.MoeLayer(H, E, k, 128, bf16_dev(w_r), dummy, dummy, torch.ones(E + 1, device="cuda"),
                         logit_bias=dev(bias), prepacked=True)
    ids, w, _, _ = moe.moe_route_topk(bf16_dev(x), layer)
    moe.moe_read_device_status()
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    assert np.all(w.cpu().numpy() == np.float32(1.0 / k))


@pytest.mark.parametrize("n_tied", [40, 200, 512])
def test_route_topk_tied_groups_fused(moe, n_tied):
    # the fused router of 512 experts (from 12288 tokens; 12365: a ragged last block): 40 equal logits
    # fit a row's candidate list, 200 and 512 overflow it and the whole warp inserts from a second
    # pass over the accumulator; the lowest ids among the tied experts win, in id order
    E, H, k, T = 512, 256, 10, 12365
    w_r, bias, tied = _tied_router(E + n_tied, E, H, n_tied)
    if n_tied == E:
        w_r[:E] = 0.0
        bias[:] = 0.0
    x = wl.gen_x(8, T, H)
    ids_ref, _, _, _ = oracle.router(x, w_r, k, bias=bias.astype(np.float64))
    np.testing.assert_array_equal(ids_ref, np.broadcast_to(tied[:k], (T, k)))
    dummy = (torch.zeros(1, 1, 8, dtype=torch.uint8, device="cuda"),) * 2 + (torch.ones(1, 2, device="cuda"),)
    layer = moe.MoeLayer(H, E, k, 128, bf16_dev(w_r), dummy, dummy, torch.ones(E + 1, device="cuda"),
                         logit_bias=dev(bias), prepacked=True)
    ids, w, _, _ = moe.moe_route_topk(bf16_dev(x), layer)
    moe.moe_read_device_status()
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    assert np.all(w.cpu().numpy() == np.float32(1.0 / k))


@pytest.mark.parametrize("n_tied", [40, 70])
def test_layer_decode_tied_router(moe, n_tied):
    # the one-launch front half (T = 4) on tied logits: its own top-k must pick the same experts
    c = wl.CONFIGS["decode"]
    H, E, k, I, T = c["H"], c["E"], c["k"], c["I"], c["T"]
    w_r, bias, tied = _tied_router(n_tied, E, H, n_tied)
    x = wl.gen_x(11, T, H)
    gu, dn = I_.quantized_experts(n_tied, E, H, I, sorted(tied[:k].tolist()) + [E])
    case = dict(H=H, E=E, k=k, I=I, T=T, x=x, w_r=w_r, bias=bias, gu=gu, dn=dn,
                s_mid=np.full(E + 1, wl.s_mid_for("decode"), np.float32), rows=np.arange(T))
    _check_layer(moe, case)


# ------------------------------------------------------------------------------------------------
# permute
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("T,k,E,mode", [(64, 2, 16, "rand"), (4, 10, 512, "rand"), (1, 1, 1, "rand"),
                                        (1000, 3, 7, "one"), (16384, 10, 512, "hot"), (300, 8, 1024, "rand"),
                                        (0, 4, 16, "rand")])
def test_permute_bitexact(moe, T, k, E, mode):
    rng = np.random.default_rng(T + k + E)
    if mode == "one":
        ids = np.zeros((T, k), np.int32)
        ids[:] = np.arange(k) % E
        ids[:, 0] = 5
    elif mode == "hot":
        hot = rng.random((T, k)) < 0.5
        ids = np.where(hot, rng.integers(0, 51, (T, k)), rng.integers(51, E, (T, k))).astype(np.int32)
    else:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) if T else np.zeros((0, k), np.int32)
    off_ref, ps_ref, sp_ref = oracle.permute(ids, E) if T else (np.zeros(E + 2, np.int32), None, None)
    if T == 0:
        return  # nothing to launch; covered by the host tests
    off, ps, sp, rt = moe.moe_permute(dev(ids), E)
    np.testing.assert_array_equal(off.cpu().numpy(), off_ref)
    np.testing.assert_array_equal(ps.cpu().numpy(), ps_ref)
    np.testing.assert_array_equal(sp.cpu().numpy(), sp_ref)
    rt = rt.cpu().numpy()
    np.testing.assert_array_equal(rt[: T * k], ps_ref // k)
    np.testing.assert_array_equal(rt[T * k:], np.arange(T))


# ------------------------------------------------------------------------------------------------
# grouped GEMM
# ------------------------------------------------------------------------------------------------

def _gemm_case(seed, counts, H, I, N_kind):
    """Random activations + oracle-quantized weights for groups with the given row counts."""
    G = len(counts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    P = int(offsets[-1])
    rng = np.random.default_rng(seed)
    src_rows = max(P, 1) + 5
    K = H if N_kind == "gate_up" else I
    a = wl.bf16_round(rng.standard_normal((src_rows, K)).astype(np.float32))
    a_row = rng.integers(0, src_rows, P).astype(np.int32)
    ac, asf, sa = oracle.quantize_nvfp4(a)
    if N_kind == "gate_up":
        N = 2 * I
        bc = np.zeros((G, N, K // 2), np.uint8)
        bs = np.zeros((G, N, K // 16), np.uint8)
        bsc = np.zeros((G, 2), np.float32)
        for g in range(G):
            for h in range(2):
                w = rng.standard_normal((I, K)).astype(np.float32) * 0.02
                c, s, S = oracle.quantize_nvfp4(w)
                bc[g, h * I:(h + 1) * I], bs[g, h * I:(h + 1) * I], bsc[g, h] = c, s, S
    else:
        N = H
        bc = np.zeros((G, N, K // 2), np.uint8)
        bs = np.zeros((G, N, K // 16), np.uint8)
        bsc = np.zeros(G, np.float32)
        for g in range(G):
            c, s, S = oracle.quantize_nvfp4(rng.standard_normal((N, K)).astype(np.float32) * 0.02)
            bc[g], bs[g], bsc[g] = c, s, S
    return dict(offsets=offsets, P=P, ac=ac, asf=asf, sa=sa, a_row=a_row, bc=bc, bs=bs, bsc=bsc, N=N, K=K)


SCHEDS = ["act_on_m", "weights_on_m", "wide", "wide_rows", "weights_resident"]


def _sched(moe, name):
    return {"act_on_m": moe.SCHED_ACT_ON_M, "weights_on_m": moe.SCHED_WEIGHTS_ON_M, "wide": moe.SCHED_WIDE,
            "wide_rows": moe.SCHED_WIDE_ROWS, "weights_resident": moe.SCHED_WEIGHTS_RESIDENT}[name]


@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("counts", [[3, 0, 130, 1, 128, 257], [1] * 40, [700], [0, 0, 5], [33, 32, 31, 64, 65],
                                    [5, 4100, 0, 2049]])
def test_gemm_gate_up_f32(moe, counts, sched):
    # (4100 rows = 33 blocks of 128: a weight-resident schedule takes them in runs of at most 16)
    c = _gemm_case(len(counts), counts, 256, 128, "gate_up")
    ref = oracle.grouped_gemm(c["ac"], c["asf"], c["sa"], c["offsets"], c["bc"], c["bs"], c["bsc"], a_row=c["a_row"])
    bcp, bsp = moe.moe_prepack_nvfp4(dev(c["bc"]), dev(c["bs"]), True)
    out = moe.moe_grouped_gemm_nvfp4(dev(c["ac"]), dev(c["asf"]), dev(np.array([c["sa"]], np.float32)),
                                     dev(c["offsets"]), c["P"], bcp, bsp, dev(c["bsc"]), c["N"], c["K"], True,
                                     moe.EPI_F32, a_row_index=dev(c["a_row"]), schedule=_sched(moe, sched))
    out = out.cpu().numpy()
    assert I_.rel_frobenius(out, ref) <= GEMM_TOL
    for g in range(len(counts)):
        p0, p1 = c["offsets"][g], c["offsets"][g + 1]
        if p1 > p0:
            assert I_.rel_frobenius(out[p0:p1], ref[p0:p1]) <= GEMM_TOL, g


@pytest.mark.parametrize("sched", SCHEDS)
def test_gemm_gate_up_f32_flash_shape(moe, sched):
    c = _gemm_case(11, [2, 130, 1], 2048, 768, "gate_up")
    ref = oracle.grouped_gemm(c["ac"], c["asf"], c["sa"], c["offsets"], c["bc"], c["bs"], c["bsc"], a_row=c["a_row"])
    bcp, bsp = moe.moe_prepack_nvfp4(dev(c["bc"]), dev(c["bs"]), True)
    out = moe.moe_grouped_gemm_nvfp4(dev(c["ac"]), dev(c["asf"]), dev(np.array([c["sa"]], np.float32)),
                                     dev(c["offsets"]), c["P"], bcp, bsp, dev(c["bsc"]), c["N"], c["K"], True,
                                     moe.EPI_F32, a_row_index=dev(c["a_row"]),
                                     schedule=_sched(moe, sched)).cpu().numpy()
    assert I_.rel_frobenius(out, ref) <= GEMM_TOL
    for g in range(3):
        p0, p1 = c["offsets"][g], c["offsets"][g + 1]
        assert I_.rel_frobenius(out[p0:p1], ref[p0:p1]) <= GEMM_TOL


@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("H,I", [(256, 128), (2048, 768)])
def test_gemm_down_bf16(moe, H, I, sched):
    c = _gemm_case(5, [5, 129, 0, 2], H, I, "down")
    ref = oracle.grouped_gemm(c["ac"], c["asf"], c["sa"], c["offsets"], c["bc"], c["bs"], c["bsc"], a_row=c["a_row"])
    bcp, bsp = moe.moe_prepack_nvfp4(dev(c["bc"]), dev(c["bs"]), False)
    out = moe.moe_grouped_gemm_nvfp4(dev(c["ac"]), dev(c["asf"]), dev(np.array([c["sa"]], np.float32)),
                                     dev(c["offsets"]), c["P"], bcp, bsp, dev(c["bsc"]), c["N"], c["K"], False,
                                     moe.EPI_BF16, a_row_index=dev(c["a_row"]), schedule=_sched(moe, sched))
    out = out.float().cpu().numpy()
    # bf16 output: one rounding of each element (relative 2^-9)
    assert I_.rel_frobenius(out, ref) <= 4e-3


@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("H,I,counts", [(256, 128, [3, 0, 130, 1, 128]), (2048, 768, [1, 40, 3])])
def test_gemm_swiglu_requant(moe, H, I, counts, sched):
    c = _gemm_case(7, counts, H, I, "gate_up")
    G = len(counts)
    gu_ref = oracle.grouped_gemm(c["ac"], c["asf"], c["sa"], c["offsets"], c["bc"], c["bs"], c["bsc"], a_row=c["a_row"])
    h_ref = oracle.swiglu(gu_ref)
    s_mid = np.full(G, np.float32(np.abs(h_ref).max() / 2688.0 * 0.8), np.float32)  # some values saturate
    hc_ref, hs_ref = oracle.requantize_groups(h_ref, c["offsets"], s_mid)
    bcp, bsp = moe.moe_prepack_nvfp4(dev(c["bc"]), dev(c["bs"]), True)
    hc, hs = moe.moe_grouped_gemm_nvfp4(dev(c["ac"]), dev(c["asf"]), dev(np.array([c["sa"]], np.float32)),
                                        dev(c["offsets"]), c["P"], bcp, bsp, dev(c["bsc"]), c["N"], c["K"], True,
                                        moe.EPI_SWIGLU_NVFP4, a_row_index=dev(c["a_row"]), epi_scale=dev(s_mid),
                                        schedule=_sched(moe, sched))
    n_g, n_r = nibbles(hc.cpu().numpy()), nibbles(hc_ref)
    match = np.mean(n_g == n_r)
    assert match >= CODE_MATCH, match
    assert np.mean(hs.cpu().numpy() == hs_ref) >= CODE_MATCH


# ------------------------------------------------------------------------------------------------
# combine and the whole layer
# ------------------------------------------------------------------------------------------------

def test_combine(moe):
    rng = np.random.default_rng(8)
    T, k, H = 37, 3, 256
    P = T * k + T
    y = wl.bf16_round(rng.standard_normal((P, H)).astype(np.float32))
    tw = rng.random((T, k)).astype(np.float32)
    g = rng.random(T).astype(np.float32)
    src_perm = rng.permutation(T * k).astype(np.int32)
    res = wl.bf16_round(rng.standard_normal((T, H)).astype(np.float32))
    o64, o16 = oracle.combine(y.astype(np.float64), tw.astype(np.float64), src_perm, shared_g=g.astype(np.float64),
                              shared_row0=T * k, residual=res)
    out = moe.moe_combine(bf16_dev(y), dev(tw), dev(src_perm), shared_g=dev(g), residual=bf16_dev(res))
    out = out.float().cpu().numpy()
    assert np.max(np.abs(out - o64) / (np.abs(o64) + 1e-3)) <= 2 ** -8


def _check_layer(moe, case, residual=False):
    layer = gpu_layer(moe, case)
    x = case["x"]
    res = wl.bf16_round(np.random.default_rng(1).standard_normal(x.shape).astype(np.float32)) if residual else None
    out = moe.moe_layer_forward(layer, bf16_dev(x), residual=None if res is None else bf16_dev(res))
    moe.moe_read_device_status()
    out = out.float().cpu().numpy()
    rows = case["rows"]
    b64 = None if case["bias"] is None else case["bias"].astype(np.float64)
    Sx = oracle.tensor_scale(x)
    ref = oracle.layer_forward(x[rows], case["w_r"], case["k"], case["gu"], case["dn"], case["s_mid"], bias=b64,
                               residual=None if res is None else res[rows], x_scale=Sx)
    err = I_.rel_frobenius(out[rows], ref["out_f64"])
    assert err <= LAYER_TOL, err
    return err


def test_layer_tiny(moe):
    case = I_.layer_case("tiny")
    err = _check_layer(moe, case)
    assert err < 5e-3  # requantized codes agree, so the error is the bf16 rounding of y and out


@pytest.mark.parametrize("T", [None, 3, 1500])
def test_layer_tiny_residual(moe, T):
    # 64 tokens: separate front kernels, 3 tokens: the one-launch front half, 1500 tokens: the
    # streaming combine (one CTA per SM, rows bulk-copied into shared memory)
    _check_layer(moe, I_.layer_case("tiny", seed=0 if T is None else 21, T=T), residual=True)


def test_layer_decode_full_size(moe):
    _check_layer(moe, I_.layer_case("decode"))


def test_layer_prefill4k_sampled(moe):
    _check_layer(moe, I_.layer_case("prefill4k", sample=12))


def test_layer_prefill16k_sampled(moe):
    # 16k tokens with a hot expert set: the expert GEMMs take whole token blocks per CTA here
    _check_layer(moe, I_.layer_case("prefill16k", sample=8))


@pytest.mark.parametrize("T", [1, 4, 5, 7, 8, 9, 63, 64, 65, 130, 1023, 1024])
def test_layer_tiny_token_counts(moe, T):
    # T <= 64 with T*k <= 512 takes the one-launch front half, larger T the separate kernels; the
    # front half stages 4 tokens per router pass up to T = 4 and 8 beyond, so 4/5, 7/8/9 and
    # 63/64/65 straddle its edges
    _check_layer(moe, I_.layer_case("tiny", seed=T, T=T))


@pytest.mark.parametrize("T", [51, 52])
def test_layer_decode_shape_front_edge(moe, T):
    # T*k = 510 is the largest assignment count of the one-launch front half at k = 10; 520 is not
    _check_layer(moe, I_.layer_case("decode", seed=3, sample=6, T=T))


def test_layer_repeat_bit_identical(moe):
    # the front half's completion counter must be back at zero after every call
    case = I_.layer_case("decode", seed=5, sample=4)
    layer = gpu_layer(moe, case)
    x = bf16_dev(case["x"])
    ws = moe.Workspace(moe.moe_workspace_bytes(case["H"], case["E"], case["k"], case["I"], case["T"]))
    outs = [moe.moe_layer_forward(layer, x, ws=ws).clone() for _ in range(4)]
    moe.moe_read_device_status(ws=ws)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("name,residual", [("decode", False), ("tiny", True)])
def test_layer_host_buffers_match_device_call(moe, name, residual):
    # moe_layer_forward_host (host tensors in and out, copies enqueued by the library) gives the
    # same bits as moe_layer_forward on device copies of the same tensors
    case = I_.layer_case(name, seed=9, sample=4) if name == "decode" else I_.layer_case(name, seed=9)
    layer = gpu_layer(moe, case)
    x = bf16_dev(case["x"])
    res = bf16_dev(case["x"][::-1].copy()) if residual else None
    ref = moe.moe_layer_forward(layer, x, residual=res)
    x_h = x.cpu().pin_memory()
    res_h = res.cpu().pin_memory() if residual else None
    out_h = moe.moe_layer_forward_host(layer, x_h, residual=res_h)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(out_h.view(torch.int16), ref.cpu().view(torch.int16))
    # pageable host memory works too
    out_p = moe.moe_layer_forward_host(layer, x.cpu(), residual=res.cpu() if residual else None,
                                       out=torch.empty(out_h.shape, dtype=torch.bfloat16))
    torch.cuda.current_stream().synchronize()
    assert torch.equal(out_p.view(torch.int16), ref.cpu().view(torch.int16))


def test_layer_host_rejects_device_pointers(moe):
    case = I_.layer_case("tiny", seed=2)
    layer = gpu_layer(moe, case)
    x = bf16_dev(case["x"])
    ws = moe.Workspace(moe.moe_workspace_bytes_host(case["H"], case["E"], case["k"], case["I"], case["T"]))
    out_h = torch.empty(case["T"], case["H"], dtype=torch.bfloat16)
    L = moe.lib()
    st = L.moe_layer_forward_host(ctypes.byref(layer.desc), ctypes.c_void_p(x.data_ptr()), case["T"], None,
                                  ctypes.c_void_p(out_h.data_ptr()), ws.ptr, ws.nbytes, moe._stream())
    assert st != 0 and "device memory" in L.moe_last_error_detail().decode()


@pytest.mark.parametrize("T,k,E", [(3, 2, 8), (300, 4, 16)])
def test_permute_reports_bad_expert_ids(moe, T, k, E):
    # an id outside [0, E) is dropped on the device and reported through the workspace's status word
    # (the path a bounded wait that ran out takes as well); the valid ids are still placed stably
    rng = np.random.default_rng(T)
    ids = rng.integers(0, E, (T, k)).astype(np.int32)
    ids[0, 0] = E + 5
    ids[-1, -1] = -2
    ws = moe.Workspace(moe.moe_workspace_bytes(128, E, k, 128, T))
    off, ps, sp, rt = moe.moe_permute(dev(ids), E, ws=ws)
    with pytest.raises(moe.MoeError, match="outside"):
        moe.moe_read_device_status(ws=ws)
    moe.moe_read_device_status(ws=ws)  # reading it cleared it
    valid = ids[(ids >= 0) & (ids < E)]
    want = np.concatenate([[0], np.cumsum(np.bincount(valid, minlength=E))])
    np.testing.assert_array_equal(off.cpu().numpy()[: E + 1], want)


def test_device_status_clean(moe):
    moe.moe_read_device_status()


@pytest.mark.parametrize("name,T", [("tiny", 4), ("tiny", 64), ("tiny", 65), ("tiny", 300), ("decode", 300),
                                    ("prefill4k", 4096), ("prefill16k", 16384)])
def test_layer_launch_count(moe, name, T):
    # the kernels one layer call launches, as the CUDA activity trace lists them, against the count the
    # benchmark reports: 3 for small batches (front half, expert GEMMs, combine), up to 9 otherwise (7
    # with the fused router of 512 experts from 12288 tokens)
    from torch.autograd import DeviceType
    from torch.profiler import ProfilerActivity, profile

    import bench

    case = I_.layer_case(name, seed=4, sample=2, T=T)
    layer = gpu_layer(moe, case)
    x = bf16_dev(case["x"])
    ws = moe.Workspace(moe.moe_workspace_bytes(case["H"], case["E"], case["k"], case["I"], T))
    moe.moe_layer_forward(layer, x, ws=ws)  # first call: kernel attributes set outside the trace
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]):  # a process's first trace can come back empty
        torch.ones(1, device="cuda").add_(1)
        torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as p:
        moe.moe_layer_forward(layer, x, ws=ws)
        torch.cuda.synchronize()
    moe.moe_read_device_status(ws=ws)
    names = [e.name for e in p.events() if e.device_type == DeviceType.CUDA and "Mem" not in e.name]
    if not names:
        pytest.skip("the profiler recorded no device activity here")
    assert all("moe::" in n for n in names), names
    want = bench.launches_per_layer(dict(T=T, H=case["H"], k=case["k"], E=case["E"]))
    assert len(names) == want, names
