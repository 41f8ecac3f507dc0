"""The layer's own intermediate results against the oracle, step by step, on the path the benchmark
times: after moe_layer_forward the tests read the workspace at the offsets moe_layer_workspace_view
reports (views only; no arithmetic on the GPU's side of the comparison).

Bars:
  bit-exact  S_x, the codes and block scales of x, the expert ids in routing order, and (where the
             layer stores them) the expert offsets and the permutation indices;
  1e-4       the router logits (FP32 sums in another order than the oracle's FP64 ones);
  1e-6       the routing weights, their sum and the shared gate, against the oracle's FP64
             softmax / renormalisation / sigmoid of the layer's OWN FP32 logits (this pins the
             routing arithmetic itself, apart from the logits' summation order); the ids selected
             from those logits must equal the layer's too;
  >= 99.9 %  the requantised intermediate h (codes and block scales), row by row in permuted order:
             for small batches the expert GEMMs build the permutation in shared memory, so h at
             the oracle's permuted positions also checks that permutation;
  per row    y, the down projection of every assignment (t, j) in assignment order, against the
             oracle's row for expert ids[t][j]: within 1e-2 where the assignment's h row (codes and
             scales) equals the oracle's, within 0.25 where one of its h codes differs (the
             requantisation may differ in 0.1 % of codes; with I = 128 one differing code moves a row
             by a few percent), and within 1e-2 over all rows. A row computed in the wrong expert
             group is off by about 1.4.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from tests import inputs as I_
from tests.test_gpu_parity import bf16_dev, gpu_layer, nibbles

pytestmark = pytest.mark.gpu

# MOE_NVFP4_GEMM_PERMUTE=0 moves the small-batch permutation back into the front half (stored)
GEMM_PERMUTES = os.environ.get("MOE_NVFP4_GEMM_PERMUTE", "1")[:1] != "0"
LOGIT_TOL = 1e-4
W_TOL = 1e-6
CODE_MATCH = 0.999
Y_ROW_TOL = 1e-2      # rows whose h equals the oracle's
Y_ROW_TOL_H = 0.25    # rows with a differing h code
Y_TOL = 1e-2


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_w4a4_mixture_gb300 as m
    from nvfp4_w4a4_mixture_gb300 import build

    build.build()
    m.lib()
    return m


def _run(moe, case):
    layer = gpu_layer(moe, case)
    T = case["T"]
    ws = moe.Workspace(layer.workspace_bytes(T))
    out = moe.moe_layer_forward(layer, bf16_dev(case["x"]), ws=ws)
    torch.cuda.synchronize()
    moe.moe_read_device_status(ws=ws)
    got = moe.layer_intermediates(layer, T, ws)
    got = {k: (v.float().cpu().numpy() if torch.is_tensor(v) and v.dtype == torch.bfloat16
               else v.cpu().numpy() if torch.is_tensor(v) else v) for k, v in got.items()}
    got["out"] = out.float().cpu().numpy()
    return got


def _scale_tile_bytes(h_sf_tiles, offsets, block_rows, positions, n_cols):
    """Block scales of h at permuted rows `positions`, read out of the token-block tiles: the rows of
    group g are cut into blocks of block_rows, numbered across the groups in order."""
    cnt = np.diff(offsets.astype(np.int64))
    tb_off = np.concatenate([[0], np.cumsum((cnt + block_rows - 1) // block_rows)])
    out = np.zeros((len(positions), n_cols), np.uint8)
    for i, p in enumerate(positions):
        g = int(np.searchsorted(offsets, p, side="right")) - 1
        q = p - int(offsets[g])
        blk, r = int(tb_off[g]) + q // block_rows, q % block_rows
        for c in range(n_cols):
            out[i, c] = h_sf_tiles[blk, c // 4, (r % 32) * 16 + (r // 32) * 4 + c % 4]
    return out


def _check_front(got, case, ref_ids, ref_logits, ref_codes, ref_sf, ref_S):
    """S_x, x codes and scales, ids, logits; weights and gate against the oracle's routing of the
    layer's own logits."""
    E, k = case["E"], case["k"]
    assert np.float32(got["x_scale"][0]) == np.float32(ref_S)
    np.testing.assert_array_equal(got["x_codes"], ref_codes)
    np.testing.assert_array_equal(got["x_sf"], ref_sf)
    np.testing.assert_array_equal(got["topk_ids"], ref_ids)
    lg = got["logits"]
    assert np.max(np.abs(lg[:, :E] - ref_logits)) <= LOGIT_TOL
    ids2, w2, g2 = oracle.route_from_logits(lg[:, :E].astype(np.float64), k, gate_logit=lg[:, E].astype(np.float64))
    np.testing.assert_array_equal(ids2, got["topk_ids"])
    assert np.max(np.abs(got["topk_w"] - w2)) <= W_TOL
    assert np.max(np.abs(got["topk_w"].astype(np.float64).sum(1) - 1.0)) <= W_TOL
    assert np.max(np.abs(got["shared_g"] - g2)) <= W_TOL


def _check_rows(got, ref, gpu_pos, ref_pos, gpu_assign, ref_assign, offsets, I):
    """Entry i of the four index arrays is one assignment: its h row (permuted positions, the GPU's
    and the oracle's) and its y row (the GPU's in assignment order, the oracle's)."""
    hc = nibbles(got["h_codes"][gpu_pos])
    hc_ref = nibbles(ref["h_codes"][ref_pos])
    match = float(np.mean(hc == hc_ref))
    assert match >= CODE_MATCH, match
    hs = _scale_tile_bytes(got["h_sf"], offsets, got["h_block_rows"], gpu_pos, I // 16)
    hs_ref = ref["h_sf"][ref_pos]
    smatch = float(np.mean(hs == hs_ref))
    assert smatch >= CODE_MATCH, smatch
    h_same = np.all(hc == hc_ref, axis=1) & np.all(hs == hs_ref, axis=1)
    y = got["y"][gpu_assign].astype(np.float64)
    y_ref = ref["y"][ref_assign]
    row_err = np.linalg.norm(y - y_ref, axis=1) / np.maximum(np.linalg.norm(y_ref, axis=1), 1e-30)
    if np.any(h_same):
        e = row_err[h_same]
        assert np.max(e) <= Y_ROW_TOL, (int(np.flatnonzero(h_same)[np.argmax(e)]), float(np.max(e)))
    assert np.max(row_err) <= Y_ROW_TOL_H, (int(np.argmax(row_err)), float(np.max(row_err)))
    assert I_.rel_frobenius(y, y_ref) <= Y_TOL


def _check_full(moe, case):
    """Every token's intermediates (all routed experts carry real weights)."""
    got = _run(moe, case)
    T, E, k, I = case["T"], case["E"], case["k"], case["I"]
    b64 = None if case["bias"] is None else case["bias"].astype(np.float64)
    ref = oracle.layer_forward(case["x"], case["w_r"], k, case["gu"], case["dn"], case["s_mid"], bias=b64)
    assert I_.rel_frobenius(got["out"], ref["out_f64"]) <= 2e-2
    _check_front(got, case, ref["topk_ids"], ref["logits"], ref["x_codes"], ref["x_sf"], ref["x_scale"])
    if got["permutation_in_workspace"]:
        np.testing.assert_array_equal(got["expert_offsets"], ref["offsets"])
        np.testing.assert_array_equal(got["perm_src"], ref["perm_src"])
        np.testing.assert_array_equal(got["src_perm"], ref["src_perm"])
        np.testing.assert_array_equal(got["row_token"], ref["row_token"])
    P = T * k + T
    # assignment a: h at permuted position src_perm[a] (the shared rows at T*k + t in both orders),
    # y at row a on the GPU (assignment order) and at that permuted position in the oracle's y
    pos = np.concatenate([ref["src_perm"], np.arange(T * k, P)])
    _check_rows(got, ref, pos, pos, np.arange(P), pos, ref["offsets"], I)
    return got


@pytest.mark.parametrize("T", [1, 4, 5, 64, 65, 1100])
def test_layer_intermediates_tiny(moe, T):
    # T <= 32: one-launch front half + the expert GEMMs' own permutation (wide-narrow tiles);
    # T = 64: one-launch front half with the permutation stored (wide tiles); T = 65: separate
    # quantize / tensor-core router / top-k / permute launches; T = 1100: the CTA-chunk permutation
    # over several chunks and the streaming combine
    got = _check_full(moe, I_.layer_case("tiny", seed=T, T=T))
    assert got["permutation_in_workspace"] == (T > 32 or not GEMM_PERMUTES)
    assert not got["route_first"]


def test_layer_intermediates_fused_router(moe):
    # 512 experts and 12,365 tokens (H 256, I 128): the fused router first (logits, top-k, weights,
    # shared gate and x's maximum), then the encoder, the permutation, the expert GEMMs and the
    # combine; every token against the oracle, the last 128-token block ragged (77 tokens)
    got = _check_full(moe, I_.layer_case("wide_router"))
    assert got["route_first"] and got["permutation_in_workspace"]


@pytest.mark.parametrize("config", ["max_hidden", "max_inter", "max_experts_k"])
def test_layer_intermediates_shape_limits(moe, config):
    # the largest supported shapes on small batches (70 tokens, the separate front launches): H = 8192
    # (router and gate/up K = 8192), I = 8192 (gate/up N = 16384, down K = 8192), E = 1024 with k = 32
    got = _check_full(moe, I_.layer_case(config))
    assert got["permutation_in_workspace"] and not got["route_first"]


def test_layer_intermediates_decode(moe):
    # the benchmarked decode step: k_decode_front (quantise, logits, top-k), then the expert GEMMs
    # whose every CTA ranks the ids in shared memory
    got = _check_full(moe, I_.layer_case("decode"))
    assert got["permutation_in_workspace"] == (not GEMM_PERMUTES) and got["h_block_rows"] == 32


@pytest.mark.parametrize("n_tied", [40])
def test_layer_intermediates_decode_tied_router(moe, n_tied):
    from tests.test_gpu_parity import _tied_router
    from nvfp4_w4a4_mixture_gb300 import workloads as wl

    c = wl.CONFIGS["decode"]
    H, E, k, I, T = c["H"], c["E"], c["k"], c["I"], c["T"]
    w_r, bias, tied = _tied_router(n_tied, E, H, n_tied)
    gu, dn = I_.quantized_experts(n_tied, E, H, I, sorted(tied[:k].tolist()) + [E])
    case = dict(H=H, E=E, k=k, I=I, T=T, x=wl.gen_x(11, T, H), w_r=w_r, bias=bias, gu=gu, dn=dn,
                s_mid=np.full(E + 1, wl.s_mid_for("decode"), np.float32), rows=np.arange(T))
    got = _check_full(moe, case)
    np.testing.assert_array_equal(got["topk_ids"], np.broadcast_to(tied[:k], (T, k)))


@pytest.mark.parametrize("config,sample", [("prefill4k", 6), ("prefill16k", 8)])
def test_layer_intermediates_prefill_sampled(moe, config, sample):
    # every token's routing and x codes, the whole permutation; h and y on the sampled tokens'
    # rows (only their experts carry real weights): 16k tokens take whole token blocks per CTA
    case = I_.layer_case(config, sample=sample)
    got = _run(moe, case)
    T, E, k, I = case["T"], case["E"], case["k"], case["I"]
    x = case["x"]
    b64 = case["bias"].astype(np.float64)
    ids, _, _, lg = oracle.router(x, case["w_r"], k, bias=b64, want_logits=True)
    codes, sf, S = oracle.quantize_nvfp4(x)
    _check_front(got, case, ids, lg, codes, sf, S)
    assert got["permutation_in_workspace"]
    assert got["route_first"] == (T >= 12288)  # 512 experts: the fused router, then the encoder
    off, ps, sp = oracle.permute(ids, E)
    np.testing.assert_array_equal(got["expert_offsets"], off)
    np.testing.assert_array_equal(got["perm_src"], ps)
    np.testing.assert_array_equal(got["src_perm"], sp)
    np.testing.assert_array_equal(got["row_token"], np.concatenate([ps // k, np.arange(T)]))
    rows = case["rows"]
    Ts = len(rows)
    ref = oracle.layer_forward(x[rows], case["w_r"], k, case["gu"], case["dn"], case["s_mid"], bias=b64, x_scale=S)
    # the sampled tokens' assignments (t, j) and shared rows, on both sides
    f_full = (rows[:, None] * k + np.arange(k)).ravel()
    f_smp = np.arange(Ts * k)
    gpu_pos = np.concatenate([sp[f_full], T * k + rows])
    ref_pos = np.concatenate([ref["src_perm"][f_smp], Ts * k + np.arange(Ts)])
    gpu_assign = np.concatenate([f_full, T * k + rows])
    _check_rows(got, ref, gpu_pos, ref_pos, gpu_assign, ref_pos, off, I)
