// router.cu -- router logits (x W_r^T, bf16 inputs, FP32 accumulation) and the FP32 softmax top-k.
//
// Logits: one warp per router row, a tile of kRouterTT tokens staged in shared memory, 16-byte
// loads of the router row (each row of W_r is read once per token tile). Every product of two
// bf16 values is exact in FP32, so a fused multiply-add rounds only the sum; the sum runs in a
// fixed order (per-lane strided partial sums, then a butterfly), so the result is deterministic.
// Top-k: one warp per token (see topk.cuh): the candidates at or above the k-th largest lane
// maximum ranked on (logit desc, expert id asc), which is the lowest-index tie rule, with k rounds
// of a warp arg-max when too many logits tie for the candidate list; the renormalised weights are
// the softmax over the selected logits (the full softmax denominator cancels), the shared gate is
// sigmoid(logit E).
#include <cfloat>

#include "kernels.cuh"
#include "topk.cuh"

namespace moe {

constexpr int kRouterTT = 8;     // tokens per CTA
constexpr int kRouterWarps = 8;  // router rows per CTA

__global__ void __launch_bounds__(kRouterWarps * 32)
    k_router_logits(const uint16_t* __restrict__ x, int T, int H, int E, const uint16_t* __restrict__ w,
                    const float* __restrict__ bias, float* __restrict__ logits)
{
    ptx::griddep_wait();  // x may come from the launch before this one
    extern __shared__ __align__(16) uint16_t xs[];  // [kRouterTT][H]
    const int t0 = blockIdx.y * kRouterTT;
    const int nt = min(kRouterTT, T - t0);
    // stage the token tile (16-byte vectors)
    const int vec_per_row = H / 8;
    for (int i = threadIdx.x; i < kRouterTT * vec_per_row; i += blockDim.x) {
        const int t = i / vec_per_row, c = i % vec_per_row;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (t < nt) v = __ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t0 + t) * H) + c);
        reinterpret_cast<uint4*>(xs + t * H)[c] = v;
    }
    __syncthreads();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int e = blockIdx.x * kRouterWarps + warp;
    if (e > E) return;
    float acc[kRouterTT];
#pragma unroll
    for (int t = 0; t < kRouterTT; ++t) acc[t] = 0.0f;
    const uint16_t* wr = w + static_cast<int64_t>(e) * H;
    // the row's 16-byte vectors are loaded 8 at a time so their latencies overlap
    for (int base = 0; base < H; base += 8 * 256) {
        uint4 wv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int h0 = base + u * 256 + lane * 8;
            wv[u] = h0 < H ? __ldg(reinterpret_cast<const uint4*>(wr + h0)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int h0 = base + u * 256 + lane * 8;
            if (h0 >= H) break;
            const uint32_t ww[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
#pragma unroll
            for (int t = 0; t < kRouterTT; ++t) {
                const uint4 xv = *reinterpret_cast<const uint4*>(xs + t * H + h0);
                const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[t] = __fmaf_rn(bf16_to_f32(xx[i] & 0xFFFFu), bf16_to_f32(ww[i] & 0xFFFFu), acc[t]);
                    acc[t] = __fmaf_rn(bf16_to_f32(xx[i] >> 16), bf16_to_f32(ww[i] >> 16), acc[t]);
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kRouterTT; ++t) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[t] = __fadd_rn(acc[t], __shfl_xor_sync(0xFFFFFFFFu, acc[t], o));
    }
    if (lane < nt) {
        float v = 0.0f;
#pragma unroll
        for (int t = 0; t < kRouterTT; ++t)
            if (t == lane) v = acc[t];
        if (bias && e < E) v = __fadd_rn(v, bias[e]);
        logits[static_cast<int64_t>(t0 + lane) * (E + 1) + e] = v;
    }
}


// One warp per token (8 per CTA): the warp top-k, renormalised weights, shared gate.
constexpr int kTopkWarps = 8;

__global__ void __launch_bounds__(kTopkWarps * 32)
    k_topk(const float* __restrict__ logits, int ld, int T, int E, int k, int32_t* __restrict__ topk_ids,
           float* __restrict__ topk_w, float* __restrict__ shared_g, float* __restrict__ logits_out)
{
    ptx::griddep_wait();  // the logits come from the launch before this one
    __shared__ uint2 cand_s[kTopkWarps][kTopkCand];
    __shared__ uint2 sel_s[kTopkWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x * kTopkWarps + warp;
    if (t >= T) return;
    const float* l = logits + static_cast<int64_t>(t) * ld;
    const float l_gate = lane == 0 ? __ldcg(l + E) : 0.0f;
    float sel_l, l0;
    int sel_i;
    const bool done = E <= 512 ? warp_topk_threshold<16>(l, E, k, cand_s[warp], sel_s[warp], sel_l, sel_i, l0)
                               : warp_topk_threshold<32>(l, E, k, cand_s[warp], sel_s[warp], sel_l, sel_i, l0);
    if (!done) warp_topk(l, E, k, sel_l, sel_i, l0);
    const float w = warp_topk_weight(sel_l, l0, k);
    if (lane < k) {
        topk_ids[static_cast<int64_t>(t) * k + lane] = sel_i;
        topk_w[static_cast<int64_t>(t) * k + lane] = w;
    }
    if (shared_g && lane == 0) shared_g[t] = 1.0f / (1.0f + expf(-l_gate));
    if (logits_out)
        for (int e = lane; e < E; e += 32) logits_out[static_cast<int64_t>(t) * E + e] = __ldcg(l + e);
}

cudaError_t launch_router_logits(const uint16_t* x, int T, int H, int E, const uint16_t* w_router, const float* bias,
                                 float* logits, cudaStream_t stream)
{
    if (T <= 0) return cudaSuccess;
    const size_t smem = static_cast<size_t>(kRouterTT) * H * sizeof(uint16_t);
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(k_router_logits, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        attr_set = true;
    }
    dim3 grid((E + 1 + kRouterWarps - 1) / kRouterWarps, (T + kRouterTT - 1) / kRouterTT);
    return launch_pdl(k_router_logits, grid, dim3(kRouterWarps * 32), smem, stream, x, T, H, E, w_router, bias, logits);
}

cudaError_t launch_topk(const float* logits, int ld, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                        float* shared_g, float* logits_out, cudaStream_t stream)
{
    if (T <= 0) return cudaSuccess;
    return launch_pdl(k_topk, dim3((T + kTopkWarps - 1) / kTopkWarps), dim3(kTopkWarps * 32), 0, stream, logits, ld, T, E, k,
                      topk_ids, topk_w, shared_g, logits_out);
}

}  // namespace moe
