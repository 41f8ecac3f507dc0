// router.cu -- router logits (x W_r^T, bf16 inputs, FP32 accumulation) and the FP32 softmax top-k.
//
// Logits: one warp per router row, a tile of kRouterTT tokens staged in shared memory, 16-byte
// loads of the router row (each row of W_r is read once per token tile). Every product of two
// bf16 values is exact in FP32; the sum runs in a fixed order (per-lane strided partial sums,
// then a butterfly), so the result is deterministic.
// Top-k: one CTA of 4 warps per token; k rounds of a block arg-max on (logit desc, expert id
// asc), which is the lowest-index tie rule; the renormalised weights are the softmax over the
// selected logits (the full softmax denominator cancels), the shared gate is sigmoid(logit E).
#include <cfloat>

#include "kernels.cuh"

namespace moe {

constexpr int kRouterTT = 8;     // tokens per CTA
constexpr int kRouterWarps = 8;  // router rows per CTA

__global__ void __launch_bounds__(kRouterWarps * 32)
    k_router_logits(const uint16_t* __restrict__ x, int T, int H, int E, const uint16_t* __restrict__ w,
                    const float* __restrict__ bias, float* __restrict__ logits)
{
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
                    acc[t] = __fadd_rn(acc[t], __fmul_rn(bf16_to_f32(xx[i] & 0xFFFFu), bf16_to_f32(ww[i] & 0xFFFFu)));
                    acc[t] = __fadd_rn(acc[t], __fmul_rn(bf16_to_f32(xx[i] >> 16), bf16_to_f32(ww[i] >> 16)));
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

constexpr int kTopkThreads = 128;
constexpr int kTopkPer = 8;  // E <= 1024 = kTopkThreads * kTopkPer

// (value desc, index asc) order: true when (a, ia) comes before (b, ib)
__device__ __forceinline__ bool before(float a, int ia, float b, int ib) { return a > b || (a == b && ia < ib); }

// One CTA (4 warps) per token: each thread holds 8 logits; k rounds of a block arg-max.
__global__ void __launch_bounds__(kTopkThreads)
    k_topk(const float* __restrict__ logits, int ld, int T, int E, int k, int32_t* __restrict__ topk_ids,
           float* __restrict__ topk_w, float* __restrict__ shared_g, float* __restrict__ logits_out)
{
    __shared__ float wb[kTopkThreads / 32];
    __shared__ int wi[kTopkThreads / 32];
    __shared__ float sel_l[32];
    __shared__ int sel_i[32];
    const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* l = logits + static_cast<int64_t>(t) * ld;
    float v[kTopkPer];
    unsigned live = 0;
#pragma unroll
    for (int i = 0; i < kTopkPer; ++i) {
        const int e = i * kTopkThreads + tid;
        v[i] = e < E ? l[e] : 0.0f;
        if (e < E) {
            live |= 1u << i;
            if (logits_out) logits_out[static_cast<int64_t>(t) * E + e] = v[i];
            if (v[i] != v[i]) v[i] = -INFINITY;  // a NaN logit ranks below every number
        }
    }
    for (int j = 0; j < k; ++j) {
        float b = -INFINITY;  // (-inf, INT_MAX) loses to every live logit
        int bi = 0x7FFFFFFF;
#pragma unroll
        for (int i = 0; i < kTopkPer; ++i) {
            const int e = i * kTopkThreads + tid;
            if (((live >> i) & 1u) && before(v[i], e, b, bi)) {
                b = v[i];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ob = __shfl_xor_sync(0xFFFFFFFFu, b, o);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
            if (before(ob, oi, b, bi)) {
                b = ob;
                bi = oi;
            }
        }
        if (lane == 0) {
            wb[warp] = b;
            wi[warp] = bi;
        }
        __syncthreads();
        b = wb[0];
        bi = wi[0];
#pragma unroll
        for (int w = 1; w < kTopkThreads / 32; ++w)
            if (before(wb[w], wi[w], b, bi)) {
                b = wb[w];
                bi = wi[w];
            }
        if (tid == 0) {
            sel_l[j] = b;
            sel_i[j] = bi;
        }
#pragma unroll
        for (int i = 0; i < kTopkPer; ++i)
            if (i * kTopkThreads + tid == bi) live &= ~(1u << i);
        __syncthreads();
    }
    // renormalised weights: softmax over the selected logits (the first one is the largest)
    if (warp == 0) {
        const float p = lane < k ? expf(sel_l[lane] - sel_l[0]) : 0.0f;
        float sum = p;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        if (lane < k) {
            topk_ids[static_cast<int64_t>(t) * k + lane] = sel_i[lane];
            topk_w[static_cast<int64_t>(t) * k + lane] = p / sum;
        }
        if (shared_g && lane == 0) shared_g[t] = 1.0f / (1.0f + expf(-l[E]));
    }
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
    k_router_logits<<<grid, kRouterWarps * 32, smem, stream>>>(x, T, H, E, w_router, bias, logits);
    return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, int ld, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                        float* shared_g, float* logits_out, cudaStream_t stream)
{
    if (T <= 0) return cudaSuccess;
    k_topk<<<T, kTopkThreads, 0, stream>>>(logits, ld, T, E, k, topk_ids, topk_w, shared_g, logits_out);
    return cudaGetLastError();
}

}  // namespace moe
