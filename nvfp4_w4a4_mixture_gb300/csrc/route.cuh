// route.cuh -- block-level pieces of the small-batch routing front half (the one-launch front
// kernel): router-row logits, x quantisation, the small stable permutation.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace moe {

// Router logits of one router row for kTT staged tokens, by one warp: xs = kTT rows of H bf16 in
// shared memory, wr = the router row, w0 = its first 2048 columns already loaded (lane l holds
// columns u*256 + 8l .. +7 of each 2048-column chunk). Per-lane strided FP32 sums in a fixed order,
// then a butterfly: every caller gets bit-identical logits. A product of two bf16 values is exact in
// FP32 (8 + 8 significand bits), so each fused multiply-add rounds once, like an add of the product.
template <int kTT>
__device__ __forceinline__ void router_row_logits(const uint16_t* xs, int H, const uint16_t* wr, const uint4 (&w0)[8],
                                                  float (&acc)[kTT])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int t = 0; t < kTT; ++t) acc[t] = 0.0f;
    for (int base = 0; base < H; base += 8 * 256) {
        uint4 wv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int h0 = base + u * 256 + lane * 8;
            wv[u] = base == 0 ? w0[u] : (h0 < H ? __ldg(reinterpret_cast<const uint4*>(wr + h0)) : make_uint4(0, 0, 0, 0));
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int h0 = base + u * 256 + lane * 8;
            if (h0 >= H) break;
            const uint32_t ww[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
#pragma unroll
            for (int t = 0; t < kTT; ++t) {
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
    for (int t = 0; t < kTT; ++t) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[t] = __fadd_rn(acc[t], __shfl_xor_sync(0xFFFFFFFFu, acc[t], o));
    }
}

// The first 2048 columns of router row wr as router_row_logits expects them (zeros past H or when
// the warp has no row).
__device__ __forceinline__ void router_row_prefetch(const uint16_t* wr, int H, bool has_row, uint4 (&w0)[8])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int h0 = u * 256 + lane * 8;
        w0[u] = has_row && h0 < H ? __ldg(reinterpret_cast<const uint4*>(wr + h0)) : make_uint4(0, 0, 0, 0);
    }
}

// Largest |value| of a 16-byte vector of 8 bf16 values, as the bit pattern of a non-negative float
// (non-negative floats order like their bit patterns).
__device__ __forceinline__ uint32_t absmax8_bits(const uint4& v)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m = max(m, __float_as_uint(fabsf(bf16_to_f32(w[i] & 0xFFFFu))));
        m = max(m, __float_as_uint(fabsf(bf16_to_f32(w[i] >> 16))));
    }
    return m;
}

// The W4A4 tensor scale S = amax / (6 * 448), 1 for an all-zero tensor (amax as a float).
__device__ __forceinline__ float nvfp4_tensor_scale(float amax) { return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f); }

// NVFP4 encoding of the 16-element blocks b0 .. b1-1 of bf16 x with tensor scale S, one block per
// thread: thread tid of a group of nthreads. x is global or shared memory (row-major [T][H], H a
// multiple of 16, so block b is the 16 values from x + 16 b).
__device__ __forceinline__ void quantize_blocks(const uint16_t* x, int64_t b0, int64_t b1, float S, int tid,
                                                int nthreads, uint8_t* codes, uint8_t* sf)
{
    const float six_s = __fmul_rn(6.0f, S);
    for (int64_t b = b0 + tid; b < b1; b += nthreads) {
        float v[16];
        const uint4 p0 = reinterpret_cast<const uint4*>(x + b * 16)[0];
        const uint4 p1 = reinterpret_cast<const uint4*>(x + b * 16)[1];
        const uint32_t w8[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = bf16_to_f32(w8[i] & 0xFFFFu);
            v[2 * i + 1] = bf16_to_f32(w8[i] >> 16);
        }
        uint32_t lo, hi;
        const uint32_t s = nvfp4_encode16(v, S, six_s, lo, hi);
        *reinterpret_cast<uint2*>(codes + b * 8) = make_uint2(lo, hi);
        sf[b] = static_cast<uint8_t>(s);
    }
}

// GPU-scope fetch-and-add with acquire-release semantics: the caller's earlier writes (and those
// of its CTA, ordered before it by a block barrier) are visible to whoever reads the result, and
// writes that preceded the earlier additions are visible to the caller.
__device__ __forceinline__ unsigned atomic_add_acq_rel(unsigned* p, unsigned v)
{
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Stable permutation of the n = T*k assignments ids[0..n) (shared memory, n <= 2 * kThreads, the
// entries from n up to the next multiple of 4 set to INT_MAX) by expert id, by one CTA of kThreads
// threads: the position of assignment f is the number of assignments with a smaller id plus the
// earlier ones with the same id (ids read 4 at a time); offsets[e] (e = 0..E, E + 1 <= 5 *
// kThreads) = the assignments with an id below e, a lower bound in the ids in position order
// (sorted: n ints of shared memory), every thread running its bounds side by side; offsets[E+1] =
// n + T and the shared expert's rows n + t hold token t. Contains one block barrier (all threads
// must call).
template <int kThreads>
__device__ __forceinline__ void block_small_permute(const int32_t* ids, int n, int k, int T, int E, int32_t* sorted,
                                                    int32_t* offsets, int32_t* perm_src, int32_t* src_perm,
                                                    int32_t* row_token)
{
    const int tid = threadIdx.x;
    for (int f = tid; f < n; f += kThreads) {
        const int id = ids[f];
        int pos = 0;
#pragma unroll 2
        for (int q0 = 0; q0 < n; q0 += 4) {
            const int4 v = *reinterpret_cast<const int4*>(ids + q0);
            pos += (v.x < id) | ((v.x == id) & (q0 < f));
            pos += (v.y < id) | ((v.y == id) & (q0 + 1 < f));
            pos += (v.z < id) | ((v.z == id) & (q0 + 2 < f));
            pos += (v.w < id) | ((v.w == id) & (q0 + 3 < f));
        }
        perm_src[pos] = f;
        if (src_perm) src_perm[f] = pos;
        row_token[pos] = f / k;
        sorted[pos] = id;
    }
    __syncthreads();
    constexpr int kE = 5;
    int base[kE];
#pragma unroll
    for (int j = 0; j < kE; ++j) base[j] = 0;
    for (int len = n; len > 1;) {  // branch-free lower bounds: the answer stays in [base, base + len]
        const int half = len >> 1;
#pragma unroll
        for (int j = 0; j < kE; ++j) base[j] = sorted[base[j] + half] < tid + j * kThreads ? base[j] + half : base[j];
        len -= half;
    }
#pragma unroll
    for (int j = 0; j < kE; ++j) {
        const int e = tid + j * kThreads;
        if (e <= E) offsets[e] = base[j] + (sorted[base[j]] < e);
    }
    if (tid == 0) offsets[E + 1] = n + T;
    for (int t = tid; t < T; t += kThreads) row_token[n + t] = t;
}

}  // namespace moe
