// front.cu -- the layer's front half for small batches in one launch: W4A4 quantisation of x,
// router logits, FP32 softmax top-k with renormalised weights, shared gate, and the stable
// permutation by expert id.
//
// Every CTA computes the logits of 8 router rows for all tokens (the same per-lane strided FP32
// sums and butterfly as the standalone router, so the logits are bit-identical to it); CTA 0 also
// quantises x (it reads the whole tensor anyway for its max). Each CTA then takes a ticket; the
// last CTA to finish reads all logits and does the top-k (one warp per token, k rounds of a warp
// arg-max, lowest index first on ties) and the permutation (counts, scan, rank by direct count:
// stable and bit-exact), then returns the ticket counter to zero for the next call. No CTA waits
// for another, so the launch needs no co-residency.
#include <cfloat>

#include "kernels.cuh"

namespace moe {

namespace {

constexpr int kFrontThreads = 256;
constexpr int kFrontWarps = kFrontThreads / 32;
constexpr int kFrontTT = 8;        // tokens staged per pass
constexpr int kFrontMaxE = 1024;
constexpr int kFrontMaxT = 64;
constexpr int kSmallFrontAssign = 512;  // T * k

// Order-preserving key of a logit: a larger logit has a larger key; every logit, -inf included, has
// a key >= 1, and NaN ranks with -inf (so the selected ids always lie in [0, E)).
__device__ __forceinline__ uint32_t order_key(float v)
{
    if (v != v) v = -INFINITY;
    if (v == 0.0f) v = 0.0f;  // -0 ties with +0
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// A lane's four largest keys, largest first (equal keys: lowest slot first); unused entries hold 0.
struct Top4 {
    uint32_t k[4];
    int s[4];
};

__device__ __forceinline__ void lane_top4(const uint32_t (&key)[32], Top4& c)
{
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        c.k[q] = 0u;
        c.s[q] = 31;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        uint32_t kv = key[i];
        int sv = i;
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // insertion: a strictly larger key moves ahead
            const bool gt = kv > c.k[q];
            const uint32_t tk = gt ? c.k[q] : kv;
            const int ts = gt ? c.s[q] : sv;
            c.k[q] = gt ? kv : c.k[q];
            c.s[q] = gt ? sv : c.s[q];
            kv = tk;
            sv = ts;
        }
    }
}

// Exclusive scan of cnt[0..n) (n <= 1024) in place by 256 threads; returns the total.
__device__ int32_t block_exclusive_scan(int32_t* cnt, int n, int32_t* wsum)
{
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    int32_t v[4], s = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = t * 4 + i;
        v[i] = e < n ? cnt[e] : 0;
        s += v[i];
    }
    int32_t x = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int32_t w = lane < kFrontWarps ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kFrontWarps) wsum[lane] = w;
    }
    __syncthreads();
    int32_t run = x - s + (warp > 0 ? wsum[warp - 1] : 0);
    const int32_t total = wsum[kFrontWarps - 1];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = t * 4 + i;
        if (e < n) cnt[e] = run;
        run += v[i];
    }
    __syncthreads();
    return total;
}

}  // namespace

struct FrontArgs {
    const uint16_t* x;
    int T, H, E, k;
    const uint16_t* w_router;
    const float* bias;
    float* logits;         // scratch [T][E+1]
    uint8_t* xq_codes;     // [T][H/2]
    uint8_t* xq_sf;        // [T][H/16]
    float* s_x;
    int32_t* topk_ids;     // [T][k]
    float* topk_w;
    float* shared_g;
    int32_t* offsets;      // [E+2]
    int32_t* perm_src;     // [T*k]
    int32_t* src_perm;
    int32_t* row_token;    // [T*k + T]
    unsigned* ticket;      // zero between calls
    int32_t* ready;        // [n_ready] token-block counters of the expert GEMMs, zeroed here
    int n_ready;
};

__global__ void __launch_bounds__(kFrontThreads) k_decode_front(const FrontArgs a)
{
    extern __shared__ __align__(16) uint8_t fsm[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(fsm);  // [kFrontTT][H]
    __shared__ int32_t ids_s[kSmallFrontAssign];
    __shared__ int32_t cnt_s[kFrontMaxE];
    __shared__ int32_t wsum_s[32];
    __shared__ float red_s[kFrontWarps];
    __shared__ unsigned last_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, E = a.E, T = a.T, k = a.k;
    const int e = blockIdx.x * kFrontWarps + warp;  // this warp's router row (E = shared gate)
    const int n_logit_ctas = (E + 1 + kFrontWarps - 1) / kFrontWarps;

    // The router row does not depend on the previous launch on the stream: its first 2048 columns
    // are loaded before waiting for that launch (x and the routing outputs may still be in use there).
    const bool has_row = blockIdx.x < n_logit_ctas && e <= E;
    const uint16_t* wr = a.w_router + static_cast<int64_t>(has_row ? e : 0) * H;
    uint4 wv0[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int h0 = u * 256 + lane * 8;
        wv0[u] = has_row && h0 < H ? __ldg(reinterpret_cast<const uint4*>(wr + h0)) : make_uint4(0, 0, 0, 0);
    }
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();

    // ---- logits of this CTA's router rows, kFrontTT tokens per pass (CTAs 0 .. n_logit_ctas-1)
    for (int t0 = 0; t0 < T && blockIdx.x < n_logit_ctas; t0 += kFrontTT) {
        const int nt = min(kFrontTT, T - t0);
        const int vec_per_row = H / 8;
#pragma unroll 4
        for (int i = tid; i < nt * vec_per_row; i += kFrontThreads) {
            const int t = i / vec_per_row, c = i % vec_per_row;
            reinterpret_cast<uint4*>(xs + t * H)[c] =
                __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(t0 + t) * H) + c);
        }
        __syncthreads();
        if (has_row) {
            float acc[kFrontTT];
#pragma unroll
            for (int t = 0; t < kFrontTT; ++t) acc[t] = 0.0f;
            for (int base = 0; base < H; base += 8 * 256) {
                uint4 wv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int h0 = base + u * 256 + lane * 8;
                    wv[u] = base == 0 ? wv0[u]
                                      : (h0 < H ? __ldg(reinterpret_cast<const uint4*>(wr + h0)) : make_uint4(0, 0, 0, 0));
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int h0 = base + u * 256 + lane * 8;
                    if (h0 >= H) break;
                    const uint32_t ww[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
#pragma unroll
                    for (int t = 0; t < kFrontTT; ++t) {
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
            for (int t = 0; t < kFrontTT; ++t) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc[t] = __fadd_rn(acc[t], __shfl_xor_sync(0xFFFFFFFFu, acc[t], o));
            }
            if (lane < nt) {
                float v = 0.0f;
#pragma unroll
                for (int t = 0; t < kFrontTT; ++t)
                    if (t == lane) v = acc[t];
                if (a.bias && e < E) v = __fadd_rn(v, a.bias[e]);
                a.logits[static_cast<int64_t>(t0 + lane) * (E + 1) + e] = v;
            }
        }
        __syncthreads();
    }

    // ---- last CTA: W4A4 quantisation of x (tensor max, then one thread per 16-element block)
    if (blockIdx.x == n_logit_ctas) {
        const int64_t nblocks = static_cast<int64_t>(T) * H / 16;
        uint32_t m = 0;
        for (int64_t b = tid; b < nblocks; b += kFrontThreads) {
            const uint4 p0 = __ldg(reinterpret_cast<const uint4*>(a.x + b * 16));
            const uint4 p1 = __ldg(reinterpret_cast<const uint4*>(a.x + b * 16) + 1);
            const uint32_t w8[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                m = max(m, __float_as_uint(fabsf(bf16_to_f32(w8[i] & 0xFFFFu))));
                m = max(m, __float_as_uint(fabsf(bf16_to_f32(w8[i] >> 16))));
            }
        }
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0) red_s[warp] = __uint_as_float(m);
        __syncthreads();
        float amax = 0.0f;
#pragma unroll
        for (int w = 0; w < kFrontWarps; ++w) amax = fmaxf(amax, red_s[w]);
        const float S = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
        if (tid == 0) *a.s_x = S;
        const float six_s = __fmul_rn(6.0f, S);
        for (int64_t b = tid; b < nblocks; b += kFrontThreads) {
            float v[16];
            const uint4 p0 = __ldg(reinterpret_cast<const uint4*>(a.x + b * 16));
            const uint4 p1 = __ldg(reinterpret_cast<const uint4*>(a.x + b * 16) + 1);
            const uint32_t w8[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                v[2 * i] = bf16_to_f32(w8[i] & 0xFFFFu);
                v[2 * i + 1] = bf16_to_f32(w8[i] >> 16);
            }
            uint32_t lo, hi;
            const uint32_t sf = nvfp4_encode16(v, S, six_s, lo, hi);
            *reinterpret_cast<uint2*>(a.xq_codes + b * 8) = make_uint2(lo, hi);
            a.xq_sf[b] = static_cast<uint8_t>(sf);
        }
    }

    // ---- ticket: the last CTA to finish routes and permutes
    __threadfence();
    __syncthreads();
    if (tid == 0) last_s = atomicAdd(a.ticket, 1u) == gridDim.x - 1 ? 1u : 0u;
    __syncthreads();
    if (!last_s) return;
    __threadfence();

    // top-k per token: warp w takes tokens w, w + 8, ...; lane l holds logits l, l + 32, ... as
    // order-preserving integer keys (a removed or absent entry has key 0, below every logit) and a
    // cache of its four largest. A round takes the warp's largest cached key with one reduction and
    // the lowest expert id holding it with a second; the winning lane pops its cache and rebuilds it
    // from its remaining keys only when it runs empty.
    for (int t = warp; t < T; t += kFrontWarps) {
        const float* l = a.logits + static_cast<int64_t>(t) * (E + 1);
        uint32_t key[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int ee = i * 32 + lane;
            key[i] = ee < E ? order_key(__ldcg(l + ee)) : 0u;
        }
        Top4 c;
        lane_top4(key, c);
        float sel_l = 0.0f;
        int sel_i = 0;
        uint32_t k0 = 0;
        for (int j = 0; j < k; ++j) {
            const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, c.k[0]);
            const int widx = static_cast<int>(__reduce_min_sync(
                0xFFFFFFFFu, c.k[0] == wmax ? static_cast<unsigned>(c.s[0] * 32 + lane) : 0x7FFFFFFFu));
            if (j == 0) k0 = wmax;
            if (lane == j) {
                sel_l = key_value(wmax);
                sel_i = widx;
            }
            if ((widx & 31) == lane) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i == c.s[0]) key[i] = 0u;
#pragma unroll
                for (int q = 0; q < 3; ++q) {
                    c.k[q] = c.k[q + 1];
                    c.s[q] = c.s[q + 1];
                }
                c.k[3] = 0u;
                c.s[3] = 31;
                if (c.k[0] == 0u) lane_top4(key, c);
            }
        }
        // renormalised weights: softmax over the selected logits (the first one is the largest)
        const float l0 = key_value(k0);
        const float p = lane < k ? expf(sel_l - l0) : 0.0f;
        float sum = p;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        if (lane < k) {
            a.topk_ids[static_cast<int64_t>(t) * k + lane] = sel_i;
            a.topk_w[static_cast<int64_t>(t) * k + lane] = p / sum;
            ids_s[t * k + lane] = sel_i;
        }
        if (lane == 0) a.shared_g[t] = 1.0f / (1.0f + expf(-__ldcg(l + E)));
    }
    // permutation: counts, exclusive scan over experts, then warp 0 places the assignments in order,
    // 32 at a time: rank = earlier lanes with the same id (match) + the id's running count
    const int n = T * k;
    for (int i = tid; i < E; i += kFrontThreads) cnt_s[i] = 0;
    __syncthreads();
    for (int f = tid; f < n; f += kFrontThreads) atomicAdd(&cnt_s[ids_s[f]], 1);
    __syncthreads();
    const int32_t total = block_exclusive_scan(cnt_s, E, wsum_s);
    for (int i = tid; i < E; i += kFrontThreads) a.offsets[i] = cnt_s[i];
    if (tid == 0) {
        a.offsets[E] = total;
        a.offsets[E + 1] = total + T;
    }
    __syncthreads();
    if (warp == 0) {
        for (int c0 = 0; c0 < n; c0 += 32) {
            const int f = c0 + lane;
            const int id = f < n ? ids_s[f] : -1;
            const unsigned m = __match_any_sync(0xFFFFFFFFu, id);
            if (f < n) {
                const int pos = cnt_s[id] + __popc(m & ((1u << lane) - 1u));
                a.perm_src[pos] = f;
                a.src_perm[f] = pos;
                a.row_token[pos] = f / k;
            }
            __syncwarp();
            if (f < n && (m >> lane) == 1u) cnt_s[id] += __popc(m);  // highest lane of each id
            __syncwarp();
        }
    }
    for (int t = tid; t < T; t += kFrontThreads) a.row_token[n + t] = t;
    for (int i = tid; i < a.n_ready; i += kFrontThreads) a.ready[i] = 0;
    if (tid == 0) *a.ticket = 0u;  // every CTA has taken its ticket: ready for the next call
}

bool front_fits(int T, int H, int E, int k)
{
    return T >= 1 && T <= kFrontMaxT && static_cast<int64_t>(T) * k <= kSmallFrontAssign && E <= kFrontMaxE && H <= 8192;
}

cudaError_t launch_front(const uint16_t* x, int T, int H, int E, int k, const uint16_t* w_router, const float* bias,
                         float* logits, uint8_t* xq_codes, uint8_t* xq_sf, float* s_x, int32_t* topk_ids, float* topk_w,
                         float* shared_g, int32_t* offsets, int32_t* perm_src, int32_t* src_perm, int32_t* row_token,
                         unsigned* ticket, int32_t* ready, int n_ready, cudaStream_t stream)
{
    const size_t smem = static_cast<size_t>(kFrontTT) * H * sizeof(uint16_t);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_decode_front, cudaFuncAttributeMaxDynamicSharedMemorySize, 150 * 1024);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    FrontArgs a{x, T, H, E, k, w_router, bias, logits, xq_codes, xq_sf, s_x, topk_ids, topk_w, shared_g, offsets,
                perm_src, src_perm, row_token, ticket, ready, n_ready};
    const int grid = (E + 1 + kFrontWarps - 1) / kFrontWarps + 1;  // router rows + one quantising CTA
    return launch_pdl(k_decode_front, dim3(grid), dim3(kFrontThreads), smem, stream, a);
}

}  // namespace moe
