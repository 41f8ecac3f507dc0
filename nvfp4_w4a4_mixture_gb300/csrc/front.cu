// front.cu -- the layer's front half for small batches in one launch: W4A4 quantisation of x,
// router logits, FP32 softmax top-k with renormalised weights, shared gate, and the stable
// permutation by expert id.
//
// Every CTA but the last computes the logits of 8 router rows for all tokens (the same per-lane
// strided FP32 sums and butterfly as the standalone router, so the logits are bit-identical to it);
// the last CTA quantises x. Each CTA then takes a ticket; the last CTA to finish reads all logits
// and does the top-k (one warp per token: integer keys, a four-entry cache per lane, lowest index
// first on ties) and the stable permutation (rank by counting, offsets by binary search over the
// ids in position order), then returns the ticket counter to zero for the next call. No CTA waits
// for another, so the launch needs no co-residency.
#include <cfloat>

#include "kernels.cuh"
#include "topk.cuh"

namespace moe {

namespace {

constexpr int kFrontThreads = 256;
constexpr int kFrontWarps = kFrontThreads / 32;
constexpr int kFrontTT = 8;        // tokens staged per pass
constexpr int kFrontMaxE = 1024;
constexpr int kFrontMaxT = 64;
constexpr int kSmallFrontAssign = 512;  // T * k

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
    __shared__ int32_t sorted_s[kSmallFrontAssign];
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

    // top-k per token: warp w takes tokens w, w + 8, ...
    for (int t = warp; t < T; t += kFrontWarps) {
        const float* l = a.logits + static_cast<int64_t>(t) * (E + 1);
        const float l_gate = lane == 0 ? __ldcg(l + E) : 0.0f;  // shared-gate logit, loaded with the rest
        float sel_l, l0;
        int sel_i;
        warp_topk(l, E, k, sel_l, sel_i, l0);
        const float w = warp_topk_weight(sel_l, l0, k);
        if (lane < k) {
            a.topk_ids[static_cast<int64_t>(t) * k + lane] = sel_i;
            a.topk_w[static_cast<int64_t>(t) * k + lane] = w;
            ids_s[t * k + lane] = sel_i;
        }
        if (lane == 0) a.shared_g[t] = 1.0f / (1.0f + expf(-l_gate));
    }
    // permutation: the position of assignment f is the number of assignments with a smaller id plus
    // the earlier ones with the same id (stable); the ids in position order then give the expert
    // offsets by binary search (offsets[e] = assignments with an id below e)
    const int n = T * k;
    __syncthreads();  // ids_s complete
    for (int f = tid; f < n; f += kFrontThreads) {
        const int id = ids_s[f];
        int pos = 0;
        for (int q = 0; q < n; ++q) {
            const int o = ids_s[q];
            pos += (o < id) | ((o == id) & (q < f));
        }
        a.perm_src[pos] = f;
        a.src_perm[f] = pos;
        a.row_token[pos] = f / k;
        sorted_s[pos] = id;
    }
    __syncthreads();
    for (int e = tid; e <= E; e += kFrontThreads) {
        int lo = 0, hi = n;  // first position whose id is >= e
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (sorted_s[mid] < e) lo = mid + 1; else hi = mid;
        }
        a.offsets[e] = lo;
    }
    if (tid == 0) a.offsets[E + 1] = n + T;
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
