// front.cu -- the layer's front half for small batches in one launch: W4A4 quantisation of x,
// router logits, FP32 softmax top-k with renormalised weights, shared gate, and the stable
// permutation by expert id.
//
// Every CTA computes the logits of 8 router rows for all tokens (the same per-lane strided FP32
// sums and butterfly as the standalone router, so the logits are bit-identical to it), takes the
// tensor max of x while staging it and quantises its share of x's 16-element blocks. Each CTA then
// takes a ticket; the last CTA to finish reads all logits and does the top-k (one warp per token:
// integer keys, a four-entry cache per lane, lowest index first on ties) and the stable
// permutation (rank by counting, offsets by binary search over the ids in position order), then
// returns the ticket counter to zero for the next call. No CTA waits for another, so the launch
// needs no co-residency.
#include <cfloat>

#include "kernels.cuh"
#include "route.cuh"
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

    // The router row does not depend on the previous launch on the stream: its first 2048 columns
    // are loaded before waiting for that launch (x and the routing outputs may still be in use there).
    const bool has_row = e <= E;
    const uint16_t* wr = a.w_router + static_cast<int64_t>(has_row ? e : 0) * H;
    uint4 wv0[8];
    router_row_prefetch(wr, H, has_row, wv0);
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();

    // ---- logits of this CTA's router rows, kFrontTT tokens per pass; every CTA sees all of x, so
    // it also takes the tensor max on the way
    uint32_t amax_bits = 0;
    for (int t0 = 0; t0 < T; t0 += kFrontTT) {
        const int nt = min(kFrontTT, T - t0);
        const int vec_per_row = H / 8;
#pragma unroll 4
        for (int i = tid; i < nt * vec_per_row; i += kFrontThreads) {
            const int t = i / vec_per_row, c = i % vec_per_row;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(t0 + t) * H) + c);
            reinterpret_cast<uint4*>(xs + t * H)[c] = v;
            amax_bits = max(amax_bits, absmax8_bits(v));
        }
        __syncthreads();
        if (has_row) {
            float acc[kFrontTT];
            router_row_logits<kFrontTT>(xs, H, wr, wv0, acc);
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

    // ---- W4A4 quantisation of x: the tensor scale from the max, then this CTA's share of the blocks
    amax_bits = __reduce_max_sync(0xFFFFFFFFu, amax_bits);
    if (lane == 0) red_s[warp] = __uint_as_float(amax_bits);
    __syncthreads();
    float amax = 0.0f;
#pragma unroll
    for (int w = 0; w < kFrontWarps; ++w) amax = fmaxf(amax, red_s[w]);
    const float S = nvfp4_tensor_scale(amax);
    if (blockIdx.x == 0 && tid == 0) *a.s_x = S;
    {
        const int64_t nblocks = static_cast<int64_t>(T) * H / 16;
        const int64_t per = (nblocks + gridDim.x - 1) / gridDim.x;
        const int64_t b0 = min(nblocks, static_cast<int64_t>(blockIdx.x) * per), b1 = min(nblocks, b0 + per);
        quantize_blocks(a.x, b0, b1, S, kFrontThreads, a.xq_codes, a.xq_sf);
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
    // permutation (stable; offsets by binary search over the ids in position order)
    __syncthreads();  // ids_s complete
    block_small_permute(ids_s, T * k, k, T, E, kFrontThreads, sorted_s, a.offsets, a.perm_src, a.src_perm, a.row_token);
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
    const int grid = (E + 1 + kFrontWarps - 1) / kFrontWarps;  // 8 router rows per CTA
    return launch_pdl(k_decode_front, dim3(grid), dim3(kFrontThreads), smem, stream, a);
}

}  // namespace moe
