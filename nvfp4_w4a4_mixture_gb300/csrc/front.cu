// front.cu -- the layer's front half for small batches in one launch: W4A4 quantisation of x,
// router logits, FP32 softmax top-k with renormalised weights, shared gate, and the stable
// permutation by expert id.
//
// Every CTA computes the logits of 4 router rows for all tokens, two warps per row, each taking
// half of every pass of staged tokens (per token the same per-lane strided FP32 sums and butterfly
// as the standalone router, so the logits are bit-identical to it), and takes the tensor max of x
// while staging it. Each CTA then takes a ticket (an acquire-release addition, so the logits of
// every CTA before it are visible to it) and quantises a chunk of x's 16-element blocks chosen by
// its arrival (from the staged copy when one pass holds every token); the chunks cover x without
// the last CTA. The last CTA to arrive reads all logits and does the top-k (one warp per token:
// integer keys, candidates above the k-th largest lane maximum ranked in shared memory, lowest
// index first on ties) and the stable permutation (rank by counting, offsets by lower bounds in the
// ids in position order), then returns the ticket counter to zero for the next call. No CTA waits
// for another, so the launch needs no co-residency. The last CTA's part is the launch's critical
// path: short dependency chains, few barriers.
#include <cfloat>
#include <climits>

#include "kernels.cuh"
#include "route.cuh"
#include "topk.cuh"

namespace moe {

namespace {

constexpr int kFrontThreads = 256;
constexpr int kFrontWarps = kFrontThreads / 32;
constexpr int kFrontRows = kFrontWarps / 2;  // router rows per CTA: two warps per row, each half the tokens
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
    int32_t* offsets;      // [E+2]; null: no permutation (the expert GEMMs build it)
    int32_t* perm_src;     // [T*k]
    int32_t* src_perm;
    int32_t* row_token;    // [T*k + T]
    unsigned* ticket;      // zero between calls
    int32_t* ready;        // [n_ready] token-block counters of the expert GEMMs, zeroed here
    int n_ready;
};

// kTT = tokens staged per pass (4 or 8); each warp of a row pair takes kTT / 2 of them.
template <int kTT>
__global__ void __launch_bounds__(kFrontThreads) k_decode_front(const FrontArgs a)
{
    extern __shared__ __align__(16) uint8_t fsm[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(fsm);  // [kTT][H]
    __shared__ __align__(16) int32_t ids_s[kSmallFrontAssign + 4];
    __shared__ int32_t sorted_s[kSmallFrontAssign];
    __shared__ uint2 cand_s[kFrontWarps][kTopkCand];
    __shared__ uint2 sel_s[kFrontWarps][32];
    __shared__ float red_s[kFrontWarps];
    __shared__ unsigned last_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, E = a.E, T = a.T, k = a.k;
    const int e = blockIdx.x * kFrontRows + (warp >> 1);  // this warp's router row (E = shared gate)
    const int half = warp & 1;                              // which half of each token pass
    constexpr int kHT = kTT / 2;

    // The router row does not depend on the previous launch on the stream: its first 2048 columns
    // are loaded before waiting for that launch (x and the routing outputs may still be in use there).
    const bool has_row = e <= E;
    const uint16_t* wr = a.w_router + static_cast<int64_t>(has_row ? e : 0) * H;
    uint4 wv0[8];
    router_row_prefetch(wr, H, has_row, wv0);
    ptx::griddep_wait();

    // ---- logits of this CTA's router rows, kTT tokens per pass; every CTA sees all of x, so it
    // also takes the tensor max on the way
    uint32_t amax_bits = 0;
    for (int t0 = 0; t0 < T; t0 += kTT) {
        const int nt = min(kTT, T - t0);
        const int vec_per_row = H / 8;
#pragma unroll 4
        for (int i = tid; i < nt * vec_per_row; i += kFrontThreads) {
            const int t = i / vec_per_row, c = i % vec_per_row;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(t0 + t) * H) + c);
            reinterpret_cast<uint4*>(xs + t * H)[c] = v;
            amax_bits = max(amax_bits, absmax8_bits(v));
        }
        __syncthreads();
        if (has_row && half * kHT < nt) {
            float acc[kHT];
            router_row_logits<kHT>(xs + half * kHT * H, H, wr, wv0, acc);
            if (lane < min(kHT, nt - half * kHT)) {
                float v = 0.0f;
#pragma unroll
                for (int t = 0; t < kHT; ++t)
                    if (t == lane) v = acc[t];
                if (a.bias && e < E) v = __fadd_rn(v, a.bias[e]);
                a.logits[static_cast<int64_t>(t0 + half * kHT + lane) * (E + 1) + e] = v;
            }
        }
        if (t0 + kTT < T) __syncthreads();  // xs is restaged; a single pass keeps it for the quantiser
    }

    // ---- the tensor max of x, then the ticket: the last CTA to publish its logits routes and
    // permutes; every CTA quantises its share of x's blocks after the ticket, off that path
    amax_bits = __reduce_max_sync(0xFFFFFFFFu, amax_bits);
    if (lane == 0) red_s[warp] = __uint_as_float(amax_bits);
    __syncthreads();  // (orders this CTA's logits before thread 0's release)
    if (tid == 0) last_s = atomic_add_acq_rel(a.ticket, 1u);
    __syncthreads();
    const unsigned arrival = last_s;  // 0 .. gridDim.x - 1 in ticket order
    float amax = 0.0f;
#pragma unroll
    for (int w = 0; w < kFrontWarps; ++w) amax = fmaxf(amax, red_s[w]);
    const float S = nvfp4_tensor_scale(amax);
    if (blockIdx.x == 0 && tid == 0) *a.s_x = S;
    // x's blocks in chunks by arrival: the first gridDim.x - 1 CTAs share them, the last has none
    const int64_t nblocks = static_cast<int64_t>(T) * H / 16;
    const int nq = max(1u, gridDim.x - 1);
    const int64_t per = (nblocks + nq - 1) / nq;
    const int64_t b0 = min(nblocks, static_cast<int64_t>(arrival) * per), b1 = min(nblocks, b0 + per);
    const uint16_t* xq = T <= kTT ? xs : a.x;  // a single pass left every token staged
    quantize_blocks(xq, b0, b1, S, tid, kFrontThreads, a.xq_codes, a.xq_sf);
    if (arrival != gridDim.x - 1) {
        ptx::griddep_launch_dependents();  // this CTA's outputs are written
        return;
    }

    // ---- last CTA: one warp per token (top-k), then the permutation. The next launch may start
    // now: its CTAs take the SMs the other CTAs have left and run their prologue during this tail
    // (their dependent reads wait for this grid to complete)
    ptx::griddep_launch_dependents();
    for (int t = warp; t < T; t += kFrontWarps) {
        const float* l = a.logits + static_cast<int64_t>(t) * (E + 1);
        const float l_gate = lane == 0 ? __ldcg(l + E) : 0.0f;  // shared-gate logit, loaded with the rest
        float sel_l, l0;
        int sel_i;
        const bool done = E <= 512 ? warp_topk_threshold<16>(l, E, k, cand_s[warp], sel_s[warp], sel_l, sel_i, l0)
                                   : warp_topk_threshold<32>(l, E, k, cand_s[warp], sel_s[warp], sel_l, sel_i, l0);
        if (!done) warp_topk(l, E, k, sel_l, sel_i, l0);
        const float w = warp_topk_weight(sel_l, l0, k);
        if (lane < k) {
            a.topk_ids[static_cast<int64_t>(t) * k + lane] = sel_i;
            a.topk_w[static_cast<int64_t>(t) * k + lane] = w;
            ids_s[t * k + lane] = sel_i;
        }
        if (lane == 0) a.shared_g[t] = 1.0f / (1.0f + expf(-l_gate));
    }
    const int n = T * k;
    if (tid < 4) ids_s[n + tid] = INT_MAX;  // pads the ids to a multiple of 4 (n + 4 <= 516)
    __syncthreads();  // ids_s complete
    // stable permutation (rank by counting; offsets by lower bounds in the ids in position order),
    // unless the expert GEMMs build it themselves from the ids (offsets null)
    if (a.offsets)
        block_small_permute<kFrontThreads>(ids_s, n, k, T, E, sorted_s, a.offsets, a.perm_src, a.src_perm, a.row_token);
    for (int i = tid; i < a.n_ready; i += kFrontThreads) a.ready[i] = 0;
    if (tid == 0) *a.ticket = 0u;  // every CTA has taken its ticket: ready for the next call
    ptx::griddep_launch_dependents();
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
    const int tt = T <= 4 ? 4 : 8;
    const size_t smem = static_cast<size_t>(tt) * H * sizeof(uint16_t);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_decode_front<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, 150 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_decode_front<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, 150 * 1024);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    FrontArgs a{x, T, H, E, k, w_router, bias, logits, xq_codes, xq_sf, s_x, topk_ids, topk_w, shared_g, offsets,
                perm_src, src_perm, row_token, ticket, ready, n_ready};
    const int grid = (E + 1 + kFrontRows - 1) / kFrontRows;
    return tt == 4 ? launch_pdl(k_decode_front<4>, dim3(grid), dim3(kFrontThreads), smem, stream, a)
                   : launch_pdl(k_decode_front<8>, dim3(grid), dim3(kFrontThreads), smem, stream, a);
}

}  // namespace moe
