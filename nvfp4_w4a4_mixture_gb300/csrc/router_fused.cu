// router_fused.cu -- the routing half of the layer's front for large batches with 512 routed experts,
// in one launch per call:
//   logits[t][e] = sum_h x[t][h] * w_router[e][h] (+ bias[e]) for e < 512, on the tensor cores
//     (tcgen05.mma kind::f16, bf16 operands, FP32 accumulation in tensor memory; two 256-column
//     accumulators hold all 512 logits of a 128-token block, so one CTA sees whole rows);
//   the shared-gate logit (router row 512) as a sequential FP32 sum on the CUDA cores;
//   the top-k of the 512 logits (larger logit first, lower expert id first on equal logits), the
//     weights renormalised over the k selected (the softmax denominator cancels) and the shared gate
//     sigmoid(gate logit), as the gating network of the layer defines them;
//   max |x| over the block's rows, one slot per CTA (the W4A4 quantizer's tensor scale reduces them).
// Every product of two bf16 values is exact in FP32, so the logits differ from a sequential FP32 sum
// by the order of the additions only (here: K-slices of 64 in a rotated order, see k_rot).
//
// One CTA per 128-token block (one wave up to 152 x 128 tokens; below about 12k tokens the separate
// router and top-k launches spread the same work over more SMs and are faster). Three warps load the
// 64-column K-slices (128 bytes per row, 128-byte swizzle) into a 2-deep ring of 80 KB stages, one
// TMA box each per slice: warp 0 the 128 x rows, warps 6 and 7 router rows 0-255 and 256-511 (with
// one thread issuing a slice's boxes the measured time per slice was about the same, 1.08 against
// 1.03 us). Warp 1 owns the 512 tensor-memory columns and issues, per slice, four K=16 steps of two
// 128 x 256 MMAs. Warps 2-5 own one tensor-memory lane quarter each and one token row per thread:
// during the main loop they read each staged slice of x for the gate logit and the maximum (and free
// the stage together with the MMA's commit); afterwards they read their row's 512 accumulator columns,
// store the logits and select the top-k (below).
#include <cfloat>

#include "kernels.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kRfM = 128;         // tokens per CTA (MMA M, tensor-memory lanes)
constexpr int kRfE = 512;         // routed experts (two 256-column accumulators)
constexpr int kRfBK = 64;         // bf16 K-values per slice (128 bytes per row)
constexpr int kRfStages = 2;
constexpr int kRfABytes = kRfM * kRfBK * 2;           // 16 KB
constexpr int kRfBBytes = kRfE * kRfBK * 2;           // 64 KB
constexpr int kRfStageBytes = kRfABytes + kRfBBytes;  // 80 KB
constexpr int kRfThreads = 256;
constexpr int kRfLoaders = 3;  // warps 0, 6, 7: one TMA box each per slice
constexpr int kRfEpiWarps = 4;
constexpr int kRfMaxK = 16;
constexpr int kRfMaxH = 8192;
constexpr int kRfCand = 95;  // top-k candidates per row kept in shared memory (+1 scratch slot)
constexpr int kRfXpOff = (kRfCand + 1) * 8 * kRfM;  // per-warp 32 x 36-float transpose buffers after them
static_assert(kRfStageBytes % 1024 == 0 && kRfABytes % 1024 == 0, "128-byte swizzle atoms stay aligned");
static_assert(kRfXpOff + kRfEpiWarps * 32 * 36 * 4 <= kRfStages * kRfStageBytes,
              "candidate lists and transpose buffers fit in the idle ring");

struct RfTail {
    uint64_t full[kRfStages];
    uint64_t empty[kRfStages];
    uint64_t acc_full;
    uint32_t tmem_base;
    int abort;
    uint32_t amax_w[kRfEpiWarps];
};

size_t rf_smem(int H)
{
    return 1024 + static_cast<size_t>(kRfStages) * kRfStageBytes + static_cast<size_t>(H) * 2 + sizeof(RfTail);
}

struct RfArgs {
    int T, H, k;
    const uint16_t* w_gate;  // router row 512 (the shared gate), H bf16
    const float* bias;       // nullable [512]
    float* logits;           // [T][ld], column 512 = gate logit
    int ld;
    int32_t* topk_ids;       // [T][k]
    float* topk_w;           // [T][k]
    float* shared_g;         // nullable [T]
    uint32_t* amax_slots;    // nullable [gridDim.x]: max |x| of each CTA's rows, as float bits
    int32_t* zero;           // nullable [n_zero]: zeroed for the launches that follow
    int n_zero;
    int* status;
};

__global__ void __launch_bounds__(kRfThreads, 1)
    k_router_topk(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w, const RfArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint16_t* wg_s = reinterpret_cast<uint16_t*>(smem + kRfStages * kRfStageBytes);
    RfTail& st = *reinterpret_cast<RfTail*>(smem + kRfStages * kRfStageBytes + a.H * 2);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int tb = blockIdx.x;
    const int n_k = a.H / kRfBK;
    // every CTA streams the same router rows: each starts its K walk at another slice (7 x block
    // index, modulo the slice count), so the CTAs' requests for a router line do not all reach its
    // L2 slice at once (16k tokens: 71 -> 63 us). The sums then run in a K order rotated per 128-token
    // block, fixed for a given block.
    const int k_rot = static_cast<int>((static_cast<int64_t>(tb) * 7) % n_k);
    auto slice = [&](int kt) { return kt + k_rot < n_k ? kt + k_rot : kt + k_rot - n_k; };

    if (tid == 0) {
        for (int s = 0; s < kRfStages; ++s) {
            ptx::mbar_init(&st.full[s], kRfLoaders);
            ptx::mbar_init(&st.empty[s], 1 + kRfEpiWarps);  // the MMA's commit + one arrival per epilogue warp
        }
        ptx::mbar_init(&st.acc_full, 1);
        st.abort = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmap_x);
        ptx::prefetch_tmap(&tmap_w);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&st.tmem_base, 512);
        ptx::tmem_relinquish();
    }
    // the gate row does not depend on the previous launch: staged before waiting for it
    for (int i = tid; i < a.H / 8; i += kRfThreads)
        reinterpret_cast<uint4*>(wg_s)[i] = __ldg(reinterpret_cast<const uint4*>(a.w_gate) + i);
    ptx::griddep_wait();  // x may come from the previous launch, which may also still use zero[]
    if (a.zero)
        for (int i = tb * kRfThreads + tid; i < a.n_zero; i += gridDim.x * kRfThreads) a.zero[i] = 0;
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = st.tmem_base;
    auto fail = [&]() {
        if (atomicExch(&st.abort, 1) == 0) record_status(a.status, kDevTimeoutRouter);
    };
    auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&st.abort) != 0; };

    if (warp == 0 || warp >= 6) {
        // ================================ TMA producers: x rows (warp 0), router rows (warps 6, 7)
        if (lane == 0) {
            const int part = warp == 0 ? 0 : warp - 5;  // 0: x, 1: router rows 0-255, 2: rows 256-511
            const uint32_t bytes = part == 0 ? kRfABytes : kRfBBytes / 2;
            const int off = part == 0 ? 0 : kRfABytes + (part - 1) * (kRfBBytes / 2);
            int s = 0, kt = 0;
            uint32_t ph = 0;
            for (; kt < n_k && !aborted(); ++kt) {
                if (!ptx::mbar_wait(&st.empty[s], ph ^ 1)) { fail(); break; }
                uint8_t* sb = smem + s * kRfStageBytes + off;
                ptx::mbar_arrive_expect_tx(&st.full[s], bytes);
                if (part == 0)
                    ptx::tma_load_2d(sb, &tmap_x, &st.full[s], slice(kt) * kRfBK, tb * kRfM);
                else
                    ptx::tma_load_2d(sb, &tmap_w, &st.full[s], slice(kt) * kRfBK, (part - 1) * 256);
                if (++s == kRfStages) { s = 0; ph ^= 1; }
            }
            if (!ptx::ring_drain(st.full, kRfStages, kt)) fail();
        }
    } else if (warp == 1) {
        // ================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_bf16(kRfM, 256);
            const uint32_t s0 = ptx::smem_u32(smem);
            const uint64_t da0 = ptx::sdesc_sw128(s0);
            const uint64_t db0 = ptx::sdesc_sw128(s0 + kRfABytes), db1 = ptx::sdesc_sw128(s0 + kRfABytes + kRfBBytes / 2);
            constexpr uint64_t kStageAdv = kRfStageBytes >> 4, kKAdv = 32 >> 4;  // K=16 bf16 = 32 bytes
            int s = 0;
            uint32_t ph = 0, acc = 0;
            for (int kt = 0; kt < n_k; ++kt) {
                if (!ptx::mbar_wait(&st.full[s], ph)) { fail(); break; }
                ptx::tc_fence_after();
                const uint64_t so = static_cast<uint64_t>(s) * kStageAdv;
#pragma unroll
                for (int kk = 0; kk < kRfBK / 16; ++kk) {
                    ptx::mma_bf16(tmem, da0 + so + kk * kKAdv, db0 + so + kk * kKAdv, idesc, acc);
                    ptx::mma_bf16(tmem + 256, da0 + so + kk * kKAdv, db1 + so + kk * kKAdv, idesc, acc);
                    acc = 1;
                }
                ptx::tc_commit(&st.empty[s]);
                if (++s == kRfStages) { s = 0; ph ^= 1; }
            }
            // both accumulators complete (or, after a timeout, every issued MMA has finished)
            ptx::tc_commit(&st.acc_full);
        }
    } else {
        // ================================ token rows: gate logit and max |x|, then logits and top-k
        const int q = warp & 3;  // the lane quarter this warp may read
        const int r = q * 32 + lane;
        const int64_t t = static_cast<int64_t>(tb) * kRfM + r;
        const bool row_ok = t < a.T;
        float gate = 0.0f;
        uint32_t amax = 0;
        {
            int s = 0;
            uint32_t ph = 0;
            // 16-byte chunk c of row r sits at chunk c ^ (r & 7) of the row (128-byte swizzle:
            // address bits [4,7) XOR bits [7,10), the slice 1024-byte aligned)
            const int sw = r & 7;
            for (int kt = 0; kt < n_k; ++kt) {
                if (!ptx::mbar_wait(&st.full[s], ph)) { fail(); break; }
                const uint8_t* row = smem + s * kRfStageBytes + r * (kRfBK * 2);
                const uint16_t* wg = wg_s + slice(kt) * kRfBK;
#pragma unroll
                for (int c = 0; c < kRfBK / 8; ++c) {
                    const uint4 v = *reinterpret_cast<const uint4*>(row + ((c ^ sw) * 16));
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float x0 = bf16_to_f32(w4[i] & 0xFFFFu), x1 = bf16_to_f32(w4[i] >> 16);
                        gate = __fmaf_rn(x0, bf16_to_f32(wg[c * 8 + 2 * i]), gate);
                        gate = __fmaf_rn(x1, bf16_to_f32(wg[c * 8 + 2 * i + 1]), gate);
                        amax = max(amax, __float_as_uint(fabsf(x0)));
                        amax = max(amax, __float_as_uint(fabsf(x1)));
                    }
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&st.empty[s]);
                if (++s == kRfStages) { s = 0; ph ^= 1; }
            }
        }
        // the CTA's maximum |x| (rows past T were filled with zeros)
        amax = __reduce_max_sync(0xFFFFFFFFu, amax);
        if (lane == 0) st.amax_w[q] = amax;
        const bool got = ptx::mbar_wait(&st.acc_full, 0);
        if (!got) fail();
        ptx::tc_fence_after();
        // every row warp has left the main loop (another may still be reading its x rows from the
        // ring) before the ring holds candidate lists; all four always arrive here
        asm volatile("bar.sync 1, %0;" ::"r"(32 * kRfEpiWarps) : "memory");
        // one decision per warp: the tensor-memory loads below are warp-collective
        if (__all_sync(0xFFFFFFFFu, got && !aborted())) {
            const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16);
            float* lrow = a.logits + t * a.ld;
            // Top-k in three steps, each thread on its own row. (1) The logits (+ bias) are stored and
            // tau = the k-th largest of 16 chunk maxima is found, chunk c holding the columns e with
            // e % 16 == c (each chunk samples every part of the expert range, so a popularity prior
            // that falls with the id does not loosen the bound): k chunks hold a value >= tau, so the
            // row's k-th largest is >= tau. (2) The keys >= tau (typically 10-30 of 512) go in id
            // order to this thread's candidate list in shared memory (the ring is idle now). (3) They
            // are inserted into a sorted list in registers (key desc, id asc). Inserting every logit
            // directly would cost each warp the insertion at almost every column (some lane inserts
            // at almost every one). When a lane's list overflows, its whole warp inserts from a
            // second pass over the accumulator (the tensor-memory loads stay warp-uniform).
            const int k = a.k;
            uint32_t lk[kRfMaxK];
            int li[kRfMaxK];
            // entries past k hold the largest key, so nothing moves into them and the list's minimum
            // is its k-th entry (every index stays a constant: the list lives in registers)
            auto reset = [&]() {
#pragma unroll
                for (int j = 0; j < kRfMaxK; ++j) {
                    lk[j] = j < k ? 0u : 0xFFFFFFFFu;
                    li[j] = 0;
                }
            };
            auto insert = [&](uint32_t ck, int ci) {  // after every key >= ck
#pragma unroll
                for (int j = 0; j < kRfMaxK; ++j) {
                    const bool gt = ck > lk[j];
                    const uint32_t tk = gt ? lk[j] : ck;
                    const int ti = gt ? li[j] : ci;
                    lk[j] = gt ? ck : lk[j];
                    li[j] = gt ? ci : li[j];
                    ck = tk;
                    ci = ti;
                }
            };
            // this warp's 32 x 32 block of logits, for stores of whole 128-byte row segments
            float* xp = reinterpret_cast<float*>(smem + kRfXpOff) + q * 32 * 36;
            const int64_t t_warp = static_cast<int64_t>(tb) * kRfM + q * 32;
            // this row's logits (+ bias) of columns c0 .. c0 + 31 as keys (stored on the first pass);
            // warp-uniform: every lane of the warp calls it with the same c0
            auto chunk = [&](int c0, bool store, uint32_t (&key)[32]) {
                uint32_t v[32];
                ptx::tmem_ld16(tbase + c0, *reinterpret_cast<uint32_t(*)[16]>(v));
                ptx::tmem_ld16(tbase + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
                ptx::tmem_ld_wait();
                float o[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(v[i]);
                if (a.bias) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 b4 = __ldg(reinterpret_cast<const float4*>(a.bias + c0) + i);
                        o[4 * i] = __fadd_rn(o[4 * i], b4.x);
                        o[4 * i + 1] = __fadd_rn(o[4 * i + 1], b4.y);
                        o[4 * i + 2] = __fadd_rn(o[4 * i + 2], b4.z);
                        o[4 * i + 3] = __fadd_rn(o[4 * i + 3], b4.w);
                    }
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) key[i] = order_key(o[i]);
                if (store) {
                    // lane = row: through shared memory, then 8 lanes per row segment
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *reinterpret_cast<float4*>(xp + lane * 36 + 4 * i) =
                            make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int rr = j * 4 + (lane >> 3), cc = (lane & 7) * 4;
                        const float4 w = *reinterpret_cast<const float4*>(xp + rr * 36 + cc);
                        if (t_warp + rr < a.T) *reinterpret_cast<float4*>(a.logits + (t_warp + rr) * a.ld + c0 + cc) = w;
                    }
                }
            };
            // (1)
            uint32_t cm[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) cm[j] = 0u;
#pragma unroll 1
            for (int c0 = 0; c0 < kRfE; c0 += 32) {
                uint32_t key[32];
                chunk(c0, true, key);
#pragma unroll
                for (int j = 0; j < 16; ++j) cm[j] = max(cm[j], max(key[j], key[j + 16]));
            }
            reset();
#pragma unroll
            for (int j = 0; j < 16; ++j) insert(cm[j], 0);
            uint32_t tau = lk[0];
#pragma unroll
            for (int j = 1; j < kRfMaxK; ++j) tau = min(tau, lk[j]);
            if (!row_ok) tau = 0xFFFFFFFFu;  // rows past T select nothing
            // (2)
            uint2* cand = reinterpret_cast<uint2*>(smem) + r;  // entry j at cand[j * kRfM]
            int n = 0;
#pragma unroll 1
            for (int c0 = 0; c0 < kRfE; c0 += 32) {
                uint32_t key[32];
                chunk(c0, false, key);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    // without branches: every key goes to the next free slot (the spare slot once
                    // the list is full), which only advances for a key >= tau
                    const bool take = key[i] >= tau && tau != 0xFFFFFFFFu;
                    cand[(n < kRfCand ? n : kRfCand) * kRfM] = make_uint2(key[i], static_cast<uint32_t>(c0 + i));
                    n += take ? 1 : 0;
                }
            }
            // (3)
            reset();
            const bool over = n > kRfCand;
            if (!__any_sync(0xFFFFFFFFu, over)) {
#pragma unroll 1
                for (int j = 0; j < n; ++j) {
                    const uint2 c = cand[j * kRfM];
                    insert(c.x, static_cast<int>(c.y));
                }
            } else {
#pragma unroll 1
                for (int c0 = 0; c0 < kRfE; c0 += 32) {
                    uint32_t key[32];
                    chunk(c0, false, key);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (key[i] >= tau && tau != 0xFFFFFFFFu) insert(key[i], c0 + i);
                }
            }
            if (row_ok) {
                // gate logit in column 512 (no bias), the shared gate, the renormalised weights
                lrow[kRfE] = gate;
                if (a.shared_g) a.shared_g[t] = 1.0f / (1.0f + expf(-gate));
                const float l0 = key_value(lk[0]);
                float p[kRfMaxK];
                float sum = 0.0f;
#pragma unroll
                for (int j = 0; j < kRfMaxK; ++j) {
                    p[j] = j < k ? expf(key_value(lk[j]) - l0) : 0.0f;
                    sum += p[j];
                }
#pragma unroll
                for (int j = 0; j < kRfMaxK; ++j)
                    if (j < k) {
                        a.topk_ids[t * k + j] = li[j];
                        a.topk_w[t * k + j] = p[j] / sum;
                    }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (tid == 0 && a.amax_slots) {
        uint32_t m = 0;
#pragma unroll
        for (int w = 0; w < kRfEpiWarps; ++w) m = max(m, st.amax_w[w]);
        a.amax_slots[tb] = m;
    }
    if (warp == 1) {
        __syncwarp();
        ptx::tmem_dealloc(tmem, 512);
    }
    ptx::griddep_launch_dependents();  // this CTA's outputs are written
}

}  // namespace

bool router_topk_fits(int H, int E, int k)
{
    return E == kRfE && H % kRfBK == 0 && H >= kRfBK && H <= kRfMaxH && k >= 1 && k <= kRfMaxK;
}

cudaError_t launch_router_topk(const uint16_t* x, int T, int H, int E, int k, const uint16_t* w_router, const float* bias,
                               float* logits, int ld, int32_t* topk_ids, float* topk_w, float* shared_g,
                               uint32_t* amax_slots, int32_t* zero, int n_zero, int* status, cudaStream_t stream)
{
    if (T <= 0) return cudaSuccess;
    if (!router_topk_fits(H, E, k) || ld < E + 1 || ld % 4 != 0) return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_router_topk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(rf_smem(kRfMaxH)));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    CUtensorMap tx, tw;
    const uint64_t dx[2] = {static_cast<uint64_t>(H), static_cast<uint64_t>(T)};
    const uint64_t sx[1] = {static_cast<uint64_t>(H) * 2};
    const uint32_t bx[2] = {kRfBK, kRfM};
    // router rows 0..511 (row 512, the shared gate, is summed on the CUDA cores), boxes of 256 rows
    const uint64_t dw[2] = {static_cast<uint64_t>(H), static_cast<uint64_t>(kRfE)};
    const uint32_t bw[2] = {kRfBK, 256};
    if (encode_tmap_bf16(&tx, x, 2, dx, sx, bx, 128) != CUDA_SUCCESS ||
        encode_tmap_bf16(&tw, w_router, 2, dw, sx, bw, 128) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    RfArgs a{T, H, k, w_router + static_cast<int64_t>(E) * H, bias, logits, ld, topk_ids, topk_w, shared_g, amax_slots,
             zero, n_zero, status};
    const int n_tb = (T + kRfM - 1) / kRfM;
    return launch_pdl(k_router_topk, dim3(n_tb), dim3(kRfThreads), rf_smem(H), stream, tx, tw, a);
}

}  // namespace moe
