// router_tc.cu -- router logits for large batches on the tensor cores:
//   logits[t][e] = sum_h x[t][h] * w_router[e][h] (+ bias[e] for e < E),  e = 0..E (E: shared gate)
// tcgen05.mma kind::f16 with bf16 operands and FP32 accumulation in tensor memory. Every product of
// two bf16 values is exact in FP32; the sums run in the tensor core's order, so the logits differ
// from a sequential FP32 sum by rounding only (the top-k decision is unaffected unless two logits lie
// within that rounding of each other).
//
// One CTA per output tile of 128 tokens x kN router rows (176: three tiles cover E + 1 = 513; for
// fewer tokens 96 or 64, so that more CTAs share the work), adjacent CTAs share the token block. Warp 0 loads 64-column K-slices of both operands by TMA (128-byte
// swizzle) into a 5-deep ring, warp 1 owns tensor memory and issues four K=16 MMAs per slice, warps
// 2-5 read the accumulator (one TMEM lane quarter each) and store FP32 rows of stride ld.
#include "kernels.cuh"

namespace moe {

namespace {

constexpr int kRtM = 128, kRtStages = 5;
constexpr int kRtABytes = kRtM * 128;
constexpr int kRtThreads = 192;
template <int kN>
struct RtShape {
    static constexpr int B_BYTES = kN * 128, STAGE_BYTES = kRtABytes + B_BYTES;
    static_assert(STAGE_BYTES % 1024 == 0 && kN % 16 == 0 && kN <= 256, "tile shape");
};

struct RtTail {
    uint64_t full[kRtStages];
    uint64_t empty[kRtStages];
    uint64_t acc_full;
    uint32_t tmem_base;
    int abort;
};

template <int kN>
constexpr size_t rt_smem()
{
    return 1024 + static_cast<size_t>(kRtStages) * RtShape<kN>::STAGE_BYTES + sizeof(RtTail);
}

template <int kN>
__global__ void __launch_bounds__(kRtThreads, 1)
    k_router_tc(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w, int T, int H,
                int E, const float* __restrict__ bias, float* __restrict__ logits, int ld, int n_ntiles, int* status)
{
    constexpr int kRtN = kN, kRtBBytes = RtShape<kN>::B_BYTES, kRtStageBytes = RtShape<kN>::STAGE_BYTES;
    (void)kRtBBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    RtTail& st = *reinterpret_cast<RtTail*>(smem + kRtStages * kRtStageBytes);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int tb = blockIdx.x / n_ntiles, nt = blockIdx.x % n_ntiles;
    const int n_k = H / 64;

    if (tid == 0) {
        for (int s = 0; s < kRtStages; ++s) {
            ptx::mbar_init(&st.full[s], 1);
            ptx::mbar_init(&st.empty[s], 1);
        }
        ptx::mbar_init(&st.acc_full, 1);
        st.abort = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmap_x);
        ptx::prefetch_tmap(&tmap_w);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&st.tmem_base, 256);
        ptx::tmem_relinquish();
    }
    ptx::griddep_wait();  // x may come from the previous launch
    ptx::griddep_launch_dependents();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = st.tmem_base;
    auto fail = [&]() {
        if (atomicExch(&st.abort, 1) == 0) record_status(status, kDevTimeoutRouter);
    };

    if (warp == 0) {
        if (lane == 0) {
            int s = 0, kt = 0;
            uint32_t ph = 0;
            for (; kt < n_k; ++kt) {
                if (!ptx::mbar_wait(&st.empty[s], ph ^ 1)) { fail(); break; }
                uint8_t* sb = smem + s * kRtStageBytes;
                ptx::mbar_arrive_expect_tx(&st.full[s], kRtStageBytes);
                ptx::tma_load_2d(sb, &tmap_x, &st.full[s], kt * 64, tb * kRtM);
                ptx::tma_load_2d(sb + kRtABytes, &tmap_w, &st.full[s], kt * 64, nt * kRtN);
                if (++s == kRtStages) { s = 0; ph ^= 1; }
            }
            if (!ptx::ring_drain(st.full, kRtStages, kt)) fail();
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_bf16(kRtM, kRtN);
            const uint32_t s0 = ptx::smem_u32(smem);
            const uint64_t da0 = ptx::sdesc_sw128(s0), db0 = ptx::sdesc_sw128(s0 + kRtABytes);
            constexpr uint64_t kStageAdv = kRtStageBytes >> 4, kKAdv = 32 >> 4;  // K=16 bf16 = 32 bytes
            int s = 0;
            uint32_t ph = 0, acc = 0;
            bool ok = true;
            for (int kt = 0; kt < n_k; ++kt) {
                if (!ptx::mbar_wait(&st.full[s], ph)) { fail(); ok = false; break; }
                ptx::tc_fence_after();
                const uint64_t so = static_cast<uint64_t>(s) * kStageAdv;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    ptx::mma_bf16(tmem, da0 + so + kk * kKAdv, db0 + so + kk * kKAdv, idesc, acc);
                    acc = 1;
                }
                ptx::tc_commit(&st.empty[s]);
                if (++s == kRtStages) { s = 0; ph ^= 1; }
            }
            // the accumulator is complete (or, after a timeout, every issued MMA has finished)
            ptx::tc_commit(&st.acc_full);
            (void)ok;
        }
    } else {
        // epilogue: warp w reads TMEM lanes 32 * (w % 4) .. + 31 = token rows of the tile
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const int64_t t = static_cast<int64_t>(tb) * kRtM + r;
        const bool got = ptx::mbar_wait(&st.acc_full, 0);
        if (!got) fail();
        ptx::tc_fence_after();
        if (__all_sync(0xFFFFFFFFu, got) && !*reinterpret_cast<volatile int*>(&st.abort)) {
            const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16);
            float* row = logits + t * ld;
#pragma unroll 1
            for (int c0 = 0; c0 < kRtN; c0 += 16) {
                uint32_t v[16];
                ptx::tmem_ld16(tbase + c0, v);
                ptx::tmem_ld_wait();
                const int e0 = nt * kRtN + c0;
                if (t < T && e0 <= E) {
                    float o[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int e = e0 + i;
                        o[i] = __uint_as_float(v[i]);
                        if (bias && e < E) o[i] = __fadd_rn(o[i], __ldg(bias + e));
                    }
                    if (e0 + 16 <= ld) {  // ld % 16 == 0: the 16 columns are one aligned 64-byte chunk
                        float4* d = reinterpret_cast<float4*>(row + e0);
#pragma unroll
                        for (int i = 0; i < 4; ++i) d[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                    }
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        ptx::tmem_dealloc(tmem, 256);
    }
}

}  // namespace

int router_tc_ld(int E) { return (E + 1 + 15) / 16 * 16; }

template <int kN>
static cudaError_t launch_tc(const uint16_t* x, int T, int H, int E, const uint16_t* w_router, const float* bias,
                             float* logits, int ld, int* status, cudaStream_t stream)
{
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_router_tc<kN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(rt_smem<kN>()));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    CUtensorMap tx, tw;
    if (encode_tmap_2d_bf16(&tx, x, static_cast<uint64_t>(H), static_cast<uint64_t>(T), 64, kRtM) != CUDA_SUCCESS ||
        encode_tmap_2d_bf16(&tw, w_router, static_cast<uint64_t>(H), static_cast<uint64_t>(E + 1), 64, kN) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int n_ntiles = (E + 1 + kN - 1) / kN;
    const int n_tb = (T + kRtM - 1) / kRtM;
    return launch_pdl(k_router_tc<kN>, dim3(n_tb * n_ntiles), dim3(kRtThreads), rt_smem<kN>(), stream, tx, tw, T, H, E, bias,
                      logits, ld, n_ntiles, status);
}

cudaError_t launch_router_logits_tc(const uint16_t* x, int T, int H, int E, const uint16_t* w_router, const float* bias,
                                    float* logits, int ld, int* status, cudaStream_t stream)
{
    if (T <= 0) return cudaSuccess;
    if (H % 64 != 0 || ld % 16 != 0 || ld < E + 1) return cudaErrorInvalidValue;
    // the narrowest tile whose CTAs still fit in one wave (more CTAs share the work, each streaming
    // less); beyond one wave the widest (a partial second wave costs more: 4096 tokens took 37 us
    // with 96-row tiles against 29 us with 176)
    const int n_tb = (T + kRtM - 1) / kRtM, sms = device_sm_count();
    if (n_tb * ((E + 1 + 63) / 64) <= sms) return launch_tc<64>(x, T, H, E, w_router, bias, logits, ld, status, stream);
    if (n_tb * ((E + 1 + 95) / 96) <= sms) return launch_tc<96>(x, T, H, E, w_router, bias, logits, ld, status, stream);
    return launch_tc<176>(x, T, H, E, w_router, bias, logits, ld, status, stream);
}

}  // namespace moe
