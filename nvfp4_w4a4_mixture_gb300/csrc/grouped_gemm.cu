// grouped_gemm.cu -- block-scaled NVFP4 grouped GEMM on the 5th-generation tensor cores.
//
// One persistent CTA per SM walks a list of 128 x 128 output tiles (group, M-tile, N-tile),
// N-tile fastest so that consecutive CTAs share the same gathered activation rows and the same
// expert's weights stay hot in L2. Warp roles (256 threads):
//   warp 0     B producer: TMA of the expert's weight codes (128 rows x 128 bytes, 128-byte swizzle)
//              and one bulk copy of the matching scale-factor tiles, per K-stage of 256 elements;
//   warp 1     TMEM owner and MMA issuer: per stage, tcgen05.cp of the scale factors into tensor
//              memory, then 4 x tcgen05.mma kind::mxf4nvf4 (M = 128, N = 128, K = 64) into an FP32
//              accumulator in TMEM (two accumulator buffers);
//   warps 2-3  A producers: gather the activation rows of the tile (row index list) with
//              cp.async into the swizzled layout, and their scale factors into tile layout;
//   warps 4-7  epilogue: tcgen05.ld the accumulator (one 32-lane quarter per warp), apply the
//              tensor scales and write FP32 / bf16 rows, or SwiGLU + NVFP4 requantisation.
// Stages are handed over with mbarriers (full: producers -> MMA; empty: MMA commit ->
// producers; acc_full / acc_empty: MMA <-> epilogue). Every wait is bounded (ptx::mbar_wait): on
// timeout the CTA records kDevTimeoutGemm in the status word, stops all roles and frees TMEM.
#include "kernels.cuh"

namespace moe {

namespace {

constexpr int BM = 128, BN = 128;
constexpr int BK_BYTES = 128;                 // one swizzle row = 256 E2M1 values
constexpr int STAGES = 6;
constexpr int THREADS = 256;
constexpr int A_BYTES = BM * BK_BYTES;        // 16 KiB
constexpr int B_BYTES = BN * BK_BYTES;        // 16 KiB
constexpr int SF_BYTES = 4 * 512;             // 4 scale tiles (K = 4 x 64)
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + 2 * SF_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int ACC_COL = 0;                    // accumulators: columns [0, 256), 2 x 128
constexpr int SF_COL = 256;                   // scale factors: 32 columns per stage
constexpr int kNumAProducers = 64;

struct SmemTail {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int32_t tile_off[kGemmMaxG + 1];
};

constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + sizeof(SmemTail);

struct TileInfo {
    int g, nt, row0, rows;
};

__device__ __forceinline__ TileInfo tile_info(const SmemTail& t, const GemmArgs& a, int n_tiles, int L)
{
    const int mtg = L / n_tiles;
    TileInfo ti;
    ti.nt = L - mtg * n_tiles;
    // largest g with tile_off[g] <= mtg (groups with no tiles have tile_off[g] == tile_off[g+1])
    int lo = 0, hi = a.G;  // invariant: tile_off[lo] <= mtg < tile_off[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (t.tile_off[mid] <= mtg) lo = mid; else hi = mid;
    }
    ti.g = lo;
    const int mt = mtg - t.tile_off[lo];
    const int g0 = __ldg(a.offsets + lo), g1 = __ldg(a.offsets + lo + 1);
    ti.row0 = g0 + mt * BM;
    ti.rows = min(BM, g1 - ti.row0);
    return ti;
}

__device__ __forceinline__ void set_abort(SmemTail& t, int* status)
{
    if (atomicExch(&t.abort, 1) == 0) record_status(status, kDevTimeoutGemm);
}

__device__ __forceinline__ bool aborted(const SmemTail& t) { return *reinterpret_cast<const volatile int*>(&t.abort) != 0; }

}  // namespace

__global__ void __launch_bounds__(THREADS, 1)
    k_grouped_gemm_nvf4(const __grid_constant__ CUtensorMap tmap_b, const GemmArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    SmemTail& st = *reinterpret_cast<SmemTail*>(smem + STAGES * STAGE_BYTES);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

    // ---- setup
    for (int i = tid; i <= a.G; i += THREADS) st.tile_off[i] = __ldg(a.tile_off + i);
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&st.full[s], 1 + kNumAProducers);
            ptx::mbar_init(&st.empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&st.acc_full[s], 1);
            ptx::mbar_init(&st.acc_empty[s], 128);
        }
        ptx::mbar_init(&st.drain, 1);
        st.abort = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmap_b);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&st.tmem_base, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = st.tmem_base;

    const int n_tiles = a.N / BN;
    const int total = st.tile_off[a.G] * n_tiles;
    const int k_stages = (a.K + 255) / 256;
    const int k_blocks64 = a.K / 64;
    const int64_t a_ld = a.K / 2, sf_ld = a.K / 16;

    if (warp == 0) {
        // ================================ B producer
        if (lane == 0) {
            uint32_t it = 0;
            for (int L = blockIdx.x; L < total && !aborted(st); L += gridDim.x) {
                const TileInfo ti = tile_info(st, a, n_tiles, L);
                const uint8_t* sf_base =
                    a.b_sf + ((static_cast<int64_t>(ti.g) * (a.N / 128) + ti.nt) * k_blocks64) * 512;
                for (int kt = 0; kt < k_stages; ++kt, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!ptx::mbar_wait(&st.empty[s], ph ^ 1)) { set_abort(st, a.status); break; }
                    uint8_t* sbase = smem + s * STAGE_BYTES;
                    const int nat = min(4, k_blocks64 - kt * 4);
                    ptx::mbar_arrive_expect_tx(&st.full[s], B_BYTES + nat * 512);
                    ptx::tma_load_3d(sbase + A_BYTES, &tmap_b, &st.full[s], kt * BK_BYTES, ti.nt * BN, ti.g);
                    ptx::bulk_load(sbase + A_BYTES + B_BYTES + SF_BYTES, sf_base + static_cast<int64_t>(kt) * 4 * 512,
                                   nat * 512, &st.full[s]);
                }
            }
        }
    } else if (warp == 1) {
        // ================================ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_nvf4(BM, BN);
            uint32_t it = 0, lt = 0;
            for (int L = blockIdx.x; L < total && !aborted(st); L += gridDim.x, ++lt) {
                const uint32_t as = lt & 1, aph = (lt >> 1) & 1;
                if (!ptx::mbar_wait(&st.acc_empty[as], aph ^ 1)) { set_abort(st, a.status); break; }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem + ACC_COL + as * BN;
                for (int kt = 0; kt < k_stages; ++kt, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!ptx::mbar_wait(&st.full[s], ph)) { set_abort(st, a.status); break; }
                    ptx::tc_fence_after();
                    uint8_t* sbase = smem + s * STAGE_BYTES;
                    const uint32_t sa = ptx::smem_u32(sbase), sb = ptx::smem_u32(sbase + A_BYTES);
                    const uint32_t ssfa = ptx::smem_u32(sbase + A_BYTES + B_BYTES);
                    const uint32_t ssfb = ssfa + SF_BYTES;
                    const uint32_t tsfa = tmem + SF_COL + s * 32, tsfb = tsfa + 16;
                    const int nk = min(4, k_blocks64 - kt * 4);
                    for (int kk = 0; kk < nk; ++kk) {
                        ptx::tmem_cp_32x128b_x4(tsfa + kk * 4, ptx::sdesc_sf(ssfa + kk * 512));
                        ptx::tmem_cp_32x128b_x4(tsfb + kk * 4, ptx::sdesc_sf(ssfb + kk * 512));
                        ptx::mma_nvf4(d_tmem, ptx::sdesc_sw128(sa + kk * 32), ptx::sdesc_sw128(sb + kk * 32), idesc,
                                      tsfa + kk * 4, tsfb + kk * 4, (kt | kk) != 0);
                    }
                    ptx::tc_commit(&st.empty[s]);
                }
                if (aborted(st)) break;
                ptx::tc_commit(&st.acc_full[as]);
            }
            // wait until every issued tensor-core operation has finished before TMEM is freed
            ptx::tc_commit(&st.drain);
            if (!ptx::mbar_wait(&st.drain, 0)) set_abort(st, a.status);
        }
    } else if (warp < 4) {
        // ================================ A producers (gather)
        const int pt = tid - 64;  // 0..63, rows pt and pt + 64
        uint32_t it = 0;
        int pending_stage = -1;
        for (int L = blockIdx.x; L < total && !aborted(st); L += gridDim.x) {
            const TileInfo ti = tile_info(st, a, n_tiles, L);
            int64_t src[2];
            bool valid[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = pt + h * 64;
                valid[h] = r < ti.rows;
                const int64_t p = ti.row0 + r;
                src[h] = valid[h] ? (a.a_row ? static_cast<int64_t>(__ldg(a.a_row + p)) : p) : 0;
            }
            bool ok = true;
            for (int kt = 0; kt < k_stages; ++kt, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1;
                if (!ptx::mbar_wait(&st.empty[s], ph ^ 1)) { set_abort(st, a.status); ok = false; break; }
                uint8_t* sA = smem + s * STAGE_BYTES;
                uint8_t* sSFA = sA + A_BYTES + B_BYTES;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = pt + h * 64;
                    const uint8_t* row = a.a_codes + src[h] * a_ld;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int64_t kb = static_cast<int64_t>(kt) * BK_BYTES + c * 16;
                        const bool v = valid[h] && kb < a_ld;
                        ptx::cp_async_16(sA + r * 128 + ((c ^ (r & 7)) * 16), v ? row + kb : a.a_codes, v);
                    }
                    const uint8_t* srow = a.a_sf + src[h] * sf_ld;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int64_t kb = static_cast<int64_t>(kt) * 16 + j * 4;
                        const bool v = valid[h] && kb < sf_ld;
                        ptx::cp_async_4(sSFA + j * 512 + (r % 32) * 16 + (r / 32) * 4, v ? srow + kb : a.a_sf, v);
                    }
                }
                ptx::cp_async_commit();
                // the previous stage's copies have landed: publish it
                ptx::cp_async_wait<1>();
                if (pending_stage >= 0) {
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive(&st.full[pending_stage]);
                }
                pending_stage = s;
            }
            if (!ok) break;
        }
        ptx::cp_async_wait<0>();
        if (pending_stage >= 0) {
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&st.full[pending_stage]);
        }
    } else {
        // ================================ epilogue
        const int q = warp - 4;            // TMEM lane quarter
        const int r = q * 32 + lane;       // tile row
        uint32_t lt = 0;
        for (int L = blockIdx.x; L < total && !aborted(st); L += gridDim.x, ++lt) {
            const TileInfo ti = tile_info(st, a, n_tiles, L);
            const uint32_t as = lt & 1, aph = (lt >> 1) & 1;
            const bool got = ptx::mbar_wait(&st.acc_full[as], aph);
            __syncwarp();  // tcgen05.ld below is warp-collective
            if (!__all_sync(0xFFFFFFFFu, got)) { set_abort(st, a.status); break; }
            ptx::tc_fence_after();
            const uint32_t taddr = tmem + ACC_COL + as * BN + (static_cast<uint32_t>(q * 32) << 16);
            const bool valid = r < ti.rows;
            const int64_t p = ti.row0 + r;
            const float sa = __ldg(a.a_scale + (a.a_scale_per_group ? ti.g : 0));
            if (a.epilogue == kEpiSwiGLU) {
                const float sg = sa * __ldg(a.b_scale + 2 * ti.g), su = sa * __ldg(a.b_scale + 2 * ti.g + 1);
                const float S = __ldg(a.epi_scale + ti.g);
                const float six_s = __fmul_rn(6.0f, S);
                const int I = a.N / 2;
                uint8_t* hrow = static_cast<uint8_t*>(a.out) + p * (I / 2) + ti.nt * 32;
                uint8_t* srow = a.out_sf + p * (I / 16) + ti.nt * 4;
                uint32_t sfw = 0;
                uint32_t cw[8];
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
                    uint32_t g[16], u[16];
                    ptx::tmem_ld16(taddr + blk * 16, g);
                    ptx::tmem_ld16(taddr + 64 + blk * 16, u);
                    ptx::tmem_ld_wait();
                    float h[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float gv = __uint_as_float(g[i]) * sg;
                        const float uv = __uint_as_float(u[i]) * su;
                        h[i] = gv / (1.0f + __expf(-gv)) * uv;
                    }
                    uint32_t lo, hi;
                    sfw |= nvfp4_encode16(h, S, six_s, lo, hi) << (8 * blk);
                    cw[2 * blk] = lo;
                    cw[2 * blk + 1] = hi;
                }
                if (valid) {
                    reinterpret_cast<uint4*>(hrow)[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
                    reinterpret_cast<uint4*>(hrow)[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
                    *reinterpret_cast<uint32_t*>(srow) = sfw;
                }
            } else {
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 16) {
                    uint32_t v[16];
                    ptx::tmem_ld16(taddr + c0, v);
                    ptx::tmem_ld_wait();
                    int col;
                    float sb;
                    if (a.gate_up) {
                        const int half = c0 >= 64;
                        col = (half ? a.N / 2 : 0) + ti.nt * 64 + (c0 & 63);
                        sb = __ldg(a.b_scale + 2 * ti.g + half);
                    } else {
                        col = ti.nt * BN + c0;
                        sb = __ldg(a.b_scale + ti.g);
                    }
                    const float s = sa * sb;
                    if (valid) {
                        if (a.epilogue == kEpiF32) {
                            float4* o = reinterpret_cast<float4*>(static_cast<float*>(a.out) + p * a.N + col);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                o[i] = make_float4(__uint_as_float(v[4 * i]) * s, __uint_as_float(v[4 * i + 1]) * s,
                                                   __uint_as_float(v[4 * i + 2]) * s, __uint_as_float(v[4 * i + 3]) * s);
                        } else {
                            uint32_t w[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                w[i] = f32_to_bf16(__uint_as_float(v[2 * i]) * s) |
                                       (f32_to_bf16(__uint_as_float(v[2 * i + 1]) * s) << 16);
                            uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + p * a.N + col);
                            o[0] = make_uint4(w[0], w[1], w[2], w[3]);
                            o[1] = make_uint4(w[4], w[5], w[6], w[7]);
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&st.acc_empty[as]);
        }
    }

    // ---- teardown
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

size_t grouped_gemm_smem_bytes() { return kSmemBytes; }

cudaError_t launch_grouped_gemm(const GemmArgs& a, int64_t p_max, int sms, cudaStream_t stream)
{
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_grouped_gemm_nvf4, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    CUtensorMap tmap;
    CUresult cr = encode_tmap_3d_u8(&tmap, a.b_codes, static_cast<uint64_t>(a.K / 2), static_cast<uint64_t>(a.N),
                                    static_cast<uint64_t>(a.G), BK_BYTES, BN);
    if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
    const int64_t mtiles_ub = (p_max + BM - 1) / BM + a.G;
    const int64_t tiles_ub = mtiles_ub * (a.N / BN);
    const int grid = static_cast<int>(tiles_ub < sms ? (tiles_ub < 1 ? 1 : tiles_ub) : sms);
    k_grouped_gemm_nvf4<<<grid, THREADS, kSmemBytes, stream>>>(tmap, a);
    return cudaGetLastError();
}

}  // namespace moe
