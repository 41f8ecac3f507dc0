// kernels.cuh -- internal launchers of libmoe_nvfp4 (not part of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "common.cuh"

namespace moe {

// ---- quantize.cu
cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t K, const float* s_in, uint8_t* codes, uint8_t* sf,
                            float* s_out, unsigned* amax_scratch, int sms, cudaStream_t stream,
                            bool amax_zeroed = false);
cudaError_t launch_quantize_f32(const float* x, int64_t rows, int64_t K, const float* s_in, uint8_t* codes,
                                uint8_t* sf, float* s_out, unsigned* amax_scratch, int sms, cudaStream_t stream);
// The layer's quantizer (dynamic tensor scale): per-CTA maxima in slots (layer_amax_slots(sms) of
// them), no atomics; it also zeroes zero[0 .. n_zero) for the launches that follow.
int layer_amax_slots(int sms);
// The encoding pass alone, its tensor scale reduced from n_slots maxima written by an earlier launch.
cudaError_t launch_quantize_from_slots(const uint16_t* x, int64_t rows, int64_t K, uint8_t* codes, uint8_t* sf,
                                       float* s_out, const uint32_t* slots, int n_slots, int sms, cudaStream_t stream);
cudaError_t launch_quantize_layer(const uint16_t* x, int64_t rows, int64_t K, uint8_t* codes, uint8_t* sf, float* s_out,
                                  uint32_t* slots, int32_t* zero, int n_zero, int sms, cudaStream_t stream);

// ---- router.cu
// logits: FP32 [T][E+1] (column E = shared-gate logit, no bias).
cudaError_t launch_router_logits(const uint16_t* x, int T, int H, int E, const uint16_t* w_router, const float* bias,
                                 float* logits, cudaStream_t stream);
// logits rows ld floats apart (ld >= E + 1)
cudaError_t launch_topk(const float* logits, int ld, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                        float* shared_g, float* logits_out, cudaStream_t stream);

// ---- router_tc.cu (large batches: router logits on the tensor cores)
// logits: FP32 [T][ld] with ld = router_tc_ld(E) (a multiple of 16; columns E+1.. hold 0);
// H % 64 == 0. A bounded wait that runs out sets kDevTimeoutRouter in *status.
int router_tc_ld(int E);
cudaError_t launch_router_logits_tc(const uint16_t* x, int T, int H, int E, const uint16_t* w_router, const float* bias,
                                    float* logits, int ld, int* status, cudaStream_t stream);

// ---- router_fused.cu (large batches, E = 512: logits, top-k, weights, shared gate and max |x| in
// one launch; one CTA per 128 tokens)
// logits: FP32 [T][ld] (ld >= E + 1, ld % 4 == 0; column E = gate logit). amax_slots (nullable):
// one max |x| per CTA, as float bits, ceil(T / 128) of them. zero (nullable): zero[0 .. n_zero)
// is zeroed after the previous launch completes. A bounded wait that runs out sets kDevTimeoutRouter.
bool router_topk_fits(int H, int E, int k);
inline int router_topk_slots(int T) { return (T + 127) / 128; }
cudaError_t launch_router_topk(const uint16_t* x, int T, int H, int E, int k, const uint16_t* w_router, const float* bias,
                               float* logits, int ld, int32_t* topk_ids, float* topk_w, float* shared_g,
                               uint32_t* amax_slots, int32_t* zero, int n_zero, int* status, cudaStream_t stream);

// ---- permute.cu
constexpr int kPermChunk = 512;  // assignments per chunk (one CTA of the permutation kernels)
inline int64_t perm_chunks(int64_t n) { return n <= 0 ? 1 : (n + kPermChunk - 1) / kPermChunk; }
// offsets: [E+2]; hist: (perm_chunks(n) + 1) * E ints of scratch; ticket: zero between calls.
cudaError_t launch_permute(const int32_t* topk_ids, int T, int k, int E, int with_shared, int32_t* offsets,
                           int32_t* perm_src, int32_t* src_perm, int32_t* row_token, int32_t* hist, unsigned* ticket,
                           int* status, cudaStream_t stream);

// ---- front.cu (small batches: quantize + router + top-k + permute in one launch)
bool front_fits(int T, int H, int E, int k);
cudaError_t launch_front(const uint16_t* x, int T, int H, int E, int k, const uint16_t* w_router, const float* bias,
                         float* logits, uint8_t* xq_codes, uint8_t* xq_sf, float* s_x, int32_t* topk_ids, float* topk_w,
                         float* shared_g, int32_t* offsets, int32_t* perm_src, int32_t* src_perm, int32_t* row_token,
                         unsigned* ticket, int32_t* ready, int n_ready, cudaStream_t stream);

// ---- prepack.cu
cudaError_t launch_prepack(const uint8_t* codes, const uint8_t* sf, int G, int N, int K, int interleave,
                           uint8_t* codes_out, uint8_t* sf_out, cudaStream_t stream);

// ---- grouped_gemm.cu
enum EpiKind : int { kEpiF32 = 0, kEpiBF16 = 1, kEpiSwiGLU = 2 };

// One grouped GEMM over the groups of a launch (see grouped_gemm.cu).
struct GemmProblem {
    const uint8_t* a_codes;   // [*][K/2]
    const uint8_t* a_sf;      // [*][K/16] row-major, or token-block tiles when a_sf_tiled
    const float* a_scale;     // [1] or [G]
    int a_scale_per_group;
    const int32_t* a_row;     // nullable gather index, [P]
    int a_sf_tiled;           // A scales in tiles [token block][K/64][512 B] (written by a SwiGLU phase)
    const uint8_t* b_codes;   // prepacked [G][N][K/2] (described by the tensor map)
    const uint8_t* b_sf;      // prepacked tiles [G][N/128][K/64][512]
    const float* b_scale;     // [G][gate_up ? 2 : 1]
    int gate_up;
    int N, K;
    int epilogue;
    const float* epi_scale;   // [G] static scale of h (SwiGLU epilogue)
    void* out;
    uint8_t* out_sf;          // SwiGLU: h scales, row-major [P][N/32] or tiles when out_sf_tiled
    int out_sf_tiled;
    const int32_t* out_row;   // nullable (FP32 / bf16 epilogues): row p < out_row_n goes to out row
    int out_row_n;            //   out_row[p] (e.g. back to assignment order), rows p >= out_row_n stay
};

// A launch: one problem, or the gate/up problem (phase 0) followed by the down problem (phase 1)
// over the same groups; phase-1 tiles of a token block wait for that block's phase-0 tiles.
// Routing the launch turns into its own permutation (32-row token blocks only): the top-k ids of
// T <= 32 tokens (T * k <= 512), expert E being the shared one. Each CTA builds the group offsets,
// the gate/up gather rows and the down output rows in shared memory; offsets and the a_row / out_row
// indices of the problems are then unused.
struct GemmRoute {
    const int32_t* topk_ids;  // [T][k], null: offsets and row indices come from global memory
    int T, k, E;
};
constexpr int kRouteMaxT = 32, kRouteMaxAssign = 512;

struct GemmArgs {
    GemmProblem p[2];
    int nphase;
    const int32_t* offsets;   // [G+1]
    int G;
    GemmRoute route;
    int32_t* ready;           // [token blocks], zeroed before a two-phase launch
    int32_t* tile_counter;    // tiles handed out beyond the first gridDim.x, zeroed before each launch
    int* status;
    const WsHeader* hooks;    // nullable: the workspace header whose test_* fields the waits read
    int a_tma[2];             // set by the launcher: phase i's activation rows are contiguous and come
                              // as TMA boxes (token-block units with two MMA threads only)
};
constexpr int kGemmMaxG = 1025;
// Tile schedules: activations on the MMA's M side (128-row token blocks x 128 weight rows),
// weights on M (128 weight rows x 32-row token blocks, for small groups), or activations on M with
// 256 weight rows per tile (wide: fewer MMAs and scale copies per weight byte; needs N % 256 == 0,
// else it falls back to activations on M). Auto picks weights-on-M when p_max <= 64.
// Wide-narrow: the wide shape with 32-row token blocks and a fifth stage (groups of few rows).
// Weight-resident units: one 128-row weight block (all of K <= 2048) per CTA in shared memory, up to
// 16 token blocks of its group streamed past it into a double-buffered accumulator.
enum GemmSchedule : int {
    kSchedAuto = 0, kSchedActOnM = 1, kSchedWeightsOnM = 2, kSchedWide = 3, kSchedWideNarrow = 4, kSchedWideRows = 5,
    kSchedWeightsResident = 6
};
bool gemm_wide_fits(const GemmArgs& a);
// whether a launch of p_max rows is large enough for token-block units (kSchedWideRows)
bool gemm_rows_pays(int64_t p_max, int sms);
cudaError_t launch_grouped_gemm(const GemmArgs& a, int64_t p_max, int schedule, int sms, cudaStream_t stream);
int gemm_schedule_rows(int schedule);  // token rows per block of a (resolved) schedule

// ---- combine.cu
// status: nullable device status word (the streaming variant records kDevTimeoutCombine there)
cudaError_t launch_combine(const uint16_t* y, const float* topk_w, const float* shared_g, const int32_t* src_perm, int T,
                           int k, int H, const uint16_t* residual, uint16_t* out, int* status, cudaStream_t stream);

// ---- api.cu
int device_sm_count();

// Launches with programmatic stream serialisation when MOE_NVFP4_PDL=1 (the kernel calls
// ptx::griddep_wait() before it touches anything the previous launch writes or reads; without the
// attribute that call returns at once).
bool pdl_enabled();
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}
void set_last_error_detail(const char* msg);  // text returned by moe_last_error_detail()
CUresult encode_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                             uint32_t box_outer);
CUresult encode_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                          const uint32_t* box, int swizzle_bytes);
CUresult encode_tmap_3d_u8(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                           uint32_t box1);

}  // namespace moe
