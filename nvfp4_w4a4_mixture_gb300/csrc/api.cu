// api.cu -- the C ABI of libmoe_nvfp4 (include/moe_nvfp4.h): argument validation on the host,
// workspace layout, and the launch sequence of the layer forward.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <string>

#include "../../include/moe_nvfp4.h"

#include "kernels.cuh"

namespace moe {

namespace {

thread_local std::string g_detail;
constexpr int kLayerStageEvents = 6;

moe_status_t fail(moe_status_t s, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_detail = buf;
    return s;
}

moe_status_t cuda_fail(cudaError_t e, const char* what)
{
    return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

moe_status_t check_device()
{
    static int ok = -1;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (ok < 0) {
        int dev = 0, major = 0, minor = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return fail(MOE_ERR_UNSUPPORTED_DEVICE, "no CUDA device");
        }
        ok = (major == 10 && minor == 3) ? 1 : 0;
        if (!ok) return fail(MOE_ERR_UNSUPPORTED_DEVICE, "device is sm_%d%d, this library is built for sm_103a", major, minor);
    }
    return ok ? MOE_OK : fail(MOE_ERR_UNSUPPORTED_DEVICE, "device is not sm_103");
}

struct WsLayout {
    size_t hdr, amax_slots, topk_ids, topk_w, shared_g, logits, x_codes, x_sf, offsets, perm_src, src_perm, row_token,
        hist, h_codes, h_sf, ready, y, total;
};
// per-CTA maxima of |x|: the layer quantizer's (layer_amax_slots(SM count) of them, far below this on
// any device this library runs on) or the fused router's (one per 128 tokens: up to 524,288 tokens)
constexpr int kMaxAmaxSlots = 4096;

WsLayout ws_layout(int64_t H, int64_t E, int64_t k, int64_t I, int64_t T)
{
    WsLayout L{};
    size_t off = 0;
    auto take = [&](int64_t bytes) {
        const size_t o = off;
        off += (static_cast<size_t>(bytes < 0 ? 0 : bytes) + 255) & ~size_t(255);
        return o;
    };
    const int64_t n = T * k, P = T * k + T;
    L.hdr = take(sizeof(WsHeader));
    L.amax_slots = take(kMaxAmaxSlots * 4);  // per-CTA maxima of |x| (quantizer or fused router)
    L.topk_ids = take(n * 4);
    L.topk_w = take(n * 4);
    L.shared_g = take(T * 4);
    L.logits = take(T * router_tc_ld(static_cast<int>(E)) * 4);  // rows router_tc_ld(E) >= E + 1 floats apart
    L.x_codes = take(T * H / 2);
    L.x_sf = take(T * H / 16);
    L.offsets = take((E + 2) * 4);
    L.perm_src = take(n * 4);
    L.src_perm = take(n * 4);
    L.row_token = take(P * 4);
    L.hist = take((perm_chunks(n) + 1) * E * 4);  // per-chunk counts + per-expert totals
    // token blocks of the expert GEMMs: at most ceil(P / 32) + E + 1 (32-row blocks in the smallest schedule)
    const int64_t nblk = (P + 31) / 32 + E + 1;
    L.h_codes = take(P * I / 2);
    L.h_sf = take(nblk * (I / 64) * 512);  // h block scales in token-block tiles
    L.ready = take((nblk + 1) * 4);  // + the expert GEMMs' tile counter
    L.y = take(P * H * 2);
    L.total = off;
    return L;
}

// moe_layer_forward_host: x (and the residual) from page-locked host memory into the staging
// buffers, 16 bytes per thread (n16 = bytes / 16 of each); the previous launch may still read them
__global__ void k_stage_in(const uint4* __restrict__ x, uint4* __restrict__ xd, const uint4* __restrict__ r,
                           uint4* __restrict__ rd, int64_t n16)
{
    ptx::griddep_wait();
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        xd[i] = x[i];
        if (r) rd[i] = r[i];
    }
    ptx::griddep_launch_dependents();
}

// moe_set_wait_test_hook: the two test fields of a workspace header, written in stream order
__global__ void k_set_wait_hook(WsHeader* hdr, unsigned wait_us, int ready_extra)
{
    hdr->test_wait_us = wait_us;
    hdr->test_ready_extra = ready_extra;
}

// one device staging buffer of moe_layer_forward_host: T x H bf16, 256-byte aligned
size_t host_stage_bytes(int64_t H, int64_t T) { return (static_cast<size_t>(T * H * 2) + 255) & ~size_t(255); }

moe_status_t check_layer_shape(int H, int E, int k, int I)
{
    if (H < 128 || H > 8192 || H % 128) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "H=%d not a multiple of 128 in [128, 8192]", H);
    if (I < 128 || I > 8192 || I % 128) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "I=%d not a multiple of 128 in [128, 8192]", I);
    if (E < 1 || E > 1024) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "E=%d outside [1, 1024]", E);
    if (k < 1 || k > 32 || k > E) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "k=%d outside [1, min(E=%d, 32)]", k, E);
    return MOE_OK;
}

moe_status_t check_ws(const void* ws, size_t ws_bytes, size_t need)
{
    if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
    if (!aligned(ws, 256)) return fail(MOE_ERR_MISALIGNED, "workspace %p not 256-byte aligned", ws);
    if (ws_bytes < need) return fail(MOE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", ws_bytes, need);
    return MOE_OK;
}

#define MOE_TRY(x)                              \
    do {                                        \
        moe_status_t s_ = (x);                  \
        if (s_ != MOE_OK) return s_;            \
    } while (0)

#define MOE_CUDA(x, what)                       \
    do {                                        \
        cudaError_t e_ = (x);                   \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

}  // namespace

void set_last_error_detail(const char* msg) { g_detail = msg ? msg : ""; }

int device_sm_count()
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

CUresult encode_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                             uint32_t box_outer)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = tmap_encoder();
    if (!fn) return CUDA_ERROR_NOT_FOUND;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

bool gemm_permute_enabled()
{
    // on unless MOE_NVFP4_GEMM_PERMUTE=0
    static const bool on = [] {
        const char* v = std::getenv("MOE_NVFP4_GEMM_PERMUTE");
        return !(v && v[0] == '0');
    }();
    return on;
}

bool pdl_enabled()
{
    // On unless MOE_NVFP4_PDL=0. Each CTA of the front half and of the expert GEMMs allows the next
    // launch only when its own work is done, so the next kernel's launch and prologue overlap the
    // previous one's tail (triggered at the start instead, the early CTAs of the next launch held
    // SMs and a decode step was 4-5 us slower than plain stream order).
    static const bool on = [] {
        const char* v = std::getenv("MOE_NVFP4_PDL");
        return !(v && v[0] == '0');
    }();
    return on;
}

CUresult encode_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                          const uint32_t* box, int swizzle_bytes)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = tmap_encoder();
    if (!fn || rank < 1 || rank > 5) return CUDA_ERROR_NOT_FOUND;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    const CUtensorMapSwizzle sw = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                  : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                        : CU_TENSOR_MAP_SWIZZLE_NONE;
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, st, b, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_tmap_3d_u8(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                           uint32_t box1)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = tmap_encoder();
    if (!fn) return CUDA_ERROR_NOT_FOUND;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0, d0 * d1};
    cuuint32_t box[3] = {box0, box1, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status_t s)
{
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE: unsupported shape";
        case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL: workspace too small";
        case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED: misaligned pointer";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: CUDA error";
        case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT: a device-side wait ran out";
        case MOE_ERR_UNSUPPORTED_DEVICE: return "MOE_ERR_UNSUPPORTED_DEVICE: not an sm_103 device";
    }
    return "unknown moe_status_t";
}

const char* moe_last_error_detail(void) { return g_detail.c_str(); }

size_t moe_workspace_bytes(int H, int E, int k, int I, int T)
{
    if (H < 0 || E < 0 || k < 0 || I < 0 || T < 0) return 0;
    return ws_layout(H, E, k, I, T).total;
}

size_t moe_workspace_bytes_host(int H, int E, int k, int I, int T)
{
    if (H < 0 || E < 0 || k < 0 || I < 0 || T < 0) return 0;
    return ws_layout(H, E, k, I, T).total + 3 * host_stage_bytes(H, T);
}

moe_status_t moe_read_device_status(void* ws, moe_stream_t stream)
{
    if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MOE_CUDA(cudaStreamSynchronize(s), "cudaStreamSynchronize");
    int status = 0;
    MOE_CUDA(cudaMemcpy(&status, ws, sizeof(int), cudaMemcpyDeviceToHost), "read status");
    MOE_CUDA(cudaMemset(ws, 0, sizeof(int)), "clear status");
    if (status & kDevTimeoutGemm) return fail(MOE_ERR_DEVICE_TIMEOUT, "device status 0x%x: grouped GEMM wait timed out", status);
    if (status & kDevTimeoutRouter) return fail(MOE_ERR_DEVICE_TIMEOUT, "device status 0x%x: router wait timed out", status);
    if (status & kDevTimeoutCombine) return fail(MOE_ERR_DEVICE_TIMEOUT, "device status 0x%x: combine wait timed out", status);
    if (status & kDevBadExpertId) return fail(MOE_ERR_INVALID_ARG, "device status 0x%x: expert id outside [0, E)", status);
    return MOE_OK;
}

static moe_status_t quantize_common(const void* x, bool f32, int64_t rows, int64_t K, const float* s_in, uint8_t* codes,
                                    uint8_t* sf, float* s_out, void* ws, size_t ws_bytes, moe_stream_t stream)
{
    if (rows < 0 || K <= 0 || K % 16) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "rows=%lld K=%lld: K must be a positive multiple of 16", (long long)rows, (long long)K);
    if (!x || !codes || !sf || !s_out) return fail(MOE_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned(x, 16) || !aligned(codes, 8) || !aligned(s_out, 4) || (s_in && !aligned(s_in, 4)))
        return fail(MOE_ERR_MISALIGNED, "x must be 16-byte, codes 8-byte aligned");
    MOE_TRY(check_ws(ws, ws_bytes, sizeof(WsHeader)));
    MOE_TRY(check_device());
    WsHeader* hdr = static_cast<WsHeader*>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int sms = device_sm_count();
    cudaError_t e = f32 ? launch_quantize_f32(static_cast<const float*>(x), rows, K, s_in, codes, sf, s_out, &hdr->amax_bits, sms, s)
                        : launch_quantize(static_cast<const uint16_t*>(x), rows, K, s_in, codes, sf, s_out, &hdr->amax_bits, sms, s);
    MOE_CUDA(e, "quantize launch");
    return MOE_OK;
}

moe_status_t moe_quantize_nvfp4(const uint16_t* x, int64_t rows, int64_t K, const float* s_in, uint8_t* codes,
                                uint8_t* sf, float* s_out, void* ws, size_t ws_bytes, moe_stream_t stream)
{
    return quantize_common(x, false, rows, K, s_in, codes, sf, s_out, ws, ws_bytes, stream);
}

moe_status_t moe_quantize_nvfp4_f32(const float* x, int64_t rows, int64_t K, const float* s_in, uint8_t* codes,
                                    uint8_t* sf, float* s_out, void* ws, size_t ws_bytes, moe_stream_t stream)
{
    return quantize_common(x, true, rows, K, s_in, codes, sf, s_out, ws, ws_bytes, stream);
}

// Router logits into the workspace: tensor cores above kRouterTcMinT tokens (rows router_tc_ld(E)
// apart), else the CUDA-core kernel with its fixed summation order (rows E + 1 apart).
constexpr int kRouterTcMinT = 64;
// From this many tokens (E = 512, k <= 16) routing runs as one launch that also takes x's maximum
// (k_router_topk: one CTA per 128 tokens holds all 512 logits of its rows), and the activation
// encoder follows it.
constexpr int kFusedRouteMinT = 12288;

static bool fused_route_for(int T, int H, int E, int k)
{
    return T >= kFusedRouteMinT && router_topk_fits(H, E, k);
}

// How moe_layer_forward runs a batch of T tokens: which front half, whether the expert GEMMs
// build the permutation themselves, their tile schedule and token-block height, and the row
// stride of the logits it leaves in the workspace.
struct LayerPlan {
    bool one_launch_front;  // quantise + route (+ permute) in one launch (small batches)
    bool gemm_permutes;     // the expert GEMMs rank the ids in shared memory (offsets etc. not stored)
    bool fused_route;       // routing (with x's maximum) in one launch before the activation encoder
    int sched;              // GemmSchedule of the expert-GEMM launch
    int block_rows;         // token rows per block of that schedule (h's scale tiles)
    int logits_ld;          // floats between two tokens' logits in the workspace
    int n_ready;            // token-block counters of the expert GEMMs
};

static LayerPlan layer_plan(int H, int E, int k, int I, int T, int sms)
{
    LayerPlan p{};
    const int64_t P = static_cast<int64_t>(T) * k + T;
    p.n_ready = static_cast<int>((P + 31) / 32 + E + 1);
    p.one_launch_front = front_fits(T, H, E, k);
    // small batches on wide-narrow tiles: the front half stops at the top-k and every CTA of the
    // expert GEMMs builds the permutation from the ids in its own shared memory (off the front
    // half's single-CTA tail)
    p.gemm_permutes = p.one_launch_front && T <= kRouteMaxT && static_cast<int64_t>(T) * k <= kRouteMaxAssign &&
                      (2 * I) % 256 == 0 && H % 256 == 0 && gemm_permute_enabled();
    // 256-row weight tiles when H allows (half the MMAs and scale copies per weight byte); else
    // weights on the MMA's M side for few rows per expert (decode), 128 x 128 tiles otherwise
    // (token-block units once there are enough of them to keep every SM busy to the end)
    const bool wide = (2 * I) % 256 == 0 && H % 256 == 0;
    const bool small = static_cast<int64_t>(T) * k <= 16LL * E;
    p.sched = wide ? (T <= 32 ? kSchedWideNarrow : gemm_rows_pays(P, sms) ? kSchedWideRows : kSchedWide)
                   : small ? kSchedWeightsOnM : kSchedActOnM;
    p.block_rows = gemm_schedule_rows(p.sched);
    p.fused_route = !p.one_launch_front && fused_route_for(T, H, E, k) && router_topk_slots(T) <= kMaxAmaxSlots;
    p.logits_ld = (!p.one_launch_front && T > kRouterTcMinT) ? router_tc_ld(E) : E + 1;
    return p;
}
cudaError_t route_logits(const uint16_t* x, int T, const moe_layer_t* L, float* logits, WsHeader* hdr, cudaStream_t s)
{
    if (T > kRouterTcMinT)
        return launch_router_logits_tc(x, T, L->H, L->E, L->w_router, L->logit_bias, logits, router_tc_ld(L->E), &hdr->status, s);
    return launch_router_logits(x, T, L->H, L->E, L->w_router, L->logit_bias, logits, s);
}

moe_status_t moe_route_topk(const uint16_t* x, int T, const moe_layer_t* L, int32_t* topk_ids, float* topk_w,
                            float* shared_g, float* logits_out, void* ws, size_t ws_bytes, moe_stream_t stream)
{
    if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    MOE_TRY(check_layer_shape(L->H, L->E, L->k, L->I));
    if (T < 0) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "T=%d < 0", T);
    if (T == 0) return MOE_OK;  // an empty batch: nothing is read or written, the pointers may be NULL
    if (!x || !L->w_router || !topk_ids || !topk_w) return fail(MOE_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned(x, 16) || !aligned(L->w_router, 16) || (L->logit_bias && !aligned(L->logit_bias, 16)))
        return fail(MOE_ERR_MISALIGNED, "x, w_router and logit_bias must be 16-byte aligned");
    const WsLayout W = ws_layout(L->H, L->E, L->k, L->I, T);
    const int ld = router_tc_ld(L->E);
    MOE_TRY(check_ws(ws, ws_bytes, W.logits + static_cast<size_t>(T) * ld * 4));
    MOE_TRY(check_device());
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* logits = reinterpret_cast<float*>(static_cast<char*>(ws) + W.logits);
    if (fused_route_for(T, L->H, L->E, L->k)) {
        MOE_CUDA(launch_router_topk(x, T, L->H, L->E, L->k, L->w_router, L->logit_bias, logits, ld, topk_ids, topk_w,
                                    shared_g, nullptr, nullptr, 0, &reinterpret_cast<WsHeader*>(ws)->status, s),
                 "router launch");
        if (logits_out)
            MOE_CUDA(cudaMemcpy2DAsync(logits_out, static_cast<size_t>(L->E) * 4, logits, static_cast<size_t>(ld) * 4,
                                       static_cast<size_t>(L->E) * 4, static_cast<size_t>(T), cudaMemcpyDeviceToDevice, s),
                     "logits copy");
        return MOE_OK;
    }
    MOE_CUDA(route_logits(x, T, L, logits, reinterpret_cast<WsHeader*>(ws), s), "router launch");
    MOE_CUDA(launch_topk(logits, T > kRouterTcMinT ? ld : L->E + 1, T, L->E, L->k, topk_ids, topk_w, shared_g, logits_out, s),
             "top-k launch");
    return MOE_OK;
}

moe_status_t moe_permute(const int32_t* topk_ids, int T, int k, int E, int with_shared, int32_t* expert_offsets,
                         int32_t* perm_src, int32_t* src_perm, int32_t* row_token, void* ws, size_t ws_bytes,
                         moe_stream_t stream)
{
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E)
        return fail(MOE_ERR_UNSUPPORTED_SHAPE, "T=%d k=%d E=%d outside the supported range", T, k, E);
    if (!topk_ids || !expert_offsets || !perm_src || !src_perm) return fail(MOE_ERR_INVALID_ARG, "NULL tensor pointer");
    const size_t need = 256 + static_cast<size_t>(perm_chunks(static_cast<int64_t>(T) * k) + 1) * E * 4;
    MOE_TRY(check_ws(ws, ws_bytes, need));
    MOE_TRY(check_device());
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsHeader* hdr = static_cast<WsHeader*>(ws);
    int32_t* hist = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + 256);
    MOE_CUDA(launch_permute(topk_ids, T, k, E, with_shared ? 1 : 0, expert_offsets, perm_src, src_perm, row_token, hist,
                            &hdr->perm_ticket, &hdr->status, s),
             "permute launch");
    return MOE_OK;
}

moe_status_t moe_prepack_nvfp4(const uint8_t* codes, const uint8_t* sf, int G, int N, int K, int gate_up_interleave,
                               uint8_t* codes_out, uint8_t* sf_out, moe_stream_t stream)
{
    if (G < 1 || N < 128 || N % 128 || K < 64 || K % 64)
        return fail(MOE_ERR_UNSUPPORTED_SHAPE, "G=%d N=%d K=%d: N must be a multiple of 128 and K of 64", G, N, K);
    if (!codes || !sf || !codes_out || !sf_out) return fail(MOE_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned(codes, 16) || !aligned(codes_out, 16) || !aligned(sf, 4) || !aligned(sf_out, 16))
        return fail(MOE_ERR_MISALIGNED, "codes 16-byte, sf 4-byte, sf_out 16-byte alignment required");
    MOE_TRY(check_device());
    MOE_CUDA(launch_prepack(codes, sf, G, N, K, gate_up_interleave ? 1 : 0, codes_out, sf_out,
                            static_cast<cudaStream_t>(stream)),
             "prepack launch");
    return MOE_OK;
}

static moe_status_t check_bank(const moe_nvfp4_bank_t* b, const char* name)
{
    if (!b || !b->codes || !b->sf || !b->gscale) return fail(MOE_ERR_INVALID_ARG, "bank %s has a NULL pointer", name);
    if (!aligned(b->codes, 16) || !aligned(b->sf, 16) || !aligned(b->gscale, 4))
        return fail(MOE_ERR_MISALIGNED, "bank %s: codes and sf must be 16-byte aligned", name);
    return MOE_OK;
}

moe_status_t moe_grouped_gemm_nvfp4(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_scale,
                                    int a_scale_per_group, const int32_t* a_row_index, const int32_t* group_offsets,
                                    int G, int64_t p_max, const moe_nvfp4_bank_t* b, int N, int K, int gate_up,
                                    int epilogue, const float* epi_scale, void* out, uint8_t* out_sf, void* ws,
                                    size_t ws_bytes, moe_stream_t stream)
{
    if (G < 1 || G > kGemmMaxG) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "G=%d outside [1, %d]", G, kGemmMaxG);
    if (N < 128 || N % 128 || K < 64 || K % 64 || K > 16384)
        return fail(MOE_ERR_UNSUPPORTED_SHAPE, "N=%d K=%d: N must be a multiple of 128, K of 64 (<= 16384)", N, K);
    if (p_max < 0) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "p_max=%lld < 0", (long long)p_max);
    constexpr int kSchedBits = MOE_GEMM_SCHED_ACT_ON_M | MOE_GEMM_SCHED_WEIGHTS_ON_M | MOE_GEMM_SCHED_WIDE |
                               MOE_GEMM_SCHED_WIDE_ROWS | MOE_GEMM_SCHED_WEIGHTS_RESIDENT;
    const int sched_bits = epilogue & kSchedBits;
    if (sched_bits & (sched_bits - 1)) return fail(MOE_ERR_INVALID_ARG, "epilogue=0x%x: pick one schedule flag", epilogue);
    const int schedule = sched_bits == MOE_GEMM_SCHED_ACT_ON_M      ? kSchedActOnM
                         : sched_bits == MOE_GEMM_SCHED_WEIGHTS_ON_M ? kSchedWeightsOnM
                         : sched_bits == MOE_GEMM_SCHED_WIDE         ? kSchedWide
                         : sched_bits == MOE_GEMM_SCHED_WIDE_ROWS    ? kSchedWideRows
                         : sched_bits == MOE_GEMM_SCHED_WEIGHTS_RESIDENT ? kSchedWeightsResident
                                                                     : kSchedAuto;
    epilogue &= ~kSchedBits;
    if (epilogue < MOE_EPI_F32 || epilogue > MOE_EPI_SWIGLU_NVFP4) return fail(MOE_ERR_INVALID_ARG, "epilogue=%d", epilogue);
    if (epilogue == MOE_EPI_SWIGLU_NVFP4 && (!gate_up || !epi_scale || !out_sf))
        return fail(MOE_ERR_INVALID_ARG, "the SwiGLU epilogue needs a gate/up bank, epi_scale and out_sf");
    if (!a_codes || !a_sf || !a_scale || !group_offsets || !out) return fail(MOE_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned(a_codes, 16) || !aligned(a_sf, 4) || !aligned(out, 16) || (out_sf && !aligned(out_sf, 4)))
        return fail(MOE_ERR_MISALIGNED, "a_codes / out must be 16-byte, a_sf / out_sf 4-byte aligned");
    MOE_TRY(check_bank(b, "b"));
    MOE_TRY(check_ws(ws, ws_bytes, sizeof(WsHeader)));
    MOE_TRY(check_device());
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsHeader* hdr = static_cast<WsHeader*>(ws);
    GemmArgs ga{};
    GemmProblem& P = ga.p[0];
    P.a_codes = a_codes;
    P.a_sf = a_sf;
    P.a_scale = a_scale;
    P.a_scale_per_group = a_scale_per_group ? 1 : 0;
    P.a_row = a_row_index;
    P.b_codes = b->codes;
    P.b_sf = b->sf;
    P.b_scale = b->gscale;
    P.gate_up = gate_up ? 1 : 0;
    P.N = N;
    P.K = K;
    P.epilogue = epilogue;
    P.epi_scale = epi_scale;
    P.out = out;
    P.out_sf = out_sf;
    ga.nphase = 1;
    ga.offsets = group_offsets;
    ga.G = G;
    ga.status = &hdr->status;
    ga.tile_counter = &hdr->gemm_tiles;
    MOE_CUDA(cudaMemsetAsync(&hdr->gemm_tiles, 0, sizeof(int32_t), s), "clear tile counter");
    MOE_CUDA(launch_grouped_gemm(ga, p_max, schedule, device_sm_count(), s), "grouped GEMM launch");
    return MOE_OK;
}

moe_status_t moe_combine(const uint16_t* y, const float* topk_w, const float* shared_g, const int32_t* src_perm, int T,
                         int k, int H, const uint16_t* residual, uint16_t* out, moe_stream_t stream)
{
    if (T < 0 || k < 1 || k > 32 || H < 8 || H % 8) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "T=%d k=%d H=%d", T, k, H);
    if (T == 0) return MOE_OK;  // an empty batch: nothing is read or written, the pointers may be NULL
    if (!y || !topk_w || !src_perm || !out) return fail(MOE_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned(y, 16) || !aligned(out, 16) || (residual && !aligned(residual, 16)))
        return fail(MOE_ERR_MISALIGNED, "y, out and residual must be 16-byte aligned");
    MOE_TRY(check_device());
    MOE_CUDA(launch_combine(y, topk_w, shared_g, src_perm, T, k, H, residual, out, nullptr, static_cast<cudaStream_t>(stream)),
             "combine launch");
    return MOE_OK;
}

moe_status_t moe_layer_forward_profiled(const moe_layer_t* L, const uint16_t* x, int T, const uint16_t* residual,
                                        uint16_t* out, void* ws, size_t ws_bytes, moe_stream_t stream,
                                        void* const* events, int n_events)
{
    if (n_events != 0 && n_events != kLayerStageEvents)
        return fail(MOE_ERR_INVALID_ARG, "n_events=%d: pass 0 or %d events", n_events, kLayerStageEvents);
    if (n_events && !events) return fail(MOE_ERR_INVALID_ARG, "events is NULL");
    for (int i = 0; i < n_events; ++i)
        if (!events[i]) return fail(MOE_ERR_INVALID_ARG, "events[%d] is NULL", i);
    if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    const int H = L->H, E = L->E, k = L->k, I = L->I;
    MOE_TRY(check_layer_shape(H, E, k, I));
    if (T < 0) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "T=%d < 0", T);
    if (T == 0 && n_events == 0) return MOE_OK;  // an empty batch: nothing is read or written, the pointers may be NULL
    if (!x || !out || !L->w_router || !L->s_mid) return fail(MOE_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned(x, 16) || !aligned(out, 16) || (residual && !aligned(residual, 16)) || !aligned(L->w_router, 16) ||
        (L->logit_bias && !aligned(L->logit_bias, 16)))
        return fail(MOE_ERR_MISALIGNED, "x, out, residual, w_router and logit_bias must be 16-byte aligned");
    if (x == out) return fail(MOE_ERR_INVALID_ARG, "out must not alias x");
    MOE_TRY(check_bank(&L->w_gate_up, "w_gate_up"));
    MOE_TRY(check_bank(&L->w_down, "w_down"));
    const WsLayout W = ws_layout(H, E, k, I, T);
    MOE_TRY(check_ws(ws, ws_bytes, W.total));
    MOE_TRY(check_device());
    if (T == 0) {  // an empty batch with events: each is recorded, so every stage reads zero time
        for (int i = 0; i < n_events; ++i)
            MOE_CUDA(cudaEventRecord(static_cast<cudaEvent_t>(events[i]), static_cast<cudaStream_t>(stream)), "event record");
        return MOE_OK;
    }

    char* base = static_cast<char*>(ws);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(base + W.hdr);
    auto P32 = [&](size_t o) { return reinterpret_cast<int32_t*>(base + o); };
    auto PF = [&](size_t o) { return reinterpret_cast<float*>(base + o); };
    auto P8 = [&](size_t o) { return reinterpret_cast<uint8_t*>(base + o); };
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int sms = device_sm_count();
    const int64_t P = static_cast<int64_t>(T) * k + T;
    auto mark = [&](int i) -> cudaError_t {
        return n_events ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) : cudaSuccess;
    };

    const LayerPlan plan = layer_plan(H, E, k, I, T, sms);
    // token-block counters of the expert GEMMs, then their tile counter (all zeroed before the launch)
    const int n_ready = plan.n_ready;
    const bool one_launch_front = plan.one_launch_front;
    const bool gemm_permutes = plan.gemm_permutes;
    MOE_CUDA(mark(0), "event record");
    if (one_launch_front) {
        // small batch: quantisation, router, top-k, shared gate and permutation in one launch
        MOE_CUDA(launch_front(x, T, H, E, k, L->w_router, L->logit_bias, PF(W.logits), P8(W.x_codes), P8(W.x_sf),
                              &hdr->s_x, P32(W.topk_ids), PF(W.topk_w), PF(W.shared_g),
                              gemm_permutes ? nullptr : P32(W.offsets),
                              P32(W.perm_src), P32(W.src_perm), P32(W.row_token), &hdr->ticket, P32(W.ready),
                              n_ready + 1, s),
                 "front");
        MOE_CUDA(mark(1), "event record");
        MOE_CUDA(mark(2), "event record");
    } else if (plan.fused_route) {
        // routing first: logits, top-k, weights, shared gate and each CTA's max |x| in one launch
        // (which also zeroes the expert GEMMs' counters), then the W4A4 encoding of x with the
        // tensor scale reduced from those maxima
        uint32_t* slots = reinterpret_cast<uint32_t*>(base + W.amax_slots);
        MOE_CUDA(launch_router_topk(x, T, H, E, k, L->w_router, L->logit_bias, PF(W.logits), plan.logits_ld,
                                    P32(W.topk_ids), PF(W.topk_w), PF(W.shared_g), slots, P32(W.ready), n_ready + 1,
                                    &hdr->status, s),
                 "router");
        MOE_CUDA(mark(1), "event record");
        MOE_CUDA(launch_quantize_from_slots(x, T, H, P8(W.x_codes), P8(W.x_sf), &hdr->s_x, slots, router_topk_slots(T),
                                            sms, s),
                 "quantize");
        MOE_CUDA(mark(2), "event record");
        MOE_CUDA(launch_permute(P32(W.topk_ids), T, k, E, 1, P32(W.offsets), P32(W.perm_src), P32(W.src_perm),
                                P32(W.row_token), P32(W.hist), &hdr->perm_ticket, &hdr->status, s),
                 "permute");
    } else {
        // W4A4: quantize the layer input once per token (dynamic tensor scale); the quantizer's first
        // launch also zeroes the counters of the expert GEMMs (no memset between two kernels: each
        // launch overlaps the one before it, programmatic dependent launch)
        if (layer_amax_slots(sms) > kMaxAmaxSlots) return fail(MOE_ERR_UNSUPPORTED_DEVICE, "%d SMs: too many", sms);
        MOE_CUDA(launch_quantize_layer(x, T, H, P8(W.x_codes), P8(W.x_sf), &hdr->s_x,
                                       reinterpret_cast<uint32_t*>(base + W.amax_slots), P32(W.ready), n_ready + 1, sms, s),
                 "quantize");
        MOE_CUDA(mark(1), "event record");
        // router, softmax, top-k, shared gate
        MOE_CUDA(route_logits(x, T, L, PF(W.logits), hdr, s), "router");
        MOE_CUDA(launch_topk(PF(W.logits), plan.logits_ld, T, E, k, P32(W.topk_ids),
                             PF(W.topk_w), PF(W.shared_g), nullptr, s),
                 "top-k");
        MOE_CUDA(mark(2), "event record");
        // permutation by expert id, the shared expert appended as group E
        MOE_CUDA(launch_permute(P32(W.topk_ids), T, k, E, 1, P32(W.offsets), P32(W.perm_src), P32(W.src_perm),
                                P32(W.row_token), P32(W.hist), &hdr->perm_ticket, &hdr->status, s),
                 "permute");
    }
    MOE_CUDA(mark(3), "event record");
    // expert GEMMs in one launch: gate/up with the fused SwiGLU + NVFP4 requantisation of h,
    // then down (bf16 rows in permuted order); a down tile waits for its token block's h
    GemmArgs ga{};
    GemmProblem& g1 = ga.p[0];
    g1.a_codes = P8(W.x_codes);
    g1.a_sf = P8(W.x_sf);
    g1.a_scale = &hdr->s_x;
    g1.a_row = P32(W.row_token);
    g1.b_codes = L->w_gate_up.codes;
    g1.b_sf = L->w_gate_up.sf;
    g1.b_scale = L->w_gate_up.gscale;
    g1.gate_up = 1;
    g1.N = 2 * I;
    g1.K = H;
    g1.epilogue = kEpiSwiGLU;
    g1.epi_scale = L->s_mid;
    g1.out = P8(W.h_codes);
    g1.out_sf = P8(W.h_sf);
    g1.out_sf_tiled = 1;
    GemmProblem& g2 = ga.p[1];
    g2.a_codes = P8(W.h_codes);
    g2.a_sf = P8(W.h_sf);
    g2.a_sf_tiled = 1;
    g2.a_scale = L->s_mid;
    g2.a_scale_per_group = 1;
    g2.b_codes = L->w_down.codes;
    g2.b_sf = L->w_down.sf;
    g2.b_scale = L->w_down.gscale;
    g2.N = H;
    g2.K = I;
    g2.epilogue = kEpiBF16;
    g2.out = base + W.y;
    g2.out_row = P32(W.perm_src);  // routed rows back in assignment order t*k + j; shared rows stay
    g2.out_row_n = static_cast<int>(static_cast<int64_t>(T) * k);
    ga.nphase = 2;
    ga.offsets = P32(W.offsets);
    ga.G = E + 1;
    ga.ready = P32(W.ready);
    ga.tile_counter = P32(W.ready) + n_ready;
    ga.status = &hdr->status;
    ga.hooks = hdr;
    if (gemm_permutes) ga.route = GemmRoute{P32(W.topk_ids), T, k, E};
    MOE_CUDA(launch_grouped_gemm(ga, P, plan.sched, sms, s), "expert GEMMs");
    MOE_CUDA(mark(4), "event record");
    // weighted combine (+ residual)
    MOE_CUDA(launch_combine(reinterpret_cast<const uint16_t*>(base + W.y), PF(W.topk_w), PF(W.shared_g), nullptr, T, k,
                            H, residual, out, &hdr->status, s),
             "combine");
    MOE_CUDA(mark(5), "event record");
    return MOE_OK;
}

moe_status_t moe_set_wait_test_hook(void* ws, unsigned wait_limit_us, int ready_extra, moe_stream_t stream)
{
    if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
    if (!aligned(ws, 256)) return fail(MOE_ERR_MISALIGNED, "workspace %p not 256-byte aligned", ws);
    if (ready_extra < 0) return fail(MOE_ERR_INVALID_ARG, "ready_extra=%d < 0", ready_extra);
    MOE_TRY(check_device());
    k_set_wait_hook<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<WsHeader*>(ws), wait_limit_us, ready_extra);
    MOE_CUDA(cudaGetLastError(), "test hook launch");
    return MOE_OK;
}

moe_status_t moe_layer_workspace_view(const moe_layer_t* L, int T, moe_layer_view_t* view)
{
    if (!L || !view) return fail(MOE_ERR_INVALID_ARG, "layer or view is NULL");
    MOE_TRY(check_layer_shape(L->H, L->E, L->k, L->I));
    if (T < 0) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "T=%d < 0", T);
    MOE_TRY(check_device());
    const WsLayout W = ws_layout(L->H, L->E, L->k, L->I, T);
    const LayerPlan plan = layer_plan(L->H, L->E, L->k, L->I, T, device_sm_count());
    moe_layer_view_t v{};
    v.bytes = static_cast<int64_t>(W.total);
    v.x_scale = static_cast<int64_t>(W.hdr + offsetof(WsHeader, s_x));
    v.x_codes = static_cast<int64_t>(W.x_codes);
    v.x_sf = static_cast<int64_t>(W.x_sf);
    v.logits = static_cast<int64_t>(W.logits);
    v.logits_ld = plan.logits_ld;
    v.topk_ids = static_cast<int64_t>(W.topk_ids);
    v.topk_w = static_cast<int64_t>(W.topk_w);
    v.shared_g = static_cast<int64_t>(W.shared_g);
    v.permutation_in_workspace = plan.gemm_permutes ? 0 : 1;
    v.expert_offsets = static_cast<int64_t>(W.offsets);
    v.perm_src = static_cast<int64_t>(W.perm_src);
    v.src_perm = static_cast<int64_t>(W.src_perm);
    v.row_token = static_cast<int64_t>(W.row_token);
    v.h_codes = static_cast<int64_t>(W.h_codes);
    v.h_sf = static_cast<int64_t>(W.h_sf);
    v.h_block_rows = plan.block_rows;
    v.y = static_cast<int64_t>(W.y);
    v.route_first = plan.fused_route ? 1 : 0;
    *view = v;
    return MOE_OK;
}

moe_status_t moe_layer_forward(const moe_layer_t* L, const uint16_t* x, int T, const uint16_t* residual, uint16_t* out,
                               void* ws, size_t ws_bytes, moe_stream_t stream)
{
    return moe_layer_forward_profiled(L, x, T, residual, out, ws, ws_bytes, stream, nullptr, 0);
}

moe_status_t moe_layer_forward_host(const moe_layer_t* L, const uint16_t* x, int T, const uint16_t* residual,
                                    uint16_t* out, void* ws, size_t ws_bytes, moe_stream_t stream)
{
    if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    MOE_TRY(check_layer_shape(L->H, L->E, L->k, L->I));
    if (T < 0) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "T=%d < 0", T);
    if (T == 0) return MOE_OK;  // an empty batch: nothing is read or written, the pointers may be NULL
    if (!x || !out) return fail(MOE_ERR_INVALID_ARG, "NULL tensor pointer");
    const size_t bytes = static_cast<size_t>(T) * L->H * 2;
    const char *xb = reinterpret_cast<const char*>(x), *ob = reinterpret_cast<const char*>(out);
    const char* rb = reinterpret_cast<const char*>(residual);
    if (bytes && ((ob < xb + bytes && xb < ob + bytes) || (rb && ob < rb + bytes && rb < ob + bytes)))
        return fail(MOE_ERR_INVALID_ARG, "out overlaps x or residual");
    const WsLayout W = ws_layout(L->H, L->E, L->k, L->I, T);
    const size_t stage = host_stage_bytes(L->H, T);
    MOE_TRY(check_ws(ws, ws_bytes, W.total + 3 * stage));
    MOE_TRY(check_device());
    const void* host_ptrs[3] = {x, residual, out};
    const char* names[3] = {"x", "residual", "out"};
    const uint16_t* in_dev[2] = {nullptr, nullptr};  // page-locked x / residual, as the device addresses them
    uint16_t* out_dev = nullptr;                      // page-locked out, as the device addresses it
    for (int i = 0; i < 3; ++i) {
        if (!host_ptrs[i]) continue;
        cudaPointerAttributes at{};
        if (cudaPointerGetAttributes(&at, host_ptrs[i]) != cudaSuccess) {
            cudaGetLastError();
            return fail(MOE_ERR_INVALID_ARG, "%s: not a valid pointer", names[i]);
        }
        if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged)
            return fail(MOE_ERR_INVALID_ARG, "%s is device memory; moe_layer_forward_host takes host buffers", names[i]);
        const bool mapped = at.type == cudaMemoryTypeHost && at.devicePointer && aligned(at.devicePointer, 16);
        if (mapped && i < 2) in_dev[i] = static_cast<const uint16_t*>(at.devicePointer);
        if (mapped && i == 2) out_dev = static_cast<uint16_t*>(at.devicePointer);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(ws);
    uint16_t* xd = reinterpret_cast<uint16_t*>(base + W.total);
    uint16_t* od = reinterpret_cast<uint16_t*>(base + W.total + stage);
    uint16_t* rd = residual ? reinterpret_cast<uint16_t*>(base + W.total + 2 * stage) : nullptr;
    // page-locked inputs come in through one small kernel reading them over the host link (launched
    // like the layer's kernels, so the front half's prologue overlaps it); others by copy
    if (in_dev[0] && (!residual || in_dev[1])) {
        const int64_t n16 = static_cast<int64_t>(bytes / 16);
        const int grid = static_cast<int>(std::min<int64_t>((n16 + 255) / 256, 4LL * device_sm_count()));
        MOE_CUDA(launch_pdl(k_stage_in, dim3(grid), dim3(256), 0, s, reinterpret_cast<const uint4*>(in_dev[0]),
                            reinterpret_cast<uint4*>(xd), reinterpret_cast<const uint4*>(in_dev[1]),
                            reinterpret_cast<uint4*>(rd), n16),
                 "stage the inputs in");
    } else {
        MOE_CUDA(cudaMemcpyAsync(xd, x, bytes, cudaMemcpyHostToDevice, s), "copy x to the device");
        if (rd) MOE_CUDA(cudaMemcpyAsync(rd, residual, bytes, cudaMemcpyHostToDevice, s), "copy residual to the device");
    }
    // page-locked output: the combine writes it directly over the host link (no separate copy);
    // otherwise the result is staged on the device and copied back
    MOE_TRY(moe_layer_forward_profiled(L, xd, T, rd, out_dev ? out_dev : od, ws, W.total, stream, nullptr, 0));
    if (!out_dev) MOE_CUDA(cudaMemcpyAsync(out, od, bytes, cudaMemcpyDeviceToHost, s), "copy the result to the host");
    return MOE_OK;
}

}  // extern "C"
