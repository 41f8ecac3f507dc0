// noalloc.cu -- moe_route_topk_noalloc: the router + top-k call without a caller workspace.
//
// Some callers cannot hand the library device scratch: an application whose device memory is
// owned by another allocator (a serving runtime that budgets every byte and forbids extra
// cudaMalloc calls), or a hot decode loop that must not pay cudaMalloc's implicit device
// synchronisation. For them this entry point keeps the router's logits scratch in a fixed
// array compiled into the library, so it allocates nothing and needs no workspace.
//
// The array lives in device memory of every GPU that loads the library, for the life of the
// process. Host code cannot use the array's name as a device address: the per-device address is
// looked up once with cudaGetSymbolAddress and cached. All calls share the array, so two calls
// that overlap on the GPU (different streams, or different host threads) race on it.
#include <mutex>

#include "../../include/moe_nvfp4.h"
#include "kernels.cuh"

namespace moe {

namespace {

constexpr int kNoallocMaxTokens = 64;
constexpr int kNoallocMaxExperts = 1024;
constexpr size_t kNoallocFloats = static_cast<size_t>(kNoallocMaxTokens) * (kNoallocMaxExperts + 1);

// logits scratch [T][E+1] of the router call (every used element is written before it is read,
// so nothing has to start at zero)
static __device__ __align__(256) float g_route_scratch[kNoallocFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};

moe_status_t noalloc_fail(moe_status_t s, const char* msg)
{
    set_last_error_detail(msg);  // read back with moe_last_error_detail()
    return s;
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_route_topk_noalloc(const uint16_t* x, int T, const moe_layer_t* L, int32_t* topk_ids,
                                               float* topk_w, float* shared_g, float* logits_out, moe_stream_t stream)
{
    // the checks of moe_route_topk, in its order: the layer's shape, the token count, then an empty
    // batch returns before anything is read (its pointers may be NULL), then this call's own limit
    if (!L) return noalloc_fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    if (L->H < 128 || L->H > 8192 || L->H % 128 || L->I < 128 || L->I > 8192 || L->I % 128 || L->E < 1 ||
        L->E > kNoallocMaxExperts || L->k < 1 || L->k > 32 || L->k > L->E)
        return noalloc_fail(MOE_ERR_UNSUPPORTED_SHAPE,
                            "H, I, E or k outside the supported range (H, I multiples of 128 in [128, 8192]; "
                            "1 <= k <= min(E, 32); E <= 1024)");
    if (T < 0) return noalloc_fail(MOE_ERR_UNSUPPORTED_SHAPE, "T < 0");
    if (T == 0) return MOE_OK;
    if (T > kNoallocMaxTokens)
        return noalloc_fail(MOE_ERR_UNSUPPORTED_SHAPE, "T > 64: the no-allocation router holds logits for at most 64 tokens");
    if (!x || !L->w_router || !topk_ids || !topk_w) return noalloc_fail(MOE_ERR_INVALID_ARG, "NULL tensor pointer");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(L->w_router) | reinterpret_cast<uintptr_t>(L->logit_bias)) %
        16)
        return noalloc_fail(MOE_ERR_MISALIGNED, "x, w_router and logit_bias must be 16-byte aligned");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return noalloc_fail(MOE_ERR_CUDA, "no current CUDA device");
    }
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) return noalloc_fail(MOE_ERR_UNSUPPORTED_DEVICE, "device is not sm_103");
    float* scratch = nullptr;
    {
        // first call on this device: look up the device address of the scratch array
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_scratch_ptr[dev]) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) {
                cudaGetLastError();
                return noalloc_fail(MOE_ERR_CUDA, "cudaGetSymbolAddress of the router scratch failed");
            }
            g_scratch_ptr[dev] = static_cast<float*>(p);
        }
        scratch = g_scratch_ptr[dev];
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (launch_router_logits(x, T, L->H, L->E, L->w_router, L->logit_bias, scratch, s) != cudaSuccess ||
        launch_topk(scratch, L->E + 1, T, L->E, L->k, topk_ids, topk_w, shared_g, logits_out, s) != cudaSuccess)
        return noalloc_fail(MOE_ERR_CUDA, "router launch failed");
    return MOE_OK;
}
