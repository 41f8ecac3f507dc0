// combine.cu -- weighted un-permute of the expert outputs with FP32 accumulation.
//
// One warp per token; each lane owns 8 consecutive hidden columns per 256-column step and reads
// 16-byte vectors of the k routed rows and the shared row (512 contiguous bytes per warp and
// row). The sum runs in a fixed order (routed slots j = 0..k-1, shared expert, residual), each
// product rounded to FP32 before it is added, so the result is deterministic.
#include "kernels.cuh"

namespace moe {

__device__ __forceinline__ void axpy8(float (&acc)[8], float w, const uint4& v)
{
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(w, bf16_to_f32(x[i] & 0xFFFFu)));
        acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(w, bf16_to_f32(x[i] >> 16)));
    }
}

__global__ void k_combine(const uint16_t* __restrict__ y, const float* __restrict__ topk_w,
                          const float* __restrict__ shared_g, const int32_t* __restrict__ src_perm, int T, int k, int H,
                          const uint16_t* __restrict__ residual, uint16_t* __restrict__ out)
{
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
    if (t >= T) return;
    const int64_t tk = static_cast<int64_t>(t) * k;
    for (int c = lane * 8; c < H; c += 256) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int j = 0; j < k; ++j) {
            const int64_t p = __ldg(src_perm + tk + j);
            const float w = __ldg(topk_w + tk + j);
            axpy8(acc, w, __ldg(reinterpret_cast<const uint4*>(y + p * H + c)));
        }
        if (shared_g) {
            const int64_t p = static_cast<int64_t>(T) * k + t;
            axpy8(acc, __ldg(shared_g + t), __ldg(reinterpret_cast<const uint4*>(y + p * H + c)));
        }
        if (residual) axpy8(acc, 1.0f, __ldg(reinterpret_cast<const uint4*>(residual + static_cast<int64_t>(t) * H + c)));
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = f32_to_bf16(acc[2 * i]) | (f32_to_bf16(acc[2 * i + 1]) << 16);
        *reinterpret_cast<uint4*>(out + static_cast<int64_t>(t) * H + c) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

cudaError_t launch_combine(const uint16_t* y, const float* topk_w, const float* shared_g, const int32_t* src_perm, int T,
                           int k, int H, const uint16_t* residual, uint16_t* out, cudaStream_t stream)
{
    if (T <= 0) return cudaSuccess;
    const int warps = 8;
    k_combine<<<(T + warps - 1) / warps, warps * 32, 0, stream>>>(y, topk_w, shared_g, src_perm, T, k, H, residual, out);
    return cudaGetLastError();
}

}  // namespace moe
