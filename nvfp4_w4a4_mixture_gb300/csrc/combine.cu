// combine.cu -- weighted un-permute of the expert outputs with FP32 accumulation.
//
// One CTA per (token, 2048-column slice): the token's k routing slots (row index and weight) are
// staged in shared memory first, then every thread owns 8 consecutive hidden columns and issues
// the 16-byte loads of all k routed rows and the shared row before it accumulates, so the loads of
// one token are in flight together. The sum runs in a fixed order (slots j = 0..k-1, then the
// shared expert, then the residual), each product rounded to FP32 before it is added:
// deterministic.
#include "kernels.cuh"

namespace moe {

constexpr int kCombineThreads = 256;  // x 8 columns = 2048 columns per CTA
constexpr int kMaxK = 32;

__device__ __forceinline__ void axpy8(float (&acc)[8], float w, const uint4& v)
{
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(w, bf16_to_f32(x[i] & 0xFFFFu)));
        acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(w, bf16_to_f32(x[i] >> 16)));
    }
}

__global__ void __launch_bounds__(kCombineThreads)
    k_combine(const uint16_t* __restrict__ y, const float* __restrict__ topk_w, const float* __restrict__ shared_g,
              const int32_t* __restrict__ src_perm, int T, int k, int H, const uint16_t* __restrict__ residual,
              uint16_t* __restrict__ out)
{
    __shared__ int64_t rows_s[kMaxK + 1];
    __shared__ float w_s[kMaxK + 1];
    ptx::griddep_wait();  // y comes from the launch before this one
    ptx::griddep_launch_dependents();
    const int t = blockIdx.x;
    const int64_t tk = static_cast<int64_t>(t) * k;
    if (threadIdx.x < k) {
        rows_s[threadIdx.x] = __ldg(src_perm + tk + threadIdx.x);
        w_s[threadIdx.x] = __ldg(topk_w + tk + threadIdx.x);
    }
    const int nslot = k + (shared_g ? 1 : 0);
    if (shared_g && threadIdx.x == 0) {
        rows_s[k] = static_cast<int64_t>(T) * k + t;
        w_s[k] = __ldg(shared_g + t);
    }
    __syncthreads();
    const int c = (blockIdx.y * kCombineThreads + threadIdx.x) * 8;
    if (c >= H) return;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    int j = 0;
    for (; j + 4 <= nslot; j += 4) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ldg(reinterpret_cast<const uint4*>(y + rows_s[j + u] * H + c));
#pragma unroll
        for (int u = 0; u < 4; ++u) axpy8(acc, w_s[j + u], v[u]);
    }
    for (; j < nslot; ++j) axpy8(acc, w_s[j], __ldg(reinterpret_cast<const uint4*>(y + rows_s[j] * H + c)));
    if (residual) axpy8(acc, 1.0f, __ldg(reinterpret_cast<const uint4*>(residual + static_cast<int64_t>(t) * H + c)));
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = f32_to_bf16(acc[2 * i]) | (f32_to_bf16(acc[2 * i + 1]) << 16);
    *reinterpret_cast<uint4*>(out + static_cast<int64_t>(t) * H + c) = make_uint4(w[0], w[1], w[2], w[3]);
}

cudaError_t launch_combine(const uint16_t* y, const float* topk_w, const float* shared_g, const int32_t* src_perm, int T,
                           int k, int H, const uint16_t* residual, uint16_t* out, cudaStream_t stream)
{
    if (T <= 0) return cudaSuccess;
    dim3 grid(T, (H + kCombineThreads * 8 - 1) / (kCombineThreads * 8));
    return launch_pdl(k_combine, grid, dim3(kCombineThreads), 0, stream, y, topk_w, shared_g, src_perm, T, k, H, residual,
                      out);
}

}  // namespace moe
