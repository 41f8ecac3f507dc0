// combine.cu -- weighted un-permute of the expert outputs with FP32 accumulation.
//
// One CTA per (token, column slice): 64 threads (512 columns) for few tokens, 256 (2048 columns)
// for many; every thread owns 8 consecutive hidden columns. With a src_perm index the token's routed rows are y[src_perm[t*k + j]] (rows in
// permuted order); without one they are y[t*k + j] (the expert GEMM wrote them back in assignment
// order), so no index load precedes the row loads. The shared expert's row is y[T*k + t]. Each
// thread issues the 16-byte loads of up to 16 slots together, then accumulates in a fixed order
// (slots j = 0..k-1, the shared expert, the residual), each product rounded to FP32 before it is
// added: deterministic.
#include "kernels.cuh"

namespace moe {

constexpr int kCombineThreadsSmall = 64;  // x 8 columns = 512 columns per CTA (few tokens: more CTAs)
constexpr int kCombineThreadsLarge = 256;
constexpr int kCombineChunk = 16;    // slots whose rows are loaded together

__device__ __forceinline__ void axpy8(float (&acc)[8], float w, const uint4& v)
{
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(w, bf16_to_f32(x[i] & 0xFFFFu)));
        acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(w, bf16_to_f32(x[i] >> 16)));
    }
}

__global__ void __launch_bounds__(kCombineThreadsLarge)
    k_combine(const uint16_t* __restrict__ y, const float* __restrict__ topk_w, const float* __restrict__ shared_g,
              const int32_t* __restrict__ src_perm, int T, int k, int H, const uint16_t* __restrict__ residual,
              uint16_t* __restrict__ out)
{
    ptx::griddep_wait();  // y comes from the launch before this one
    ptx::griddep_launch_dependents();
    const int t = blockIdx.x;
    const int c = (blockIdx.y * blockDim.x + threadIdx.x) * 8;
    if (c >= H) return;
    const int64_t tk = static_cast<int64_t>(t) * k;
    const int nslot = k + (shared_g ? 1 : 0);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    uint4 res = make_uint4(0, 0, 0, 0);
    if (residual) res = __ldg(reinterpret_cast<const uint4*>(residual + static_cast<int64_t>(t) * H + c));
    for (int j0 = 0; j0 < nslot; j0 += kCombineChunk) {
        uint4 v[kCombineChunk];
        float w[kCombineChunk];
#pragma unroll
        for (int u = 0; u < kCombineChunk; ++u) {
            const int j = j0 + u;
            if (j < nslot) {
                int64_t row;
                if (j < k) {
                    row = src_perm ? static_cast<int64_t>(__ldg(src_perm + tk + j)) : tk + j;
                    w[u] = __ldg(topk_w + tk + j);
                } else {
                    row = static_cast<int64_t>(T) * k + t;
                    w[u] = __ldg(shared_g + t);
                }
                v[u] = __ldg(reinterpret_cast<const uint4*>(y + row * H + c));
            }
        }
#pragma unroll
        for (int u = 0; u < kCombineChunk; ++u)
            if (j0 + u < nslot) axpy8(acc, w[u], v[u]);
    }
    if (residual) axpy8(acc, 1.0f, res);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
    *reinterpret_cast<uint4*>(out + static_cast<int64_t>(t) * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
}

cudaError_t launch_combine(const uint16_t* y, const float* topk_w, const float* shared_g, const int32_t* src_perm, int T,
                           int k, int H, const uint16_t* residual, uint16_t* out, cudaStream_t stream)
{
    if (T <= 0) return cudaSuccess;
    const int threads = T >= 256 ? kCombineThreadsLarge : kCombineThreadsSmall;
    dim3 grid(T, (H + threads * 8 - 1) / (threads * 8));
    return launch_pdl(k_combine, grid, dim3(threads), 0, stream, y, topk_w, shared_g, src_perm, T, k, H, residual, out);
}

}  // namespace moe
