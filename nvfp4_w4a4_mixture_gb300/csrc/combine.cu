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

// ---- streaming variant for many tokens (y in assignment order): one CTA per SM walks tokens
// blockIdx.x, blockIdx.x + gridDim.x, ...; a producer thread bulk-copies each token's k routed rows
// of y (contiguous), its shared-expert row and its residual row into one of kStreamBufs shared-memory
// buffers, and eight warps combine a buffered token (thread per 8 columns, the same fixed-order FP32
// sums as k_combine) while the next tokens' rows are in flight. Every wait is bounded.
constexpr int kStreamBufs = 4;
constexpr int kStreamWarps = 8;
constexpr int kStreamThreads = 32 * (kStreamWarps + 1);
constexpr size_t kStreamSmem = 200 * 1024;

__device__ __forceinline__ void axpy8_smem(float (&acc)[8], float w, const uint16_t* row, int c)
{
    axpy8(acc, w, *reinterpret_cast<const uint4*>(row + c));
}

__global__ void __launch_bounds__(kStreamThreads, 1)
    k_combine_stream(const uint16_t* __restrict__ y, const float* __restrict__ topk_w, const float* __restrict__ shared_g,
                     int T, int k, int H, const uint16_t* __restrict__ residual, uint16_t* __restrict__ out,
                     int* status)
{
    extern __shared__ __align__(128) uint8_t csm[];
    __shared__ __align__(8) uint64_t full[kStreamBufs], empty[kStreamBufs];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nrows = k + 1 + (residual ? 1 : 0);                  // routed rows, shared row, residual
    const size_t row_bytes = static_cast<size_t>(H) * 2;
    const size_t buf_bytes = (nrows * row_bytes + 127) & ~size_t(127);
    if (tid == 0) {
        for (int b = 0; b < kStreamBufs; ++b) {
            ptx::mbar_init(&full[b], 1);
            ptx::mbar_init(&empty[b], kStreamWarps);
        }
        ptx::fence_mbar_init();
    }
    __syncthreads();
    ptx::griddep_wait();  // y comes from the launch before this one
    if (warp == kStreamWarps) {
        if (lane == 0) {
            uint32_t i = 0;
            for (int t = blockIdx.x; t < T; t += gridDim.x, ++i) {
                const int b = i % kStreamBufs;
                const uint32_t ph = (i / kStreamBufs) & 1;
                if (!ptx::mbar_wait(&empty[b], ph ^ 1)) { record_status(status, kDevTimeoutCombine); break; }
                uint8_t* buf = csm + b * buf_bytes;
                ptx::mbar_arrive_expect_tx(&full[b], static_cast<uint32_t>(nrows * row_bytes));
                ptx::bulk_load(buf, y + static_cast<int64_t>(t) * k * H, static_cast<uint32_t>(k * row_bytes), &full[b]);
                ptx::bulk_load(buf + k * row_bytes, y + (static_cast<int64_t>(T) * k + t) * H, static_cast<uint32_t>(row_bytes),
                               &full[b]);
                if (residual)
                    ptx::bulk_load(buf + (k + 1) * row_bytes, residual + static_cast<int64_t>(t) * H,
                                   static_cast<uint32_t>(row_bytes), &full[b]);
            }
            if (!ptx::ring_drain(full, kStreamBufs, i)) record_status(status, kDevTimeoutCombine);
        }
    } else {
        int i = 0;
        for (int t = blockIdx.x; t < T; t += gridDim.x, ++i) {
            const int b = i % kStreamBufs;
            const uint32_t ph = (i / kStreamBufs) & 1;
            const float g = shared_g ? __ldg(shared_g + t) : 0.0f;
            if (!ptx::mbar_wait(&full[b], ph)) { record_status(status, kDevTimeoutCombine); break; }
            const uint16_t* buf = reinterpret_cast<const uint16_t*>(csm + b * buf_bytes);
            const int64_t tk = static_cast<int64_t>(t) * k;
            for (int c = tid * 8; c < H; c += kStreamWarps * 32 * 8) {
                float acc[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
                for (int j = 0; j < k; ++j) axpy8_smem(acc, __ldg(topk_w + tk + j), buf + static_cast<int64_t>(j) * H, c);
                if (shared_g) axpy8_smem(acc, g, buf + static_cast<int64_t>(k) * H, c);
                if (residual) axpy8_smem(acc, 1.0f, buf + static_cast<int64_t>(k + 1) * H, c);
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) o[q] = pack_bf16x2(acc[2 * q], acc[2 * q + 1]);
                *reinterpret_cast<uint4*>(out + static_cast<int64_t>(t) * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&empty[b]);
        }
    }
    ptx::griddep_launch_dependents();
}

cudaError_t launch_combine(const uint16_t* y, const float* topk_w, const float* shared_g, const int32_t* src_perm, int T,
                           int k, int H, const uint16_t* residual, uint16_t* out, int* status, cudaStream_t stream)
{
    if (T <= 0) return cudaSuccess;
    const size_t stream_buf = (static_cast<size_t>(k + 2) * H * 2 + 127) & ~size_t(127);
    if (!src_perm && T >= 1024 && kStreamBufs * stream_buf <= kStreamSmem) {
        static bool attr_set = false;
        if (!attr_set) {
            cudaError_t e = cudaFuncSetAttribute(k_combine_stream, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(kStreamSmem));
            if (e != cudaSuccess) return e;
            attr_set = true;
        }
        const int sms = device_sm_count();
        return launch_pdl(k_combine_stream, dim3(T < sms ? T : sms), dim3(kStreamThreads), kStreamBufs * stream_buf, stream, y,
                          topk_w, shared_g, T, k, H, residual, out, status);
    }
    const int threads = T >= 256 ? kCombineThreadsLarge : kCombineThreadsSmall;
    dim3 grid(T, (H + threads * 8 - 1) / (threads * 8));
    return launch_pdl(k_combine, grid, dim3(threads), 0, stream, y, topk_w, shared_g, src_perm, T, k, H, residual, out);
}

}  // namespace moe
