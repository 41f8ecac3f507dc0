// quantize.cu -- NVFP4 encoding of activations (W4A4) and weights.
//
// Two passes over the tensor: a max-reduction for the tensor scale (skipped with a static
// scale), then one thread per 16-element block; a tensor of at most 4096 blocks is done by a
// single CTA in one launch. Loads are 16-byte vectors, a warp reads 1 KiB of
// bf16 contiguously and writes 256 contiguous bytes of codes and 32 bytes of block scales.
#include "kernels.cuh"

namespace moe {

__device__ __forceinline__ void load16(const uint16_t* p, float (&v)[16])
{
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = bf16_to_f32(w[i] & 0xFFFFu);
        v[2 * i + 1] = bf16_to_f32(w[i] >> 16);
    }
}

__device__ __forceinline__ void load16(const float* p, float (&v)[16])
{
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p) + i);
        v[4 * i] = a.x;
        v[4 * i + 1] = a.y;
        v[4 * i + 2] = a.z;
        v[4 * i + 3] = a.w;
    }
}

__device__ __forceinline__ uint32_t abs_bits_max(uint32_t m, float f) { return max(m, __float_as_uint(fabsf(f))); }

// amax(|x|) over nblocks 16-element blocks, as the bit pattern of a non-negative float.
template <typename Tin>
__global__ void k_amax(const Tin* __restrict__ x, int64_t nblocks, unsigned* __restrict__ amax_bits)
{
    ptx::griddep_wait();  // x may come from the launch before this one
    uint32_t m = 0;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblocks; b += stride) {
        float v[16];
        load16(x + b * 16, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) m = abs_bits_max(m, v[i]);
    }
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0 && m != 0) atomicMax(amax_bits, m);
    ptx::griddep_launch_dependents();
}

template <typename Tin>
__global__ void k_quantize(const Tin* __restrict__ x, int64_t nblocks, const float* __restrict__ s_static,
                           const unsigned* __restrict__ amax_bits, uint8_t* __restrict__ codes,
                           uint8_t* __restrict__ sf, float* __restrict__ s_out)
{
    ptx::griddep_wait();  // the tensor max comes from the launch before this one
    float S;
    if (s_static) {
        S = *s_static;
    } else {
        const float amax = __uint_as_float(*amax_bits);
        S = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
    }
    if (s_out && blockIdx.x == 0 && threadIdx.x == 0) *s_out = S;
    const float six_s = __fmul_rn(6.0f, S);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblocks; b += stride) {
        float v[16];
        load16(x + b * 16, v);
        uint32_t lo, hi;
        const uint32_t s = nvfp4_encode16(v, S, six_s, lo, hi);
        *reinterpret_cast<uint2*>(codes + b * 8) = make_uint2(lo, hi);
        sf[b] = static_cast<uint8_t>(s);
    }
    ptx::griddep_launch_dependents();
}

// The layer's quantizer (layer inputs of more than kSmallBlocks blocks): no global atomic and nothing
// to zero between calls. Pass 1: every CTA writes the maximum of its share to its own slot; it also
// zeroes the layer's counters that later launches of the call rely on. Pass 2: every CTA reduces the
// slots (the same order-free maximum) and encodes its share.
constexpr int kLayerAmaxThreads = 256;

__global__ void __launch_bounds__(kLayerAmaxThreads)
    k_amax_slots(const uint16_t* __restrict__ x, int64_t nblocks, uint32_t* __restrict__ slots,
                 int32_t* __restrict__ zero, int n_zero)
{
    ptx::griddep_wait();  // x may come from the launch before this one (which may still use zero[])
    __shared__ uint32_t wmax[kLayerAmaxThreads / 32];
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t i = tid; i < n_zero; i += stride) zero[i] = 0;
    uint32_t m = 0;
    int64_t b = tid;
    // four blocks' loads in flight per thread, then the maxima
    for (; b + 3 * stride < nblocks; b += 4 * stride) {
        float v[4][16];
#pragma unroll
        for (int u = 0; u < 4; ++u) load16(x + (b + u * stride) * 16, v[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int i = 0; i < 16; ++i) m = abs_bits_max(m, v[u][i]);
    }
    for (; b < nblocks; b += stride) {
        float v[16];
        load16(x + b * 16, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) m = abs_bits_max(m, v[i]);
    }
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        uint32_t w = threadIdx.x < kLayerAmaxThreads / 32 ? wmax[threadIdx.x] : 0u;
        w = __reduce_max_sync(0xFFFFFFFFu, w);
        if (threadIdx.x == 0) slots[blockIdx.x] = w;
    }
    ptx::griddep_launch_dependents();
}

__global__ void __launch_bounds__(kLayerAmaxThreads)
    k_quantize_slots(const uint16_t* __restrict__ x, int64_t nblocks, const uint32_t* __restrict__ slots, int n_slots,
                     uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, float* __restrict__ s_out)
{
    ptx::griddep_wait();  // the slots come from the launch before this one
    __shared__ uint32_t wmax[kLayerAmaxThreads / 32];
    uint32_t m = 0;
    for (int i = threadIdx.x; i < n_slots; i += blockDim.x) m = max(m, __ldcg(slots + i));
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kLayerAmaxThreads / 32; ++w) m = max(m, wmax[w]);
    const float amax = __uint_as_float(m);
    const float S = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
    if (s_out && blockIdx.x == 0 && threadIdx.x == 0) *s_out = S;
    const float six_s = __fmul_rn(6.0f, S);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblocks; b += stride) {
        float v[16];
        load16(x + b * 16, v);
        uint32_t lo, hi;
        const uint32_t s = nvfp4_encode16(v, S, six_s, lo, hi);
        *reinterpret_cast<uint2*>(codes + b * 8) = make_uint2(lo, hi);
        sf[b] = static_cast<uint8_t>(s);
    }
    ptx::griddep_launch_dependents();
}

// Small tensors (<= kSmallBlocks blocks, e.g. a decode batch): one CTA computes the max and encodes,
// one launch instead of three.
constexpr int64_t kSmallBlocks = 4096;
constexpr int kSmallThreads = 512;

template <typename Tin>
__global__ void __launch_bounds__(kSmallThreads)
    k_quantize_small(const Tin* __restrict__ x, int64_t nblocks, const float* __restrict__ s_static,
                     uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, float* __restrict__ s_out,
                     int32_t* __restrict__ zero, int n_zero)
{
    ptx::griddep_wait();  // x may come from the launch before this one
    __shared__ uint32_t wmax[kSmallThreads / 32];
    __shared__ float S_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < n_zero; i += kSmallThreads) zero[i] = 0;
    if (s_static) {
        if (tid == 0) S_s = *s_static;
    } else {
        uint32_t m = 0;
        for (int64_t b = tid; b < nblocks; b += kSmallThreads) {
            float v[16];
            load16(x + b * 16, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) m = abs_bits_max(m, v[i]);
        }
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0) wmax[warp] = m;
        __syncthreads();
        if (warp == 0) {
            uint32_t w = lane < kSmallThreads / 32 ? wmax[lane] : 0u;
            w = __reduce_max_sync(0xFFFFFFFFu, w);
            if (lane == 0) {
                const float amax = __uint_as_float(w);
                S_s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
            }
        }
    }
    __syncthreads();
    const float S = S_s;
    if (s_out && tid == 0) *s_out = S;
    const float six_s = __fmul_rn(6.0f, S);
    for (int64_t b = tid; b < nblocks; b += kSmallThreads) {
        float v[16];
        load16(x + b * 16, v);
        uint32_t lo, hi;
        const uint32_t s = nvfp4_encode16(v, S, six_s, lo, hi);
        *reinterpret_cast<uint2*>(codes + b * 8) = make_uint2(lo, hi);
        sf[b] = static_cast<uint8_t>(s);
    }
    ptx::griddep_launch_dependents();
}

static int quant_grid(int64_t nblocks, int sms)
{
    const int64_t want = (nblocks + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    return static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
}

template <typename Tin>
cudaError_t launch_quantize_t(const Tin* x, int64_t rows, int64_t K, const float* s_in, uint8_t* codes, uint8_t* sf,
                              float* s_out, unsigned* amax_scratch, int sms, cudaStream_t stream, bool amax_zeroed)
{
    const int64_t nblocks = rows * K / 16;
    if (nblocks <= kSmallBlocks)
        return launch_pdl(k_quantize_small<Tin>, dim3(1), dim3(kSmallThreads), 0, stream, x, nblocks, s_in, codes, sf, s_out,
                          static_cast<int32_t*>(nullptr), 0);
    if (!s_in) {
        if (!amax_zeroed) {
            cudaError_t e = cudaMemsetAsync(amax_scratch, 0, sizeof(unsigned), stream);
            if (e != cudaSuccess) return e;
        }
        if (nblocks > 0) {
            cudaError_t e = launch_pdl(k_amax<Tin>, dim3(quant_grid(nblocks, sms)), dim3(256), 0, stream, x, nblocks, amax_scratch);
            if (e != cudaSuccess) return e;
        }
    }
    return launch_pdl(k_quantize<Tin>, dim3(quant_grid(nblocks, sms)), dim3(256), 0, stream, x, nblocks, s_in,
                      static_cast<const unsigned*>(amax_scratch), codes, sf, s_out);
}

cudaError_t launch_quantize(const uint16_t* x, int64_t rows, int64_t K, const float* s_in, uint8_t* codes, uint8_t* sf,
                            float* s_out, unsigned* amax_scratch, int sms, cudaStream_t stream, bool amax_zeroed)
{
    return launch_quantize_t<uint16_t>(x, rows, K, s_in, codes, sf, s_out, amax_scratch, sms, stream, amax_zeroed);
}

int layer_amax_slots(int sms) { return 4 * sms; }

cudaError_t launch_quantize_layer(const uint16_t* x, int64_t rows, int64_t K, uint8_t* codes, uint8_t* sf, float* s_out,
                                  uint32_t* slots, int32_t* zero, int n_zero, int sms, cudaStream_t stream)
{
    const int64_t nblocks = rows * K / 16;
    if (nblocks <= kSmallBlocks)
        return launch_pdl(k_quantize_small<uint16_t>, dim3(1), dim3(kSmallThreads), 0, stream, x, nblocks,
                          static_cast<const float*>(nullptr), codes, sf, s_out, zero, n_zero);
    const int64_t want = (nblocks + 4 * kLayerAmaxThreads - 1) / (4 * kLayerAmaxThreads);
    const int grid_a = static_cast<int>(want < 1 ? 1 : (want > layer_amax_slots(sms) ? layer_amax_slots(sms) : want));
    cudaError_t e = launch_pdl(k_amax_slots, dim3(grid_a), dim3(kLayerAmaxThreads), 0, stream, x, nblocks, slots, zero, n_zero);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_quantize_slots, dim3(quant_grid(nblocks, sms)), dim3(kLayerAmaxThreads), 0, stream, x, nblocks,
                      static_cast<const uint32_t*>(slots), grid_a, codes, sf, s_out);
}

cudaError_t launch_quantize_from_slots(const uint16_t* x, int64_t rows, int64_t K, uint8_t* codes, uint8_t* sf,
                                       float* s_out, const uint32_t* slots, int n_slots, int sms, cudaStream_t stream)
{
    const int64_t nblocks = rows * K / 16;
    return launch_pdl(k_quantize_slots, dim3(quant_grid(nblocks, sms)), dim3(kLayerAmaxThreads), 0, stream, x, nblocks,
                      slots, n_slots, codes, sf, s_out);
}

cudaError_t launch_quantize_f32(const float* x, int64_t rows, int64_t K, const float* s_in, uint8_t* codes,
                                uint8_t* sf, float* s_out, unsigned* amax_scratch, int sms, cudaStream_t stream)
{
    return launch_quantize_t<float>(x, rows, K, s_in, codes, sf, s_out, amax_scratch, sms, stream, false);
}

}  // namespace moe
