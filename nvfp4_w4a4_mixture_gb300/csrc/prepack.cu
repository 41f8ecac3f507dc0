// prepack.cu -- NVFP4 weights from the row-major layout to the layout the grouped GEMM streams.
//
// Codes become K-slab-major, [G][ceil(K/256)][N][128 bytes]: slab s holds bytes 128 s .. 128 s + 127
// of every row (256 E2M1 values; zero-padded past K/2), so the rows of one TMA box (a tile's K-stage)
// are one contiguous run in HBM. A gate/up matrix is reordered in 128-row blocks (64 gate rows then
// the 64 up rows of the same output columns) so one 128-column MMA tile holds matching gate and up
// columns. Block scales become 512-byte tiles, one per (128 rows, 4 K-blocks): byte
// (r%32)*16 + (r/32)*4 + j is the scale of row r, K-block j. This is the order in which tcgen05.cp
// (32x128b, replicated to the four lane quarters) places one 32-bit word of four scales per row
// into tensor memory.
#include "kernels.cuh"

namespace moe {

// source row of prepacked row `r` of an [N][K] matrix
__device__ __forceinline__ int prepack_src_row(int r, int N, int interleave)
{
    if (!interleave) return r;
    const int blk = r / 128, w = r % 128;
    return w < 64 ? blk * 64 + w : N / 2 + blk * 64 + (w - 64);
}

// one thread per 16-byte vector of the output, [G][slabs][N][8 vectors]
__global__ void k_prepack_codes(const uint8_t* __restrict__ codes, int G, int N, int K, int interleave,
                                uint8_t* __restrict__ out)
{
    const int slabs = (K + 255) / 256, row_vecs = K / 32;  // 16-byte vectors per source row of K/2 bytes
    const int64_t total = static_cast<int64_t>(G) * slabs * N * 8;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int v = static_cast<int>(i % 8);
        const int r = static_cast<int>((i / 8) % N);
        const int64_t gs = i / (8 * static_cast<int64_t>(N));
        const int sl = static_cast<int>(gs % slabs);
        const int64_t g = gs / slabs;
        const int sv = sl * 8 + v;  // vector within the source row
        uint4 val = make_uint4(0, 0, 0, 0);
        if (sv < row_vecs) {
            const int src = prepack_src_row(r, N, interleave);
            val = __ldg(reinterpret_cast<const uint4*>(codes + (g * N + src) * (K / 2)) + sv);
        }
        reinterpret_cast<uint4*>(out)[i] = val;
    }
}

// one thread per (group, row, 4-scale word)
__global__ void k_prepack_sf(const uint8_t* __restrict__ sf, int G, int N, int K, int interleave,
                             uint8_t* __restrict__ out)
{
    const int words_per_row = K / 64;
    const int64_t total = static_cast<int64_t>(G) * N * words_per_row;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int kw = static_cast<int>(i % words_per_row);
        const int64_t gr = i / words_per_row;
        const int r = static_cast<int>(gr % N);
        const int64_t g = gr / N;
        const int src = prepack_src_row(r, N, interleave);
        const uint32_t word = *reinterpret_cast<const uint32_t*>(sf + (g * N + src) * (K / 16) + kw * 4);
        const int64_t tile = (g * (N / 128) + r / 128) * words_per_row + kw;
        const int rr = r % 128;
        *reinterpret_cast<uint32_t*>(out + tile * 512 + (rr % 32) * 16 + (rr / 32) * 4) = word;
    }
}

cudaError_t launch_prepack(const uint8_t* codes, const uint8_t* sf, int G, int N, int K, int interleave,
                           uint8_t* codes_out, uint8_t* sf_out, cudaStream_t stream)
{
    const int threads = 256;
    const int sms = device_sm_count();
    k_prepack_codes<<<sms * 8, threads, 0, stream>>>(codes, G, N, K, interleave, codes_out);
    k_prepack_sf<<<sms * 8, threads, 0, stream>>>(sf, G, N, K, interleave, sf_out);
    return cudaGetLastError();
}

}  // namespace moe
