// permute.cu -- stable counting sort of the T*k (token, slot) assignments by expert id.
//
// The flat assignment list f = t*k + j is cut into chunks of kPermChunk entries, one CTA each; the
// CTA's kPermWarps warps take kPermChunk / kPermWarps consecutive entries each.
//   1. histogram: each warp counts its entries per expert (warp match: one shared-memory add per
//      run of equal ids, no atomics), the CTA sums its warps -> hist[expert][chunk];
//   2. row scan (one CTA per expert): exclusive scan of the expert's counts over the chunks, the
//      expert's total to totals[expert]; the last CTA to finish (atomic ticket, no waiting) scans
//      the totals over the experts -> expert offsets (the shared expert appended as group E);
//   3. scatter: each warp counts its entries again, an exclusive scan over the CTA's warps gives
//      every warp its base per expert (offset + chunk base + earlier warps' counts), and the warp
//      walks its entries in order, an entry's position being that base plus the number of earlier
//      entries of the same expert in the warp. Ascending f within every expert (stable),
//      independent of scheduling: bit-exact.
#include <cub/block/block_scan.cuh>

#include "kernels.cuh"

namespace moe {

constexpr int kPermWarps = 8;
constexpr int kPermWarpEntries = kPermChunk / kPermWarps;  // consecutive entries per warp
static_assert(kPermChunk % (kPermWarps * 32) == 0, "whole warp passes");

// Counts of this warp's entries per expert into my[0..E) (zeroed first); ids outside [0, E) are
// dropped (and reported when status is given).
__device__ __forceinline__ void warp_count(const int32_t* __restrict__ ids, int64_t beg, int64_t end, int E, int32_t* my,
                                           int lane, int* status)
{
    for (int e = lane; e < E; e += 32) my[e] = 0;
    __syncwarp();
    for (int64_t base = beg; base < end; base += 32) {
        const int64_t i = base + lane;
        int e = -1;
        if (i < end) {
            e = ids[i];
            if (e < 0 || e >= E) {
                if (status) record_status(status, kDevBadExpertId);
                e = -1;
            }
        }
        const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
        if (e >= 0 && lane == __ffs(m) - 1) my[e] += __popc(m);
        __syncwarp();
    }
}

__global__ void __launch_bounds__(kPermWarps * 32)
    k_perm_hist(const int32_t* __restrict__ ids, int64_t n, int E, int64_t nchunks, int32_t* __restrict__ hist,
                int* status)
{
    ptx::griddep_wait();  // inputs come from the launch before this one
    extern __shared__ int32_t cnt[];  // [kPermWarps][E]
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t c = blockIdx.x;
    const int64_t beg = min(n, c * kPermChunk + warp * kPermWarpEntries), end = min(n, beg + kPermWarpEntries);
    warp_count(ids, beg, end, E, cnt + warp * E, lane, status);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kPermWarps * 32) {
        int32_t t = 0;
#pragma unroll
        for (int w = 0; w < kPermWarps; ++w) t += cnt[w * E + e];
        hist[static_cast<int64_t>(e) * nchunks + c] = t;
    }
}

constexpr int kScanThreads = 1024;
constexpr int kRowScanThreads = 256;

// One CTA per expert row of hist [E][nchunks]: exclusive scan in place, row total to totals[e];
// the last CTA scans the totals into the expert offsets and returns the ticket to zero.
__global__ void __launch_bounds__(kRowScanThreads)
    k_perm_rowscan(int32_t* __restrict__ hist, int32_t* __restrict__ totals, int64_t nchunks, int E, int T,
                   int with_shared, int32_t* __restrict__ offsets, unsigned* ticket)
{
    ptx::griddep_wait();  // inputs come from the launch before this one
    using Scan = cub::BlockScan<int32_t, kRowScanThreads>;
    __shared__ typename Scan::TempStorage tmp;
    __shared__ unsigned last_s;
    const int e = blockIdx.x, tid = threadIdx.x;
    int32_t* row = hist + static_cast<int64_t>(e) * nchunks;
    const int64_t per = (nchunks + kRowScanThreads - 1) / kRowScanThreads;
    const int64_t c0 = tid * per, c1 = min(nchunks, c0 + per);
    int32_t sum = 0;
    for (int64_t c = c0; c < c1; ++c) sum += row[c];
    int32_t run, agg;
    Scan(tmp).ExclusiveSum(sum, run, agg);
    for (int64_t c = c0; c < c1; ++c) {
        const int32_t v = row[c];
        row[c] = run;
        run += v;
    }
    if (tid == 0) totals[e] = agg;
    __threadfence();
    __syncthreads();
    if (tid == 0) last_s = atomicAdd(ticket, 1u) == gridDim.x - 1 ? 1u : 0u;
    __syncthreads();
    if (!last_s) return;
    __threadfence();
    // expert offsets: exclusive scan of the E <= 1024 totals, 4 per thread
    int32_t v[4], o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int g = tid * 4 + i;
        v[i] = g < E ? __ldcg(totals + g) : 0;
    }
    int32_t total;
    __syncthreads();  // tmp reused
    Scan(tmp).ExclusiveSum(v, o, total);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int g = tid * 4 + i;
        if (g < E) offsets[g] = o[i];
    }
    if (tid == 0) {
        offsets[E] = total;
        offsets[E + 1] = total + (with_shared ? T : 0);
        *ticket = 0u;
    }
}

__global__ void __launch_bounds__(kPermWarps * 32)
    k_perm_scatter(const int32_t* __restrict__ ids, int64_t n, int E, int k, int T, int with_shared, int64_t nchunks,
                   const int32_t* __restrict__ hist, const int32_t* __restrict__ offsets, int32_t* __restrict__ perm_src,
                   int32_t* __restrict__ src_perm, int32_t* __restrict__ row_token)
{
    ptx::griddep_wait();  // inputs come from the launch before this one
    extern __shared__ int32_t base_s[];  // [kPermWarps][E]: this warp's counts, then its bases
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // the shared-expert rows: row T*k + t holds token t
    if (row_token && with_shared) {
        for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < T;
             t += static_cast<int64_t>(gridDim.x) * blockDim.x)
            row_token[n + t] = static_cast<int32_t>(t);
    }
    const int64_t c = blockIdx.x;
    const int64_t beg = min(n, c * kPermChunk + warp * kPermWarpEntries), end = min(n, beg + kPermWarpEntries);
    int32_t* my = base_s + warp * E;
    warp_count(ids, beg, end, E, my, lane, nullptr);
    __syncthreads();
    // each warp's base per expert: offset + the chunk's base + the counts of the earlier warps
    for (int e = threadIdx.x; e < E; e += kPermWarps * 32) {
        int32_t run = __ldg(offsets + e) + hist[static_cast<int64_t>(e) * nchunks + c];
#pragma unroll
        for (int w = 0; w < kPermWarps; ++w) {
            const int32_t v = base_s[w * E + e];
            base_s[w * E + e] = run;
            run += v;
        }
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int64_t b = beg; b < end; b += 32) {
        const int64_t i = b + lane;
        int e = -1;
        if (i < end) {
            e = ids[i];
            if (e < 0 || e >= E) e = -1;
        }
        const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
        if (e >= 0) {
            const int32_t pos = my[e] + __popc(m & lt);
            perm_src[pos] = static_cast<int32_t>(i);
            src_perm[i] = pos;
            if (row_token) row_token[pos] = static_cast<int32_t>(i / k);
        }
        __syncwarp();
        if (e >= 0 && lane == __ffs(m) - 1) my[e] += __popc(m);
        __syncwarp();
    }
}

// Small assignment lists (n <= kSmallPerm, e.g. a decode batch): one CTA, one launch. Counts by
// shared-memory atomics (order-free), offsets by a block scan, and each entry's rank within its
// expert = the number of earlier entries with the same id (a direct count): stable, bit-exact.
constexpr int kSmallPerm = 512;

__global__ void __launch_bounds__(kScanThreads)
    k_perm_small(const int32_t* __restrict__ ids, int n, int E, int k, int T, int with_shared, int32_t* __restrict__ offsets,
                 int32_t* __restrict__ perm_src, int32_t* __restrict__ src_perm, int32_t* __restrict__ row_token,
                 int* status)
{
    ptx::griddep_wait();  // inputs come from the launch before this one
    using Scan = cub::BlockScan<int32_t, kScanThreads>;
    __shared__ typename Scan::TempStorage tmp;
    __shared__ int32_t ids_s[kSmallPerm];
    __shared__ int32_t base_s[1024];
    __shared__ int32_t total_s;
    const int tid = threadIdx.x;
    if (tid < E) base_s[tid] = 0;
    __syncthreads();
    for (int f = tid; f < n; f += kScanThreads) {
        int e = ids[f];
        if (e < 0 || e >= E) {
            record_status(status, kDevBadExpertId);
            e = -1;
        }
        ids_s[f] = e;
        if (e >= 0) atomicAdd(&base_s[e], 1);
    }
    __syncthreads();
    const int32_t cnt = tid < E ? base_s[tid] : 0;
    int32_t off;
    Scan(tmp).ExclusiveSum(cnt, off);
    if (tid < E) {
        offsets[tid] = off;
        base_s[tid] = off;
    }
    if (tid == E - 1) total_s = off + cnt;
    __syncthreads();
    if (tid == 0) {
        offsets[E] = total_s;
        offsets[E + 1] = total_s + (with_shared ? T : 0);
    }
    for (int f = tid; f < n; f += kScanThreads) {
        const int e = ids_s[f];
        if (e < 0) continue;
        int r = 0;
        for (int q = 0; q < f; ++q) r += ids_s[q] == e;
        const int pos = base_s[e] + r;
        perm_src[pos] = f;
        src_perm[f] = pos;
        if (row_token) row_token[pos] = f / k;
    }
    if (row_token && with_shared)
        for (int t = tid; t < T; t += kScanThreads) row_token[n + t] = t;
}

cudaError_t launch_permute(const int32_t* topk_ids, int T, int k, int E, int with_shared, int32_t* offsets,
                           int32_t* perm_src, int32_t* src_perm, int32_t* row_token, int32_t* hist, unsigned* ticket,
                           int* status, cudaStream_t stream)
{
    const int64_t n = static_cast<int64_t>(T) * k;
    if (n <= kSmallPerm) {
        return launch_pdl(k_perm_small, dim3(1), dim3(kScanThreads), 0, stream, topk_ids, static_cast<int>(n), E, k, T,
                          with_shared, offsets, perm_src, src_perm, row_token, status);
    }
    const int64_t nchunks = perm_chunks(n);
    const int blocks = static_cast<int>(nchunks);
    const size_t smem = static_cast<size_t>(kPermWarps) * E * sizeof(int32_t);
    int32_t* totals = hist + nchunks * E;
    cudaError_t e = launch_pdl(k_perm_hist, dim3(blocks), dim3(kPermWarps * 32), smem, stream, topk_ids, n, E, nchunks, hist,
                               status);
    if (e == cudaSuccess)
        e = launch_pdl(k_perm_rowscan, dim3(E), dim3(kRowScanThreads), 0, stream, hist, totals, nchunks, E, T, with_shared,
                       offsets, ticket);
    if (e == cudaSuccess)
        e = launch_pdl(k_perm_scatter, dim3(blocks), dim3(kPermWarps * 32), smem, stream, topk_ids, n, E, k, T, with_shared,
                       nchunks, hist, static_cast<const int32_t*>(offsets), perm_src, src_perm, row_token);
    return e;
}

}  // namespace moe
