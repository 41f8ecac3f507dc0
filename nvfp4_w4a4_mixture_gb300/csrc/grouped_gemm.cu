// grouped_gemm.cu -- block-scaled NVFP4 grouped GEMM on the 5th-generation tensor cores.
//
// out[p][n] = a_scale * b_scale[g] * sum_k act[src(p)][k] * w[g][n][k] for the rows p of group g,
// computed by tcgen05.mma kind::mxf4nvf4 (E2M1 x E2M1 products, one UE4M3 scale per 16 along K,
// FP32 accumulation in tensor memory).
//
// One persistent CTA per SM; the weight producer of each CTA takes output tiles (token block of a
// group x W_ROWS weight rows) from a global counter, weight blocks fastest, so CTAs working at the
// same time share a token block's activation rows and one expert's weights stay in L2 across its
// token blocks. Tile shapes:
//   activations on M (large groups): 128 token rows x 128 weight rows, MMA 128 x 128;
//   weights on M (small groups): 128 weight rows x 32 token rows, MMA 128 x 32;
//   wide: 128 token rows x 256 weight rows, MMA 128 x 256 (half the MMAs and scale copies per
//     weight byte; single-buffered accumulator);
//   wide-narrow: wide with 32-row token blocks (decode), the accumulator finished through shared
//     memory by all epilogue warps; given the routing ids, each CTA builds the permutation itself;
//   wide, token-block units: a CTA takes a whole token block through every weight block of its
//     phase, keeping the block's activation scales in tensor memory;
//   weight-resident units (large batches): a CTA keeps one expert's 128-row weight block (all of K)
//     in shared memory and its scales in tensor memory, and streams up to 16 of the expert's token
//     blocks past it into a double-buffered 128 x 128 accumulator: each weight byte is read from
//     memory once, the streamed activation rows are L2-resident, and each K-step copies one scale
//     tile (the activations').
// A launch can hold two problems (phases) over the same groups: the gate/up GEMM with its SwiGLU
// epilogue, then the down GEMM reading the intermediate h. All phase-0 tiles are handed out before
// any phase-1 tile. A down tile of token block b waits (bounded) until every gate/up tile of block
// b has stored its part of h: the gate/up epilogue warps publish with a fence and an atomic count
// per token block. The grid is at most one CTA per SM, each needing most of an SM's shared memory,
// so all CTAs become resident and such a wait ends. h's block scales are written in 512-byte
// token-block tiles, the layout the down GEMM copies straight into shared memory.
// Warp roles:
//   warp 0       weight producer: takes the tiles and hands their indices to the other roles through
//                a shared-memory ring; per K-stage of 256 elements, TMA of the W_ROWS x 128-byte
//                weight box (128-byte swizzle) and bulk copies of its scale-factor tiles;
//   warp 1       TMEM owner and MMA issuer: per K-step of 64, tcgen05.cp of the scale-factor tiles
//                into tensor memory and one tcgen05.mma into the (double- or single-buffered)
//                accumulator;
//   warps 2-3    activation producers: gather the tile's activation rows (row index list) with
//                cp.async into the swizzled layout, and their scale factors into tile layout; a
//                stage's arrival is tracked by cp.async.mbarrier.arrive (or, for 32-row blocks,
//                made by the warp once the copies have landed);
//   warps 4..    epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes 32*(w%4)..+31), apply
//                the tensor scales and write FP32 / bf16 rows, or SwiGLU + NVFP4 requantisation.
// Stage hand-over uses mbarriers (full: producers -> MMA; empty: MMA commit -> producers;
// acc_full / acc_empty: MMA <-> epilogue). Every wait is bounded (ptx::mbar_wait, spin_until): on
// timeout the CTA records kDevTimeoutGemm in the status word, all roles stop, and TMEM is freed
// after the tensor cores drain.
#include <climits>

#include "kernels.cuh"
#include "route.cuh"

namespace moe {

namespace {

constexpr int BK_BYTES = 128;              // K-stage: one 128-byte swizzle row = 256 E2M1 values
constexpr int SF_TILE = 512;               // scale factors of 128 rows x 4 K-blocks
constexpr int SF_STAGE = 4 * SF_TILE;      // 4 MMA K-steps of 64 per stage
constexpr int kNumActProducers = 64;       // warps 2-3; each arrives on every stage's full barrier
constexpr int kTileRing = 8;               // tiles handed from the weight producer to the other roles

// Tile shapes. W_ROWS weight rows (one TMA box) by ACT_ROWS activation rows per tile; ACC_BUFS
// accumulators of ACC_COLS tensor-memory columns.
enum : int { kModeActM = 0, kModeSwap = 1, kModeWide = 2, kModeWideNarrow = 3, kModeWideRows = 4, kModeWRes = 5 };
template <int kMode>
struct Cfg;
template <>
struct Cfg<kModeActM> {                    // activations on the MMA's M side, 128 weight rows on N
    static constexpr int ACT_ROWS = 128, W_ROWS = 128, STAGES = 6, EPI_WARPS = 8, ACC_COLS = 128, ACC_BUFS = 2;
    static constexpr int MMA_M = 128, MMA_N = 128;
    static constexpr bool SWAP = false, XCHG = false, ROWS = false, WRES = false, SPLIT = false;
    static constexpr int MAX_K = 16384;
};
template <>
struct Cfg<kModeSwap> {                    // weights on the MMA's M side, 32 activation rows on N
    static constexpr int ACT_ROWS = 32, W_ROWS = 128, STAGES = 8, EPI_WARPS = 4, ACC_COLS = 32, ACC_BUFS = 2;
    static constexpr int MMA_M = 128, MMA_N = 32;
    static constexpr bool SWAP = true, XCHG = false, ROWS = false, WRES = false, SPLIT = false;
    static constexpr int MAX_K = 16384;
};
template <>
struct Cfg<kModeWide> {                    // activations on M, 256 weight rows on N: half the MMAs and
    // scale copies per weight byte of the 128-row shapes; the 256-column accumulator leaves room for
    // one buffer only, so the epilogue frees it as soon as its rows are in registers
    static constexpr int ACT_ROWS = 128, W_ROWS = 256, STAGES = 4, EPI_WARPS = 8, ACC_COLS = 256, ACC_BUFS = 1;
    static constexpr int MMA_M = 128, MMA_N = 256;
    // (two MMA threads here would each copy the activation scales every K-step: measured slower)
    static constexpr bool SWAP = false, XCHG = false, ROWS = false, WRES = false, SPLIT = false;
    static constexpr int MAX_K = 16384;
};

template <>
struct Cfg<kModeWideNarrow> {              // wide, for token blocks of at most 32 rows (decode): the
    // activation region holds 32 rows, the MMA's other 96 A rows read the weight region behind it
    // (their accumulator rows are never stored). Only lane quarter 0 of the accumulator holds rows,
    // so its two warps copy the accumulator to shared memory (XCHG) and all eight epilogue warps
    // finish it; four stages keep the ring as fast as five did
    static constexpr int ACT_ROWS = 32, W_ROWS = 256, STAGES = 4, EPI_WARPS = 8, ACC_COLS = 256, ACC_BUFS = 1;
    static constexpr int MMA_M = 128, MMA_N = 256;
    static constexpr bool SWAP = false, XCHG = true, ROWS = false, WRES = false, SPLIT = false;
    static constexpr int MAX_K = 16384;
};
template <>
struct Cfg<kModeWideRows> {                // wide tiles taken a whole token block at a time: one CTA runs
                                           // every weight block of the token block in turn, and the
                                           // activation scales of the whole K stay in tensor memory
                                           // after the first; two MMA threads, each issuing one
                                           // weight scale copy and one 128 x 128 MMA per K-step
    static constexpr int ACT_ROWS = 128, W_ROWS = 256, STAGES = 4, EPI_WARPS = 8, ACC_COLS = 256, ACC_BUFS = 1;
    static constexpr int MMA_M = 128, MMA_N = 256;
    static constexpr bool SWAP = false, XCHG = false, ROWS = true, WRES = false, SPLIT = true;
    static constexpr int MAX_K = 2048;     // resident activation scales: 4 columns per 64 of K
};
template <>
struct Cfg<kModeWRes> {                    // weight-resident units: one expert's 128-row weight block in
                                           // shared memory (8 slabs of 256 K-values) with its scales in
                                           // tensor memory; up to 16 of the expert's token blocks stream
                                           // through the stages (activations only) into two 128-column
                                           // accumulators, so the epilogue of one block overlaps the next
    static constexpr int ACT_ROWS = 128, W_ROWS = 128, STAGES = 3, EPI_WARPS = 8, ACC_COLS = 128, ACC_BUFS = 2;
    static constexpr int MMA_M = 128, MMA_N = 128;
    static constexpr bool SWAP = false, XCHG = false, ROWS = false, WRES = true, SPLIT = false;
    static constexpr int MAX_K = 2048;     // weight slabs (8 x 18 KB) and their scales (128 columns)
};

template <int kMode>
struct Lay {
    using C = Cfg<kMode>;
    static constexpr int WB = C::W_ROWS / 128;  // 128-row weight blocks per tile (scale tiles per K-step)
    static constexpr int W_BYTES = C::W_ROWS * BK_BYTES;  // one weight K-stage (a TMA box)
    // weight bytes per stage (weight-resident units keep the weights in their own region)
    static constexpr int STAGE_W = C::WRES ? 0 : W_BYTES;
    static constexpr int ACT_BYTES = C::ACT_ROWS * BK_BYTES;
    // activation rows first, so an MMA reading MMA_M > ACT_ROWS rows from them stays inside the stage
    static constexpr bool ACT_FIRST = C::ACT_ROWS < C::MMA_M && !C::SWAP;
    static_assert(!ACT_FIRST || (C::MMA_M - C::ACT_ROWS) * BK_BYTES <= W_BYTES, "A rows read past the activations");
    static constexpr int OFF_ACT = ACT_FIRST ? 0 : STAGE_W, OFF_W = ACT_FIRST ? ACT_BYTES : 0;
    static constexpr int OFF_SFW = STAGE_W + ACT_BYTES, OFF_SFACT = OFF_SFW + (C::WRES ? 0 : WB * SF_STAGE);
    static constexpr int STAGE_BYTES = OFF_SFACT + SF_STAGE;
    // resident weights (WRES): MAX_SLABS slabs of W_ROWS x 128 bytes (256 K-values, 128-byte swizzle,
    // as a stage's weight box) after the stages, then each slab's 4 scale tiles
    static constexpr int MAX_SLABS = C::WRES ? C::MAX_K / 256 : 0;
    static constexpr int B_OFF = C::STAGES * STAGE_BYTES;
    static constexpr int B_SF_OFF = B_OFF + MAX_SLABS * W_BYTES;
    static constexpr int TAIL_OFF = B_SF_OFF + MAX_SLABS * WB * SF_STAGE;
    static constexpr int THREADS = 128 + 32 * C::EPI_WARPS;
    // SPLIT: warp 0 is a second MMA thread (each owns 128 of the tile's 256 weight rows) and the
    // first activation producer warp also loads the weights
    static constexpr int MMA_THREADS = C::SPLIT ? 2 : 1;
    static constexpr int SF_COL = C::ACC_BUFS * C::ACC_COLS;  // first scale-factor column
    static constexpr int SFW_STEP_COLS = 4 * WB;               // weight scale columns per K-step
    // per stage: 4 K-steps of weight scales, and of activation scales unless they are resident
    static constexpr int STAGE_SF_COLS = 4 * ((C::WRES ? 0 : SFW_STEP_COLS) + (C::ROWS ? 0 : 4));
    static constexpr int TMEM_COLS = 512;
    // resident scales of the whole K: the activations' (ROWS, 4 columns per K-step) or the weights'
    // (WRES, 4 columns per K-step and 128 rows)
    static constexpr int RES_SF_COL = SF_COL + STAGE_SF_COLS * C::STAGES;
    // epilogue warps that take tiles: with 32-row token blocks on the MMA's M side only lane quarter
    // 0 holds rows, so unless they share the work through shared memory (XCHG) the other quarters'
    // warps stay out (no polling, no arrivals)
    static constexpr int EPI_ACTIVE =
        (!C::SWAP && !C::XCHG && C::ACT_ROWS <= 32) ? C::EPI_WARPS / 4 : C::EPI_WARPS;
    // arrivals that free the accumulator: the warps that read it
    static constexpr int ACC_READERS = C::XCHG ? C::EPI_WARPS / 4 : EPI_ACTIVE;
    static constexpr int READY_PER_TILE = EPI_ACTIVE;  // epilogue warp arrivals per gate/up tile
    // activation stages published by the producer warps (32-row token blocks) rather than by
    // cp.async-tracked arrivals
    static constexpr bool PUBLISH = C::ACT_ROWS <= 32;
    static_assert(SF_COL + STAGE_SF_COLS * C::STAGES <= TMEM_COLS, "tensor memory budget");
    static_assert(!(C::ROWS || C::WRES) || RES_SF_COL + 4 * (C::WRES ? WB : 1) * (C::MAX_K / 64) <= TMEM_COLS,
                  "resident scales");
    static_assert(B_OFF % 1024 == 0 && W_BYTES % 1024 == 0, "resident slabs keep 1024-byte alignment");
    static_assert(STAGE_BYTES % 1024 == 0, "stages keep 1024-byte alignment");
};

// 16-byte aligned size: the exchange buffers placed right after it are accessed with 16-byte loads
template <int kMode>
struct alignas(16) Tail {
    uint64_t full[Cfg<kMode>::STAGES];
    uint64_t empty[Cfg<kMode>::STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint64_t drain_b;     // SPLIT: the second MMA thread's operations finished
    uint64_t xchg_full;   // weights-on-M SwiGLU: up values written (64 arrivals)
    uint64_t xchg_empty;  // weights-on-M SwiGLU: up values consumed (64 arrivals)
    uint64_t r_full[8];   // resident weight slab loaded (TMA bytes)
    uint64_t r_empty[8];  // resident weight slab no longer read (MMA commit)
    uint64_t tile_full[kTileRing];   // tile index written (1 arrival)
    uint64_t tile_empty[kTileRing];  // tile index read by the act producers, MMA and epilogue warps
    int32_t tile_L[kTileRing];
    uint32_t tmem_base;
    int abort;
    int32_t wsum[32];
    int32_t tb_off[kGemmMaxG + 1];
    int32_t g_off[kGemmMaxG + 1];  // the group offsets, so a tile's rows need no global load
    int32_t ur_off[Cfg<kMode>::WRES ? kGemmMaxG + 1 : 1];  // weight-resident units: runs before group order s
};

// up-projection values handed from TMEM lanes 64..127 to lanes 0..63 (weights-on-M SwiGLU)
struct SwapXchg {
    float u[64][33];
};

// a 32-row tile's accumulator in shared memory (XCHG epilogue); rows padded to 260 words so a
// warp's 16-byte accesses to 32 rows at one column hit distinct banks in each 8-lane phase
struct AccXchg {
    float v[32][260];
};

// a launch's own permutation (GemmRoute): permuted row -> source row of x (gate/up gather), and
// permuted routed row -> assignment t*k + j (down output row)
struct RouteSmem {
    int32_t row[kRouteMaxAssign + kRouteMaxT];
    int32_t perm[kRouteMaxAssign];
};

template <int kMode>
constexpr size_t smem_bytes();
static_assert(sizeof(Tail<kModeWideNarrow>) % 16 == 0 && sizeof(Tail<kModeSwap>) % 16 == 0 &&
                  sizeof(Tail<kModeActM>) % 16 == 0 && sizeof(Tail<kModeWRes>) % 16 == 0,
              "exchange buffers after the tail stay 16-byte aligned");
static_assert(Lay<kModeWideNarrow>::TAIL_OFF % 16 == 0 && Lay<kModeSwap>::TAIL_OFF % 16 == 0, "tail offset");

template <int kMode>
constexpr size_t smem_bytes()
{
    return 1024 + static_cast<size_t>(Lay<kMode>::TAIL_OFF) + sizeof(Tail<kMode>) +
           (Cfg<kMode>::SWAP ? sizeof(SwapXchg) : 0) + (Cfg<kMode>::XCHG ? sizeof(AccXchg) + sizeof(RouteSmem) : 0);
}
static_assert(smem_bytes<kModeActM>() <= 232448 && smem_bytes<kModeSwap>() <= 232448 &&
                  smem_bytes<kModeWide>() <= 232448 && smem_bytes<kModeWideNarrow>() <= 232448 &&
                  smem_bytes<kModeWideRows>() <= 232448 && smem_bytes<kModeWRes>() <= 232448,
              "shared memory per CTA (227 KB)");

struct TileInfo {
    int ph, g, nb, tbg, row0, rows;
    int nbk;  // token blocks of a weight-resident unit (from tbg / row0 on), else 1
};

// tb_off[g] = sum_{g' < g} ceil(rows_g' / act_rows), g = 0..G (block-wide scan; contains barriers),
// and g_off = offsets[0..G] (offsets in global or shared memory; g_off may be offsets itself)
__device__ void block_tile_prefix(const int32_t* __restrict__ offsets, int G, int act_rows, int32_t* tb_off,
                                  int32_t* g_off, int32_t* wsum)
{
    const int nt = blockDim.x, t = threadIdx.x, lane = t & 31, warp = t >> 5, nwarps = nt >> 5;
    const int per = (G + nt - 1) / nt;
    const int g0 = min(G, t * per), g1 = min(G, g0 + per);
    int32_t s = 0;
    for (int g = g0; g < g1; ++g) {
        const int32_t r = offsets[g + 1] - offsets[g];
        s += r > 0 ? (r + act_rows - 1) / act_rows : 0;
    }
    int32_t x = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int32_t w = lane < nwarps ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nwarps) wsum[lane] = w;
    }
    __syncthreads();
    int32_t run = x - s + (warp > 0 ? wsum[warp - 1] : 0);
    for (int g = g0; g < g1; ++g) {
        tb_off[g] = run;
        const int32_t o0 = offsets[g], r = offsets[g + 1] - o0;
        if (g_off != offsets) g_off[g] = o0;
        run += r > 0 ? (r + act_rows - 1) / act_rows : 0;
    }
    if (t == nt - 1) {
        tb_off[G] = wsum[nwarps - 1];
        if (g_off != offsets) g_off[G] = offsets[G];
    }
    __syncthreads();
}

// Group, first row and row count of token block ti.tbg (tb_off[g] <= tbg < tb_off[g + 1]).
__device__ __forceinline__ void place_block(const int32_t* tb_off, const int32_t* g_off, const GemmArgs& a,
                                            int act_rows, TileInfo& ti)
{
    int lo = 0, hi = a.G;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tb_off[mid] <= ti.tbg) lo = mid; else hi = mid;
    }
    ti.g = lo;
    const int g0 = g_off[lo], g1 = g_off[lo + 1];
    ti.row0 = g0 + (ti.tbg - tb_off[lo]) * act_rows;
    ti.rows = min(act_rows, g1 - ti.row0);
}

// Tile L of the launch: phase-0 tiles first (token block major, weight block minor), then phase 1.
__device__ __forceinline__ TileInfo tile_info(const int32_t* tb_off, const int32_t* g_off, const GemmArgs& a,
                                              int act_rows, int w_rows, int tiles0, int L)
{
    TileInfo ti;
    ti.ph = L >= tiles0 ? 1 : 0;
    const int Lp = L - (ti.ph ? tiles0 : 0);
    const int n_wb = a.p[ti.ph].N / w_rows;
    ti.tbg = Lp / n_wb;
    ti.nb = Lp - ti.tbg * n_wb;
    ti.nbk = 1;
    place_block(tb_off, g_off, a, act_rows, ti);
    return ti;
}

// Weight-resident units: the groups are taken in the order G - 1 (the largest one in a layer: the
// shared expert, one row per token), 0, 1, ..., G - 2, and each group's token blocks in runs of at
// most kWresRun; ur_off[s] counts the runs of the groups before order position s.
constexpr int kWresRun = 16;
__device__ __forceinline__ int wres_group(int s, int G) { return s == 0 ? G - 1 : s - 1; }

// Work unit L of a weight-resident launch: phase-0 units first, then phase 1; within a phase the
// runs in group order, each run's 128-row weight blocks fastest (CTAs working at the same time
// stream the same activation rows from L2).
__device__ __forceinline__ TileInfo wres_unit_info(const int32_t* tb_off, const int32_t* g_off, const int32_t* ur_off,
                                                   const GemmArgs& a, int units0, int L)
{
    TileInfo ti;
    ti.ph = L >= units0 ? 1 : 0;
    const int Lp = L - (ti.ph ? units0 : 0);
    const int n_wb = a.p[ti.ph].N / 128;
    const int ur = Lp / n_wb;
    ti.nb = Lp - ur * n_wb;
    int lo = 0, hi = a.G;  // the last order position whose runs start at or before ur
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (ur_off[mid] <= ur) lo = mid; else hi = mid;
    }
    const int g = wres_group(lo, a.G);
    const int b0 = (ur - ur_off[lo]) * kWresRun;
    ti.g = g;
    ti.nbk = min(kWresRun, tb_off[g + 1] - tb_off[g] - b0);
    ti.tbg = tb_off[g] + b0;
    ti.row0 = g_off[g] + b0 * 128;
    ti.rows = min(128, g_off[g + 1] - ti.row0);
    return ti;
}

// Work unit L of a launch with token-block units (ROWS): phase-0 token blocks first, then phase 1;
// nb is left 0 (the unit covers every weight block).
__device__ __forceinline__ TileInfo unit_info(const int32_t* tb_off, const int32_t* g_off, const GemmArgs& a,
                                              int act_rows, int units0, int L)
{
    TileInfo ti;
    ti.ph = L >= units0 ? 1 : 0;
    ti.tbg = L - (ti.ph ? units0 : 0);
    ti.nb = 0;
    ti.nbk = 1;
    place_block(tb_off, g_off, a, act_rows, ti);
    return ti;
}

template <int kMode>
__device__ __forceinline__ void set_abort(Tail<kMode>& t, int* status)
{
    if (atomicExch(&t.abort, 1) == 0) record_status(status, kDevTimeoutGemm);
}

template <int kMode>
__device__ __forceinline__ bool aborted(const Tail<kMode>& t)
{
    return *reinterpret_cast<const volatile int*>(&t.abort) != 0;
}

// Tile hand-over: the weight producer takes tiles from a global counter (the first one is
// blockIdx.x) and passes each index, then a final index >= total, through the ring; the act
// producer warps, the MMA thread and the epilogue warps read them in the same order.
struct TileCursor {
    int i = 0;
    uint32_t ph = 0;
};

template <int kMode>
__device__ __forceinline__ bool tile_publish(Tail<kMode>& t, TileCursor& c, int L)
{
    if (!ptx::mbar_wait(&t.tile_empty[c.i], c.ph ^ 1)) return false;
    t.tile_L[c.i] = L;
    ptx::mbar_arrive(&t.tile_full[c.i]);
    if (++c.i == kTileRing) { c.i = 0; c.ph ^= 1; }
    return true;
}

// Warp-wide (all lanes of the calling warp, or a single thread with one_thread); returns total
// when the wait runs out.
template <int kMode>
__device__ __forceinline__ int tile_take(Tail<kMode>& t, TileCursor& c, int total, bool one_thread)
{
    int L = total;
    const bool got = ptx::mbar_wait(&t.tile_full[c.i], c.ph);
    if (got) L = *reinterpret_cast<const volatile int32_t*>(&t.tile_L[c.i]);
    if (!one_thread) __syncwarp();
    if (one_thread || (threadIdx.x & 31) == 0) ptx::mbar_arrive(&t.tile_empty[c.i]);
    if (++c.i == kTileRing) { c.i = 0; c.ph ^= 1; }
    return got ? L : total;
}

__device__ __forceinline__ int ld_acquire(const int32_t* p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait (bounded by limit_ns) until *p >= target; false on timeout.
__device__ __forceinline__ bool spin_until(const int32_t* p, int target, uint64_t limit_ns)
{
    if (ld_acquire(p) >= target) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (ld_acquire(p) < target) {
        if (ptx::globaltimer() - t0 > limit_ns) return false;
        __nanosleep(64);
    }
    return true;
}

__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Barriers of the epilogue warps alone (named barriers 1 and 2, 32 * n threads): the first also
// returns whether any of them passed true.
__device__ __forceinline__ bool epi_bar_any(bool pred, int n)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(32 * n)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void epi_bar(int n) { asm volatile("bar.sync 2, %0;" ::"r"(32 * n) : "memory"); }

// 8 x 8 transpose of 16-byte chunks within each group of 8 lanes (three butterfly exchanges): lane
// 8g + i holds chunks 0..7 of its own row on entry and chunk i of the group's rows 0..7 on return, so
// the group can store one row's 128 contiguous bytes per instruction (a warp: 4 rows x 128 bytes,
// whole sectors) instead of 32 rows x 16 bytes. Every lane of the warp must call it.
__device__ __forceinline__ void transpose_chunks8(uint4 (&x)[8], int lane)
{
#pragma unroll
    for (int b = 4; b >= 1; b >>= 1) {
        const bool hi = (lane & b) != 0;
#pragma unroll
        for (int c0 = 0; c0 < 8; ++c0) {
            if (c0 & b) continue;
            const int c1 = c0 | b;
            const uint4 snd = hi ? x[c0] : x[c1];
            uint4 rcv;
            rcv.x = __shfl_xor_sync(0xFFFFFFFFu, snd.x, b);
            rcv.y = __shfl_xor_sync(0xFFFFFFFFu, snd.y, b);
            rcv.z = __shfl_xor_sync(0xFFFFFFFFu, snd.z, b);
            rcv.w = __shfl_xor_sync(0xFFFFFFFFu, snd.w, b);
            if (hi) x[c0] = rcv;
            else x[c1] = rcv;
        }
    }
}

// Store a warp's 32 rows x 128 bytes through transpose_chunks8: chunk c of lane l's row goes to
// dst(l) + 16 c bytes; rows whose lane has valid == false are skipped.
__device__ __forceinline__ void store_rows128(uint4 (&x)[8], uint8_t* dst, bool valid, int lane)
{
    transpose_chunks8(x, lane);
    const int g0 = lane & ~7, ci = lane & 7;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint8_t* d = reinterpret_cast<uint8_t*>(__shfl_sync(0xFFFFFFFFu, reinterpret_cast<uintptr_t>(dst), g0 + j));
        if (__shfl_sync(0xFFFFFFFFu, valid, g0 + j)) *reinterpret_cast<uint4*>(d + ci * 16) = x[j];
    }
}

// NVFP4 encoding of the intermediate h (16 values, static tensor scale S): the same rule as the
// activation quantizer, with the two divisions replaced by multiplications with correctly rounded
// reciprocals (the requantised intermediate is compared by agreement rate, not bit for bit).
__device__ __forceinline__ uint32_t encode16_rcp(const float (&v)[16], float S, float inv_six_s, uint32_t& lo,
                                                 uint32_t& hi)
{
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const uint32_t sf = ptx::cvt_e4m3x2(amax * inv_six_s, 0.0f) & 0xFFu;
    const float dsf = ue4m3_to_f32(sf);
    lo = 0u;
    hi = 0u;
    if (dsf != 0.0f) {
        const float r = __frcp_rn(dsf * S);
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            lo |= ptx::cvt_e2m1x2(v[i] * r, v[i + 1] * r) << (4 * i);
            hi |= ptx::cvt_e2m1x2(v[8 + i] * r, v[8 + i + 1] * r) << (4 * i);
        }
    }
    return sf;
}

}  // namespace

template <int kMode>
__global__ void __launch_bounds__(Lay<kMode>::THREADS, 1)
    k_grouped_gemm_nvf4(const __grid_constant__ CUtensorMap tmap_w0, const __grid_constant__ CUtensorMap tmap_w1,
                        const __grid_constant__ CUtensorMap tmap_a0, const __grid_constant__ CUtensorMap tmap_a1,
                        const GemmArgs a)
{
    using C = Cfg<kMode>;
    using LY = Lay<kMode>;
    constexpr bool kSwap = C::SWAP;
    constexpr int W_ROWS = C::W_ROWS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Tail<kMode>& st = *reinterpret_cast<Tail<kMode>*>(smem + LY::TAIL_OFF);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

    // ---- setup
    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            ptx::mbar_init(&st.full[s], C::WRES ? kNumActProducers : 1 + kNumActProducers);
            ptx::mbar_init(&st.empty[s], LY::MMA_THREADS);  // one commit per MMA thread
        }
        for (int i = 0; i < LY::MAX_SLABS; ++i) {
            ptx::mbar_init(&st.r_full[i], 1);
            ptx::mbar_init(&st.r_empty[i], 1);
        }
        for (int s = 0; s < C::ACC_BUFS; ++s) {
            ptx::mbar_init(&st.acc_full[s], LY::MMA_THREADS);
            ptx::mbar_init(&st.acc_empty[s], 32 * LY::ACC_READERS);
        }
        ptx::mbar_init(&st.drain, 1);
        ptx::mbar_init(&st.drain_b, 1);
        ptx::mbar_init(&st.xchg_full, 64);
        ptx::mbar_init(&st.xchg_empty, 64);
        for (int i = 0; i < kTileRing; ++i) {
            ptx::mbar_init(&st.tile_full[i], 1);
            ptx::mbar_init(&st.tile_empty[i], 2 + LY::MMA_THREADS + LY::EPI_ACTIVE);
        }
        st.abort = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmap_w0);
        if (a.nphase > 1) ptx::prefetch_tmap(&tmap_w1);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&st.tmem_base, LY::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    // everything above overlaps the previous launch; the group offsets and activations come from it
    ptx::griddep_wait();
    // a launch given the top-k ids builds its permutation here (stage 0's buffer is scratch until the
    // producers start): offsets straight into st.g_off, rows into rs
    RouteSmem* rs = nullptr;
    if constexpr (C::XCHG) {
        if (a.route.topk_ids) {
            rs = reinterpret_cast<RouteSmem*>(smem + LY::TAIL_OFF + sizeof(Tail<kMode>) + sizeof(AccXchg));
            int32_t* ids_s = reinterpret_cast<int32_t*>(smem);          // n + 4 (padded to 16 bytes)
            int32_t* sorted_s = ids_s + kRouteMaxAssign + 4;             // n
            const int n = a.route.T * a.route.k;
            for (int i = tid; i < n + 4; i += LY::THREADS) ids_s[i] = i < n ? a.route.topk_ids[i] : INT_MAX;
            __syncthreads();
            block_small_permute<LY::THREADS>(ids_s, n, a.route.k, a.route.T, a.route.E, sorted_s, st.g_off, rs->perm,
                                             nullptr, rs->row);
            __syncthreads();
        }
    }
    block_tile_prefix(rs ? st.g_off : a.offsets, a.G, C::ACT_ROWS, st.tb_off, st.g_off, st.wsum);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = st.tmem_base;

    if constexpr (C::WRES) {
        // runs of at most kWresRun token blocks per group, counted in the units' group order
        if (warp == 0) {
            const int per = (a.G + 31) / 32;
            const int s_lo = min(a.G, lane * per), s_hi = min(a.G, s_lo + per);
            int32_t sum = 0;
            for (int q = s_lo; q < s_hi; ++q) {
                const int g = wres_group(q, a.G);
                sum += (st.tb_off[g + 1] - st.tb_off[g] + kWresRun - 1) / kWresRun;
            }
            int32_t x = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= o) x += y;
            }
            int32_t run = x - sum;
            for (int q = s_lo; q < s_hi; ++q) {
                st.ur_off[q] = run;
                const int g = wres_group(q, a.G);
                run += (st.tb_off[g + 1] - st.tb_off[g] + kWresRun - 1) / kWresRun;
            }
            if (lane == 31) st.ur_off[a.G] = x;
        }
        __syncthreads();
    }
    const int nblk = st.tb_off[a.G];
    // the launch's work items: tiles (token block x weight block), with ROWS whole token blocks
    // ("units", each taken through every weight block of its phase), with WRES runs of token blocks
    // of one group taken through one weight block
    const int nrun = C::WRES ? st.ur_off[C::WRES ? a.G : 0] : 0;
    const int tiles0 = C::ROWS ? nblk : (C::WRES ? nrun : nblk) * (a.p[0].N / W_ROWS);
    const int total = tiles0 + (a.nphase > 1 ? (C::ROWS ? nblk : (C::WRES ? nrun : nblk) * (a.p[1].N / W_ROWS)) : 0);
    auto tile_at = [&](int L) -> TileInfo {
        if constexpr (C::ROWS) return unit_info(st.tb_off, st.g_off, a, C::ACT_ROWS, tiles0, L);
        else if constexpr (C::WRES) return wres_unit_info(st.tb_off, st.g_off, st.ur_off, a, tiles0, L);
        else return tile_info(st.tb_off, st.g_off, a, C::ACT_ROWS, W_ROWS, tiles0, L);
    };
    // the tiles a work item runs through: weight blocks (ROWS), token blocks (WRES)
    auto n_sub = [&](const TileInfo& t) { return C::ROWS ? a.p[t.ph].N / W_ROWS : t.nbk; };
    // tile sub of work item t (WRES: the sub-th token block of the run)
    auto sub_tile = [&](const TileInfo& t, int sub) {
        TileInfo ti = t;
        if constexpr (C::ROWS) ti.nb = sub;
        if constexpr (C::WRES) {
            ti.tbg = t.tbg + sub;
            ti.row0 = t.row0 + sub * C::ACT_ROWS;
            ti.rows = min(C::ACT_ROWS, st.g_off[t.g + 1] - ti.row0);
        }
        return ti;
    };

    if (warp == 0 && !C::SPLIT) {
        // ================================ weight producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, rph = 0;  // rph: phase bit of each resident slab's free barrier
            uint32_t fills = 0, rfilled = 0;  // stage fills issued; resident slabs ever filled
            bool ok = true;
            // tiles in the order the CTAs come for them (phase-0 tiles first): a CTA whose tiles
            // run short takes more, and the down tiles go out in the order their inputs complete
            TileCursor tc;
            int L = blockIdx.x;
            while (ok && !aborted(st)) {
                if (L > total) L = total;
                if (!tile_publish(st, tc, L)) { set_abort(st, a.status); break; }
                if (L >= total) {
                    // this CTA's last tile is loading: the next launch may be scheduled (its CTAs
                    // start as SMs free up; its dependent reads wait for this grid to complete)
                    ptx::griddep_launch_dependents();
                    break;
                }
                // claim the next tile now: the atomic's round trip overlaps this tile's stages
                // instead of stalling the ring between tiles (a phase-1 tile is never followed by a
                // phase-0 claim, so no CTA holds back a tile another CTA waits for)
                const int L_next = static_cast<int>(gridDim.x) + atomicAdd(a.tile_counter, 1);
                const TileInfo ti = tile_at(L);
                const GemmProblem& P = a.p[ti.ph];
                const CUtensorMap* tm = ti.ph ? &tmap_w1 : &tmap_w0;
                const int kb64 = P.K / 64, k_stages = (P.K + 255) / 256, n_blk = P.N / 128;
                if constexpr (C::WRES) {
                    // the unit's weight block, slab by slab, into the resident region as the last
                    // token block of the previous unit frees each slab
                    const uint8_t* sf_src = P.b_sf + ((static_cast<int64_t>(ti.g) * n_blk + ti.nb) * kb64) * SF_TILE;
                    for (int kt = 0; kt < k_stages; ++kt) {
                        if (!ptx::mbar_wait(&st.r_empty[kt], ((rph >> kt) & 1u) ^ 1u)) { set_abort(st, a.status); ok = false; break; }
                        rph ^= 1u << kt;
                        rfilled |= 1u << kt;
                        const int nat = min(4, kb64 - kt * 4);
                        ptx::mbar_arrive_expect_tx(&st.r_full[kt], LY::W_BYTES + nat * SF_TILE);
                        ptx::tma_load_3d(smem + LY::B_OFF + kt * LY::W_BYTES, tm, &st.r_full[kt], 0, ti.nb * W_ROWS,
                                         ti.g * k_stages + kt);
                        ptx::bulk_load(smem + LY::B_SF_OFF + kt * SF_STAGE, sf_src + static_cast<int64_t>(kt) * 4 * SF_TILE,
                                       nat * SF_TILE, &st.r_full[kt]);
                    }
                    L = L_next;
                    continue;
                }
                for (int sub = 0; ok && sub < n_sub(ti); ++sub) {
                    const int nb = C::ROWS ? sub : ti.nb;
                    // scale tiles of the tile's 128-row weight blocks: [G][N/128][K/64][512 bytes]
                    const uint8_t* sf_src = P.b_sf + ((static_cast<int64_t>(ti.g) * n_blk + nb * LY::WB) * kb64) * SF_TILE;
                    const int row = nb * W_ROWS;
                    for (int kt = 0; kt < k_stages; ++kt) {
                        if (!ptx::mbar_wait(&st.empty[s], ph ^ 1)) { set_abort(st, a.status); ok = false; break; }
                        uint8_t* sbase = smem + s * LY::STAGE_BYTES;
                        const int nat = min(4, kb64 - kt * 4);
                        ptx::mbar_arrive_expect_tx(&st.full[s], LY::W_BYTES + LY::WB * nat * SF_TILE);
                        ptx::tma_load_3d(sbase + LY::OFF_W, tm, &st.full[s], 0, row, ti.g * k_stages + kt);
#pragma unroll
                        for (int j = 0; j < LY::WB; ++j)
                            ptx::bulk_load(sbase + LY::OFF_SFW + j * SF_STAGE, sf_src + static_cast<int64_t>(j) * kb64 * SF_TILE,
                                           nat * SF_TILE, &st.full[s]);
                        sf_src += 4 * SF_TILE;
                        ++fills;
                        if (++s == C::STAGES) { s = 0; ph ^= 1; }
                    }
                }
                L = L_next;
            }
            // no copy of this thread writes shared memory after the CTA exits: every stage's and
            // resident slab's last fill has landed (at once on the normal path, where all were consumed)
            bool drained = ptx::ring_drain(st.full, C::STAGES, fills);
            for (int kt = 0; kt < 8; ++kt)
                if ((rfilled >> kt) & 1u) drained = ptx::mbar_wait(&st.r_full[kt], ((rph >> kt) & 1u) ^ 1u) && drained;
            if (!drained) set_abort(st, a.status);
        }
    } else if (warp == 1 || (C::SPLIT && warp == 0)) {
        // ================================ MMA issuer(s)
        if constexpr (C::WRES) {
            if (lane == 0) {
                // Weight-resident units: per token block of the run, K-stage by K-stage, the
                // activations' scale tile of each K-step into tensor memory and one 128 x 128 x 64 MMA
                // of the stage's activation rows against the resident slab kt. The first token block
                // also waits for each weight slab and copies its scales into tensor memory (kept for
                // the run's other blocks); the last one commits each slab free once its MMAs are
                // issued, so the next unit's load of that slab overlaps the remaining slabs.
                const uint32_t idesc = ptx::idesc_nvf4(C::MMA_M, C::MMA_N);
                const uint32_t s0 = ptx::smem_u32(smem);
                const uint64_t dact0 = ptx::sdesc_sw128(s0 + LY::OFF_ACT), dsfa0 = ptx::sdesc_sf(s0 + LY::OFF_SFACT);
                const uint64_t dw0 = ptx::sdesc_sw128(s0 + LY::B_OFF), dsfw0 = ptx::sdesc_sf(s0 + LY::B_SF_OFF);
                constexpr uint64_t kStageAdv = LY::STAGE_BYTES >> 4, kOpAdv = 32 >> 4, kSfAdv = SF_TILE >> 4;
                constexpr uint64_t kSlabAdv = LY::W_BYTES >> 4, kSfSlabAdv = SF_STAGE >> 4;
                int s = 0;
                uint32_t ph = 0, lt = 0, rph = 0;  // rph: phase bit of each slab's load barrier
                bool ok = true;
                TileCursor tc;
                for (;;) {
                    const int L = tile_take(st, tc, total, true);
                    if (L >= total || aborted(st)) break;
                    const TileInfo tu = tile_at(L);
                    const int kK = a.p[tu.ph].K;
                    const int kb64 = kK / 64, k_stages = (kK + 255) / 256;
                    const int nsub = tu.nbk;
                    for (int sub = 0; ok && sub < nsub; ++sub, ++lt) {
                        const uint32_t as = lt % C::ACC_BUFS, acc_ph = (lt / C::ACC_BUFS) & 1;
                        if (!ptx::mbar_wait(&st.acc_empty[as], acc_ph ^ 1)) { set_abort(st, a.status); ok = false; break; }
                        ptx::tc_fence_after();
                        const uint32_t d_tmem = tmem + as * C::ACC_COLS;
                        uint32_t acc = 0;
                        for (int kt = 0; kt < k_stages; ++kt) {
                            if (!ptx::mbar_wait(&st.full[s], ph)) { set_abort(st, a.status); ok = false; break; }
                            ptx::fence_proxy_async_smem();  // the stage's rows came by cp.async (generic proxy)
                            if (sub == 0) {
                                if (!ptx::mbar_wait(&st.r_full[kt], (rph >> kt) & 1u)) { set_abort(st, a.status); ok = false; break; }
                                rph ^= 1u << kt;
                            }
                            const uint64_t so = static_cast<uint64_t>(s) * kStageAdv;
                            const uint64_t sw = static_cast<uint64_t>(kt) * kSlabAdv;
                            const uint32_t tsfa = tmem + LY::SF_COL + s * LY::STAGE_SF_COLS;
                            const int nk = min(4, kb64 - kt * 4);
                            auto kstep = [&](int kk) {
                                const uint32_t ta = tsfa + kk * 4;
                                const uint32_t tw = tmem + LY::RES_SF_COL + (kt * 4 + kk) * 4;
                                ptx::tmem_cp_32x128b_x4(ta, dsfa0 + so + kk * kSfAdv);
                                if (sub == 0) ptx::tmem_cp_32x128b_x4(tw, dsfw0 + kt * kSfSlabAdv + kk * kSfAdv);
                                ptx::mma_nvf4(d_tmem, dact0 + so + kk * kOpAdv, dw0 + sw + kk * kOpAdv, idesc, ta, tw, acc);
                                acc = 1;
                            };
                            if (nk == 4) {
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk) kstep(kk);
                            } else {
                                for (int kk = 0; kk < nk; ++kk) kstep(kk);
                            }
                            ptx::tc_commit(&st.empty[s]);
                            if (sub == nsub - 1) ptx::tc_commit(&st.r_empty[kt]);
                            if (++s == C::STAGES) { s = 0; ph ^= 1; }
                        }
                        if (!ok) break;
                        ptx::tc_commit(&st.acc_full[as]);
                    }
                    if (!ok) break;
                }
                ptx::tc_commit(&st.drain);
                if (!ptx::mbar_wait(&st.drain, 0)) set_abort(st, a.status);
            }
        } else if (lane == 0) {
            // SPLIT: two MMA threads (warp 1: weight rows 0..127 of the tile, warp 0: rows 128..255),
            // each issuing 128 x 128 x 64 MMAs into its half of the accumulator columns with its own
            // weight scale copy per K-step. A thread's tensor-core operations run one after another,
            // each taking about as long whatever its N, while two threads' operations overlap:
            // one K-step of the 256-row tile took 355 cycles from one thread (two scale copies and a
            // 128 x 256 MMA) and 204 from two (one copy and a 128 x 128 MMA each). Both threads copy
            // the activation scales into the same columns (identical bytes); the columns are not
            // rewritten before every operation that reads them has completed (stage slots: the empty
            // barrier counts both threads' commits; resident unit scales: the accumulator barrier).
            const int half = (C::SPLIT && warp != 1) ? 1 : 0;
            constexpr int N_MMA = C::SPLIT ? C::MMA_N / 2 : C::MMA_N;
            const uint32_t idesc = ptx::idesc_nvf4(C::MMA_M, N_MMA);
            // descriptors of stage 0; stage s adds s * STAGE_BYTES to the start address field and
            // K-step kk adds 32 bytes (operands) or one 512-byte scale tile
            const uint32_t s0 = ptx::smem_u32(smem);
            const uint64_t dw0 = ptx::sdesc_sw128(s0 + LY::OFF_W + half * N_MMA * BK_BYTES);
            const uint64_t dact0 = ptx::sdesc_sw128(s0 + LY::OFF_ACT);
            const uint64_t dsfw0 = ptx::sdesc_sf(s0 + LY::OFF_SFW), dsfact0 = ptx::sdesc_sf(s0 + LY::OFF_SFACT);
            constexpr uint64_t kStageAdv = LY::STAGE_BYTES >> 4, kOpAdv = 32 >> 4, kSfAdv = SF_TILE >> 4;
            int s = 0;
            uint32_t ph = 0, lt = 0;
            bool ok = true;
            TileCursor tc;
            for (;;) {
                const int L = tile_take(st, tc, total, true);
                if (L >= total || aborted(st)) break;
                const int uph = L >= tiles0 ? 1 : 0;
                const int kK = a.p[uph].K;
                const int kb64 = kK / 64, k_stages = (kK + 255) / 256;
                const int nsub = C::ROWS ? a.p[uph].N / W_ROWS : 1;
                for (int sub = 0; ok && sub < nsub; ++sub, ++lt) {
                    const uint32_t as = lt % C::ACC_BUFS, aph = (lt / C::ACC_BUFS) & 1;
                    if (!ptx::mbar_wait(&st.acc_empty[as], aph ^ 1)) { set_abort(st, a.status); ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem + as * C::ACC_COLS + half * N_MMA;
                    uint32_t acc = 0;
                    // one K-step: the scale tiles into tensor memory, then the MMA (the tensor pipe runs
                    // them in issue order); full stages take a straight-line path. Weight rows
                    // 128..255 of a 256-row tile have their scale tile in the next four columns. Units
                    // keep the activation scales of K-step kg in columns SFA_COL + 4 kg, copied during
                    // the first weight block.
                    auto kstep = [&](uint64_t so, uint32_t tsfw, uint32_t tsfact, int kk, int kg) {
                        const uint32_t tw = tsfw + kk * LY::SFW_STEP_COLS;
                        if constexpr (C::SPLIT) {
                            ptx::tmem_cp_32x128b_x4(tw + half * 4, dsfw0 + so + kk * kSfAdv + half * (SF_STAGE >> 4));
                        } else {
#pragma unroll
                            for (int j = 0; j < LY::WB; ++j)
                                ptx::tmem_cp_32x128b_x4(tw + j * 4, dsfw0 + so + kk * kSfAdv + j * (SF_STAGE >> 4));
                        }
                        uint32_t tsa;
                        if constexpr (C::ROWS) {
                            tsa = tmem + LY::RES_SF_COL + kg * 4;
                            if (sub == 0) ptx::tmem_cp_32x128b_x4(tsa, dsfact0 + so + kk * kSfAdv);
                        } else {
                            tsa = tsfact + kk * 4;
                            ptx::tmem_cp_32x128b_x4(tsa, dsfact0 + so + kk * kSfAdv);
                        }
                        const uint64_t dw = dw0 + so + kk * kOpAdv, dact = dact0 + so + kk * kOpAdv;
                        if (kSwap)
                            ptx::mma_nvf4(d_tmem, dw, dact, idesc, tw, tsa, acc);
                        else
                            ptx::mma_nvf4(d_tmem, dact, dw, idesc, tsa, tw + half * 4, acc);
                        acc = 1;
                    };
                    for (int kt = 0; kt < k_stages; ++kt) {
                        if (!ptx::mbar_wait(&st.full[s], ph)) { set_abort(st, a.status); ok = false; break; }
                        // the activation rows came by cp.async (generic proxy); with published stages
                        // (32-row blocks) the producers fenced them before arriving
                        if constexpr (!LY::PUBLISH) ptx::fence_proxy_async_smem();
                        const uint64_t so = static_cast<uint64_t>(s) * kStageAdv;
                        const uint32_t tsfw = tmem + LY::SF_COL + s * LY::STAGE_SF_COLS, tsfact = tsfw + 4 * LY::SFW_STEP_COLS;
                        const int nk = min(4, kb64 - kt * 4);
                        if (nk == 4) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) kstep(so, tsfw, tsfact, kk, kt * 4 + kk);
                        } else {
                            for (int kk = 0; kk < nk; ++kk) kstep(so, tsfw, tsfact, kk, kt * 4 + kk);
                        }
                        ptx::tc_commit(&st.empty[s]);
                        if (++s == C::STAGES) { s = 0; ph ^= 1; }
                    }
                    if (!ok) break;
                    ptx::tc_commit(&st.acc_full[as]);
                }
                if (!ok) break;
            }
            // every issued tensor-core operation finishes before TMEM is freed
            uint64_t* drain = half ? &st.drain_b : &st.drain;
            ptx::tc_commit(drain);
            if (!ptx::mbar_wait(drain, 0)) set_abort(st, a.status);
        }
    } else if (warp < 4) {
        // ================================ activation producers (row gather)
        // Warp w2 = warp - 2 fills rows [w2 * RW, w2 * RW + RW) of the tile. Lanes run along rows:
        // 8 lanes copy the 8 16-byte chunks of one row's 128-byte K-slice (one cache line), 4 lanes
        // the 4 scale words of one row, so each warp instruction touches few cache lines. Scales
        // stored in token-block tiles are copied as whole 512-byte tiles (both warps share them).
        constexpr int RW = C::ACT_ROWS / 2;      // rows per producer warp
        constexpr int NCR = RW / 4;              // code rows per lane (4 rows per warp instruction)
        constexpr int NSR = RW / 8;              // scale rows per lane (8 rows per warp instruction)
        // Each thread arrives on a stage's full barrier through cp.async.mbarrier.arrive: the arrival
        // lands when the thread's copies have, so the warp goes straight on to the next free stage
        // and as many stages' gathers are in flight as the ring has free slots. (The MMA thread
        // fences the generic-proxy writes of the copies against its tensor-core reads.)
        // With 32-row token blocks (decode) the copies are few and a stage instead is published by
        // the warp itself, once its copies have landed and one newer stage is issued (LAG): that
        // measured 0.4 us faster per decode launch, and a deeper lag holds each stage back until
        // LAG more slots are free (2 us slower at 3 than at 1). Every issued stage is published
        // before a wait on another CTA's h, which may be waiting for the tile those stages complete.
        constexpr int LAG = 1;
        int pub = 0;
        uint32_t issued = 0, published = 0;
        auto publish_all = [&]() {
            ptx::cp_async_wait<0>();
            ptx::fence_proxy_async_smem();
            for (; published < issued; ++published) {
                ptx::mbar_arrive(&st.full[pub]);
                if (++pub == C::STAGES) pub = 0;
            }
        };
        const int w2 = warp - 2, pt = tid - 64;
        const int chunk = lane & 7, word = lane & 3;
        // the wait for a token block's h: default limit, unless a test set the workspace hooks
        uint64_t ready_limit_ns = ptx::kWaitLimitNs;
        int ready_extra = 0;
        if (a.hooks) {
            const unsigned us = *reinterpret_cast<const volatile unsigned*>(&a.hooks->test_wait_us);
            ready_extra = *reinterpret_cast<const volatile int*>(&a.hooks->test_ready_extra);
            if (us) ready_limit_ns = static_cast<uint64_t>(us) * 1000u;
        }
        const uint8_t* cptr[NCR];
        const uint8_t* sptr[NSR];
        uint32_t cvalid = 0, svalid = 0;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        TileCursor tc;
        // SPLIT: lane 0 of the first producer warp is the weight producer too. It claims the tiles
        // (in the order the CTAs come for them, phase-0 tiles first, so a CTA whose tiles run short
        // takes more and the down tiles go out in the order their inputs complete), publishes each
        // one before taking it back from the ring, and loads each stage's weight box and weight scale
        // tiles once the stage is free.
        const bool wprod = C::SPLIT && warp == 2 && lane == 0;
        int Lw = blockIdx.x;
        bool w_done = false;
        TileCursor tcw;
        uint32_t fills = 0;
        for (;;) {
            if (wprod && !w_done) {
                if (Lw > total) Lw = total;
                if (!tile_publish(st, tcw, Lw)) {
                    set_abort(st, a.status);
                    w_done = true;
                } else if (Lw >= total) {
                    // this CTA's last tile is loading: the next launch may be scheduled (its CTAs
                    // start as SMs free up; its dependent reads wait for this grid to complete)
                    ptx::griddep_launch_dependents();
                    w_done = true;
                }
            }
            // the next claim's round trip overlaps this tile's stages
            const int Lw_next = (wprod && !w_done) ? static_cast<int>(gridDim.x) + atomicAdd(a.tile_counter, 1) : total;
            const int L = tile_take(st, tc, total, false);
            if (L >= total || !ok || aborted(st)) break;
            Lw = Lw_next;
            const TileInfo tu = tile_at(L);
            const GemmProblem& P = a.p[tu.ph];
            const int64_t a_ld = P.K / 2, sf_ld = P.K / 16;
            const int kb64 = P.K / 64, k_stages = (P.K + 255) / 256;
            const uint8_t* sf_tiles = nullptr;
            // (units: the activation scales go with the first weight block only; the MMA thread
            // keeps them in tensor memory for the others. Weight-resident units run through several
            // token blocks, each with its own rows.)
            for (int sub = 0; ok && sub < n_sub(tu); ++sub) {
                const TileInfo ti = sub_tile(tu, sub);
                if (C::SPLIT && a.a_tma[tu.ph]) {
                    // contiguous activation rows with scales in token-block tiles: the weight-producing
                    // lane loads each stage's 128 rows as one TMA box (rows past the end read as
                    // zeros) and the stage's scale tiles as one bulk copy, with the weights
                    if (sub == 0 && ti.ph == 1) {
                        const int target = LY::READY_PER_TILE * (a.p[0].N / W_ROWS) + ready_extra;
                        if (!spin_until(a.ready + ti.tbg, target, ready_limit_ns)) { set_abort(st, a.status); ok = false; break; }
                        // h, stored by other threads' generic stores, is then read by this lane's copies
                        if (wprod) ptx::fence_proxy_async_global();
                    }
                    const uint8_t* act_sf = P.a_sf + static_cast<int64_t>(ti.tbg) * kb64 * SF_TILE;
                    for (int kt = 0; kt < k_stages; ++kt) {
                        if (!ptx::mbar_wait(&st.empty[s], ph ^ 1)) { set_abort(st, a.status); ok = false; break; }
                        if (wprod) {
                            const int nat = min(4, kb64 - kt * 4);
                            const bool sf_copy = !C::ROWS || sub == 0;
                            uint8_t* sbase = smem + s * LY::STAGE_BYTES;
                            ptx::mbar_arrive_expect_tx(&st.full[s], LY::W_BYTES + LY::WB * nat * SF_TILE + LY::ACT_BYTES +
                                                                        (sf_copy ? nat * SF_TILE : 0));
                            ptx::tma_load_3d(sbase + LY::OFF_W, ti.ph ? &tmap_w1 : &tmap_w0, &st.full[s], 0, ti.nb * W_ROWS,
                                             ti.g * k_stages + kt);
                            const uint8_t* sfw =
                                P.b_sf + ((static_cast<int64_t>(ti.g) * (P.N / 128) + ti.nb * LY::WB) * kb64 + kt * 4) * SF_TILE;
#pragma unroll
                            for (int j = 0; j < LY::WB; ++j)
                                ptx::bulk_load(sbase + LY::OFF_SFW + j * SF_STAGE, sfw + static_cast<int64_t>(j) * kb64 * SF_TILE,
                                               nat * SF_TILE, &st.full[s]);
                            ptx::tma_load_3d(sbase + LY::OFF_ACT, ti.ph ? &tmap_a1 : &tmap_a0, &st.full[s], kt * BK_BYTES,
                                             static_cast<int32_t>(ti.row0), 0);
                            if (sf_copy)
                                ptx::bulk_load(sbase + LY::OFF_SFACT, act_sf + static_cast<int64_t>(kt) * 4 * SF_TILE,
                                               nat * SF_TILE, &st.full[s]);
                            ++fills;
                        }
                        ptx::mbar_arrive(&st.full[s]);  // this thread's arrival (it copied nothing)
                        if (++s == C::STAGES) { s = 0; ph ^= 1; }
                    }
                    continue;
                }
                if (sub == 0 || C::WRES) {
                    if (ti.ph == 1) {
                        // the down GEMM reads h: wait until every gate/up tile of this token block stored
                        // it (the stages already issued complete on their own meanwhile)
                        if constexpr (LY::PUBLISH) publish_all();
                        const int target = LY::READY_PER_TILE * (a.p[0].N / W_ROWS) + ready_extra;
                        if (!spin_until(a.ready + ti.tbg, target, ready_limit_ns)) { set_abort(st, a.status); ok = false; break; }
                    }
                    // source row of tile rows w2*RW + lane (+ 32): one gather-index load per row (a
                    // launch that permutes itself has the gate/up rows in shared memory)
                    const int32_t* a_row = rs && ti.ph == 0 ? rs->row : P.a_row;
                    int64_t srcv[(RW + 31) / 32];
#pragma unroll
                    for (int h = 0; h < (RW + 31) / 32; ++h) {
                        const int r = w2 * RW + h * 32 + lane;
                        const int64_t p = ti.row0 + r;
                        srcv[h] = (h * 32 + lane < RW && r < ti.rows) ? (a_row ? static_cast<int64_t>(a_row[p]) : p) : -1;
                    }
                    cvalid = 0;
                    svalid = 0;
#pragma unroll
                    for (int i = 0; i < NCR; ++i) {
                        const int rl = i * 4 + (lane >> 3);  // row within this warp's slice (same word of srcv in all lanes)
                        const int64_t src = __shfl_sync(0xFFFFFFFFu, srcv[rl >> 5], rl & 31);
                        cptr[i] = src >= 0 ? P.a_codes + src * a_ld + chunk * 16 : P.a_codes;
                        if (src >= 0) cvalid |= 1u << i;
                    }
#pragma unroll
                    for (int i = 0; i < NSR; ++i) {
                        const int rl = i * 8 + (lane >> 2);
                        const int64_t src = __shfl_sync(0xFFFFFFFFu, srcv[rl >> 5], rl & 31);
                        sptr[i] = src >= 0 ? P.a_sf + src * sf_ld + word * 4 : P.a_sf;
                        if (src >= 0) svalid |= 1u << i;
                    }
                    sf_tiles = P.a_sf + static_cast<int64_t>(ti.tbg) * kb64 * SF_TILE;
                }
                for (int kt = 0; kt < k_stages; ++kt) {
                    if (!ptx::mbar_wait(&st.empty[s], ph ^ 1)) { set_abort(st, a.status); ok = false; break; }
                    if (wprod) {
                        // the weight box (TMA) and the weight scale tiles of this stage:
                        // scale tiles are stored [G][N/128][K/64][512 bytes]
                        const int nat = min(4, kb64 - kt * 4);
                        uint8_t* sbase = smem + s * LY::STAGE_BYTES;
                        ptx::mbar_arrive_expect_tx(&st.full[s], LY::W_BYTES + LY::WB * nat * SF_TILE);
                        ptx::tma_load_3d(sbase + LY::OFF_W, ti.ph ? &tmap_w1 : &tmap_w0, &st.full[s], 0, ti.nb * W_ROWS,
                                         ti.g * k_stages + kt);
                        const uint8_t* sfw =
                            P.b_sf + ((static_cast<int64_t>(ti.g) * (P.N / 128) + ti.nb * LY::WB) * kb64 + kt * 4) * SF_TILE;
#pragma unroll
                        for (int j = 0; j < LY::WB; ++j)
                            ptx::bulk_load(sbase + LY::OFF_SFW + j * SF_STAGE, sfw + static_cast<int64_t>(j) * kb64 * SF_TILE,
                                           nat * SF_TILE, &st.full[s]);
                        ++fills;
                    }
                    uint8_t* sact = smem + s * LY::STAGE_BYTES + LY::OFF_ACT;
                    uint8_t* ssf = smem + s * LY::STAGE_BYTES + LY::OFF_SFACT;
                    const bool kin = static_cast<int64_t>(kt) * BK_BYTES + chunk * 16 < a_ld;
#pragma unroll
                    for (int i = 0; i < NCR; ++i) {
                        const int r = w2 * RW + i * 4 + (lane >> 3);
                        const bool v = ((cvalid >> i) & 1u) && kin;
                        ptx::cp_async_16(sact + r * 128 + ((chunk ^ (r & 7)) * 16), v ? cptr[i] + kt * BK_BYTES : P.a_codes, v);
                    }
                    if (C::ROWS && sub > 0) {
                    } else if (P.a_sf_tiled) {
                        // the stage's (up to) 4 scale tiles, 32 lines x 16 bytes each, 2 copies per thread
                        const int nat = min(4, kb64 - kt * 4);
#pragma unroll
                        for (int c = pt; c < 4 * 32; c += kNumActProducers) {
                            const int j = c >> 5, line = c & 31;
                            const bool v = j < nat;
                            ptx::cp_async_16(ssf + j * SF_TILE + line * 16,
                                             v ? sf_tiles + (static_cast<int64_t>(kt) * 4 + j) * SF_TILE + line * 16 : P.a_sf, v);
                        }
                    } else {
                        const bool kin_s = static_cast<int64_t>(kt) * 16 + word * 4 < sf_ld;
#pragma unroll
                        for (int i = 0; i < NSR; ++i) {
                            const int r = w2 * RW + i * 8 + (lane >> 2);
                            const bool v = ((svalid >> i) & 1u) && kin_s;
                            ptx::cp_async_4(ssf + word * SF_TILE + (r % 32) * 16 + (r / 32) * 4, v ? sptr[i] + kt * 16 : P.a_sf, v);
                        }
                    }
                    if constexpr (LY::PUBLISH) {
                        ptx::cp_async_commit();
                        ++issued;
                        ptx::cp_async_wait<LAG>();
                        if (issued > published + LAG) {
                            ptx::fence_proxy_async_smem();
                            for (; published + LAG < issued; ++published) {
                                ptx::mbar_arrive(&st.full[pub]);
                                if (++pub == C::STAGES) pub = 0;
                            }
                        }
                    } else {
                        ptx::cp_async_arrive_noinc(&st.full[s]);
                    }
                    if (++s == C::STAGES) { s = 0; ph ^= 1; }
                }
            }
        }
        if constexpr (LY::PUBLISH) publish_all();
        ptx::cp_async_wait<0>();  // no copy outlives the role
        // nor a weight load: every stage's last fill has landed
        if (wprod && !ptx::ring_drain(st.full, C::STAGES, fills)) set_abort(st, a.status);
    } else if constexpr (C::XCHG) {
        // ================================ epilogue through shared memory (32-row token blocks)
        // The two warps of lane quarter 0 copy the tile's accumulator (rows 0..31) to shared memory
        // and free it; then every epilogue warp finishes a slice of it: h block ew of the SwiGLU
        // (16 gate and 16 up columns), or 32 output columns. The per-tile loop of the epilogue
        // warps is kept in step by two barriers; the first also ends it for all of them at once.
        static_assert(!kSwap && C::ACT_ROWS == 32 && W_ROWS == 256 && C::EPI_WARPS == 8, "XCHG epilogue shape");
        AccXchg& xb = *reinterpret_cast<AccXchg*>(smem + LY::TAIL_OFF + sizeof(Tail<kMode>));
        const int ew = warp - 4;
        const int q = warp & 3;
        uint32_t lt = 0;
        TileCursor tc;
        for (;; ++lt) {
            const int L = tile_take(st, tc, total, false);
            const bool have = L < total && !aborted(st);
            TileInfo ti{};
            if (have) ti = tile_at(L);
            const GemmProblem& P = a.p[ti.ph];
            const int r = lane;  // the tile row of this lane in every slice
            const int64_t p = ti.row0 + r;
            const bool valid = have && r < ti.rows;
            float sa = 1.0f, sb0 = 1.0f, sb1 = 1.0f, S_h = 1.0f;
            int64_t po = p;
            if (have) {
                sa = __ldg(P.a_scale + (P.a_scale_per_group ? ti.g : 0));
                sb0 = __ldg(P.b_scale + (P.gate_up ? 2 * ti.g : ti.g));
                sb1 = P.gate_up ? __ldg(P.b_scale + 2 * ti.g + 1) : sb0;
                S_h = P.epilogue == kEpiSwiGLU ? __ldg(P.epi_scale + ti.g) : 1.0f;
                const int32_t* out_row = rs && ti.ph == 1 ? rs->perm : P.out_row;
                if (out_row && valid && p < P.out_row_n) po = out_row[p];
            }
            bool ok = true;
            if (have && q == 0) {
                const uint32_t as = lt % C::ACC_BUFS, aph = (lt / C::ACC_BUFS) & 1;
                const bool got = ptx::mbar_wait(&st.acc_full[as], aph);
                __syncwarp();
                ok = __all_sync(0xFFFFFFFFu, got);
                if (ok) {
                    ptx::tc_fence_after();
                    const int half = ew >> 2;  // warps 4 and 8: accumulator columns half*128 .. +127
                    const uint32_t tbase = tmem + as * C::ACC_COLS + half * 128;
#pragma unroll
                    for (int rd = 0; rd < 2; ++rd) {
                        uint32_t v[4][16];
#pragma unroll
                        for (int g = 0; g < 4; ++g) ptx::tmem_ld16(tbase + rd * 64 + g * 16, v[g]);
                        ptx::tmem_ld_wait();
                        if (rd == 1) {
                            ptx::tc_fence_before();
                            ptx::mbar_arrive(&st.acc_empty[as]);
                        }
                        float4* row = reinterpret_cast<float4*>(&xb.v[lane][half * 128 + rd * 64]);
#pragma unroll
                        for (int g = 0; g < 4; ++g)
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                row[g * 4 + j] = make_float4(__uint_as_float(v[g][4 * j]), __uint_as_float(v[g][4 * j + 1]),
                                                             __uint_as_float(v[g][4 * j + 2]), __uint_as_float(v[g][4 * j + 3]));
                    }
                } else {
                    set_abort(st, a.status);
                }
            }
            if (epi_bar_any(!have || !ok, C::EPI_WARPS)) break;  // the copy is complete (or all stop)
            const float* xr = xb.v[r];
            if (P.epilogue == kEpiSwiGLU) {
                const int I = P.N / 2;
                const int beta = ew;                                 // h block of the tile
                const int gc = (beta >> 2) * 128 + (beta & 3) * 16;  // its gate columns; up at + 64
                const float sg = sa * sb0, su = sa * sb1;
                const float S = S_h;
                const float inv_six_s = 1.0f / (6.0f * S);
                float h[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 g4 = reinterpret_cast<const float4*>(xr + gc)[j];
                    const float4 u4 = reinterpret_cast<const float4*>(xr + gc + 64)[j];
                    h[4 * j] = silu(g4.x * sg) * (u4.x * su);
                    h[4 * j + 1] = silu(g4.y * sg) * (u4.y * su);
                    h[4 * j + 2] = silu(g4.z * sg) * (u4.z * su);
                    h[4 * j + 3] = silu(g4.w * sg) * (u4.w * su);
                }
                uint32_t lo, hi;
                const uint32_t sf = encode16_rcp(h, S, inv_six_s, lo, hi);
                if (valid) {
                    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(P.out) + p * (I / 2) + ti.nb * (W_ROWS / 4) + beta * 8) =
                        make_uint2(lo, hi);
                    if (P.out_sf_tiled)
                        P.out_sf[(static_cast<int64_t>(ti.tbg) * (I / 64) + ti.nb * LY::WB + (beta >> 2)) * SF_TILE + r * 16 +
                                 (beta & 3)] = static_cast<uint8_t>(sf);
                    else
                        P.out_sf[p * (I / 16) + ti.nb * (W_ROWS / 32) + beta] = static_cast<uint8_t>(sf);
                }
            } else {
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    const int c0 = ew * 32 + g * 16;  // tile column
                    int col;
                    float sb;
                    if (P.gate_up) {
                        const int cc = c0 & 127, upper = cc >= 64;
                        col = (upper ? P.N / 2 : 0) + (ti.nb * LY::WB + (c0 >> 7)) * 64 + (cc & 63);
                        sb = upper ? sb1 : sb0;
                    } else {
                        col = ti.nb * W_ROWS + c0;
                        sb = sb0;
                    }
                    const float sc = sa * sb;
                    float x[16];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 v4 = reinterpret_cast<const float4*>(xr + c0)[j];
                        x[4 * j] = v4.x * sc;
                        x[4 * j + 1] = v4.y * sc;
                        x[4 * j + 2] = v4.z * sc;
                        x[4 * j + 3] = v4.w * sc;
                    }
                    if (valid) {
                        if (P.epilogue == kEpiF32) {
                            float4* o = reinterpret_cast<float4*>(static_cast<float*>(P.out) + po * P.N + col);
#pragma unroll
                            for (int j = 0; j < 4; ++j) o[j] = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
                        } else {
                            uint32_t w[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j) w[j] = pack_bf16x2(x[2 * j], x[2 * j + 1]);
                            uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(P.out) + po * P.N + col);
                            o[0] = make_uint4(w[0], w[1], w[2], w[3]);
                            o[1] = make_uint4(w[4], w[5], w[6], w[7]);
                        }
                    }
                }
            }
            if (a.nphase > 1 && ti.ph == 0) {
                // publish this warp's part of h (see the other epilogue)
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    atomicAdd(a.ready + ti.tbg, 1);
                }
            }
            epi_bar(C::EPI_WARPS);  // every slice read: the next tile may overwrite the copy
        }
    } else {
        // ================================ epilogue
        const int ew = warp - 4;
        const int q = warp & 3;  // TMEM lane quarter of this warp
        uint32_t lt = 0, xt = 0;
        TileCursor tc;
        const bool epi_active = LY::EPI_ACTIVE == C::EPI_WARPS || q == 0;
        bool epi_ok = true;
        for (; epi_active && epi_ok;) {
            const int L = tile_take(st, tc, total, false);
            if (L >= total || aborted(st)) break;
            const TileInfo tu = tile_at(L);
            for (int sub = 0; sub < n_sub(tu); ++sub, ++lt) {
            const TileInfo ti = sub_tile(tu, sub);
            const GemmProblem& P = a.p[ti.ph];
            const uint32_t as = lt % C::ACC_BUFS, aph = (lt / C::ACC_BUFS) & 1;
            // the tile's scales are loaded before waiting for its accumulator, hiding their latency:
            // sb0 / sb1 the gate / up (or only) weight scale, S_h the tensor scale of h (SwiGLU)
            const float sa = __ldg(P.a_scale + (P.a_scale_per_group ? ti.g : 0));
            const float sb0 = __ldg(P.b_scale + (P.gate_up ? 2 * ti.g : ti.g));
            const float sb1 = P.gate_up ? __ldg(P.b_scale + 2 * ti.g + 1) : sb0;
            const float S_h = P.epilogue == kEpiSwiGLU ? __ldg(P.epi_scale + ti.g) : 1.0f;
            // output row of this lane's tile row (row r = q*32 + lane on M, or token slot = lane on N)
            int64_t po;
            {
                const int rr = kSwap ? lane : q * 32 + lane;
                const int64_t p = ti.row0 + rr;
                po = (P.out_row && rr < ti.rows && p < P.out_row_n) ? static_cast<int64_t>(__ldg(P.out_row + p)) : p;
            }
            const bool got = ptx::mbar_wait(&st.acc_full[as], aph);
            __syncwarp();
            if (!__all_sync(0xFFFFFFFFu, got)) {
                set_abort(st, a.status);
                epi_ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t tbase = tmem + as * C::ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
            const int I = P.N / 2;  // h columns (SwiGLU)
            // scale tile of h for this token block and weight block: [token block][I/64][512 bytes]
            uint8_t* hsf_tile = P.out_sf_tiled ? P.out_sf + (static_cast<int64_t>(ti.tbg) * (I / 64) + ti.nb) * SF_TILE : nullptr;
            if constexpr (!kSwap) {
                // ---- TMEM lane = token row r; columns = the tile's weight rows. The warps of lane
                // quarter q split the columns in two halves; each loads its columns, frees the
                // accumulator, then converts and stores.
                constexpr int CPW = W_ROWS / 2;  // accumulator columns per warp
                constexpr int NLD = CPW / 16;
                constexpr int NB = W_ROWS / 64;  // SwiGLU: 16-column blocks of h per warp
                const int half = ew >> 2;
                const int r = q * 32 + lane;
                const bool valid = r < ti.rows;
                const bool any = q * 32 < ti.rows;  // warp-uniform: the quarter holds rows of the tile
                const int64_t p = ti.row0 + r;
                const bool swiglu = P.epilogue == kEpiSwiGLU;
                // The warp's columns come out of tensor memory in NR rounds of GPR 16-column groups
                // (128 columns at once would not fit in registers); the accumulator is freed right
                // after the last round's load.
                constexpr int NR = NLD > 4 ? 2 : 1;
                constexpr int GPR = NLD / NR;
                auto load_round = [&](int rd, uint32_t (&v)[GPR][16]) {
                    // SwiGLU: h block beta = half * NB + b takes gate column c*128 + jj*16 and up
                    // column + 64 (c = beta / 4, jj = beta % 4: 128-row blocks hold 64 gate then 64 up
                    // rows); otherwise the warp's columns are [half * CPW, half * CPW + CPW)
#pragma unroll
                    for (int g = 0; g < GPR; ++g) {
                        const int i = rd * GPR + g;
                        uint32_t col;
                        if (swiglu) {
                            const int beta = half * NB + (i >> 1);
                            col = (beta >> 2) * 128 + (beta & 3) * 16 + (i & 1) * 64;
                        } else {
                            col = half * CPW + i * 16;
                        }
                        ptx::tmem_ld16(tbase + col, v[g]);
                    }
                    ptx::tmem_ld_wait();
                };
                auto release = [&]() {
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(&st.acc_empty[as]);
                };
                if (any && swiglu) {
                    const float sg = sa * sb0, su = sa * sb1;
                    const float S = S_h;
                    const float inv_six_s = 1.0f / (6.0f * S);
                    constexpr int BPR = NB / NR;  // h blocks per round
                    float h[NB][16];
#pragma unroll
                    for (int rd = 0; rd < NR; ++rd) {
                        uint32_t v[GPR][16];
                        load_round(rd, v);
                        if (rd == NR - 1) release();
#pragma unroll
                        for (int bb = 0; bb < BPR; ++bb)
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                h[rd * BPR + bb][i] =
                                    silu(__uint_as_float(v[2 * bb][i]) * sg) * (__uint_as_float(v[2 * bb + 1][i]) * su);
                    }
                    uint32_t cw[2 * NB], sfw = 0;
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        uint32_t lo, hi;
                        sfw |= encode16_rcp(h[b], S, inv_six_s, lo, hi) << (8 * b);
                        cw[2 * b] = lo;
                        cw[2 * b + 1] = hi;
                    }
                    if (valid) {
                        const int beta0 = half * NB;  // first h block of this warp
                        uint8_t* hrow = static_cast<uint8_t*>(P.out) + p * (I / 2) + ti.nb * (W_ROWS / 4) + beta0 * 8;
#pragma unroll
                        for (int b = 0; b < NB; b += 2)
                            *reinterpret_cast<uint4*>(hrow + b * 8) = make_uint4(cw[2 * b], cw[2 * b + 1], cw[2 * b + 2], cw[2 * b + 3]);
                        if (P.out_sf_tiled) {
                            // tile of h's 64-column block nb * WB + beta0 / 4; the warp's bytes jj = beta0 % 4 ..
                            uint8_t* t = P.out_sf + (static_cast<int64_t>(ti.tbg) * (I / 64) + ti.nb * LY::WB + (beta0 >> 2)) * SF_TILE +
                                         (r % 32) * 16 + (r / 32) * 4 + (beta0 & 3);
                            if constexpr (NB == 4) *reinterpret_cast<uint32_t*>(t) = sfw;
                            else *reinterpret_cast<uint16_t*>(t) = static_cast<uint16_t>(sfw);
                        } else {
                            uint8_t* t = P.out_sf + p * (I / 16) + ti.nb * (W_ROWS / 32) + beta0;
                            if constexpr (NB == 4) *reinterpret_cast<uint32_t*>(t) = sfw;
                            else *reinterpret_cast<uint16_t*>(t) = static_cast<uint16_t>(sfw);
                        }
                    }
                } else if (any) {
                    // a round's 64 tile columns are 64 consecutive output columns of one scale (a
                    // gate/up bank's round lies in its gate or its up half); written 128 bytes per row
                    // and instruction through an in-warp transpose
                    static_assert(GPR == 4, "rounds of 64 columns");
                    auto round_col = [&](int rd, float& sc) {
                        const int c0 = half * CPW + rd * GPR * 16;  // first tile column of the round
                        if (P.gate_up) {
                            const int cc = c0 & 127, upper = cc >= 64;
                            sc = sa * (upper ? sb1 : sb0);
                            return (upper ? P.N / 2 : 0) + (ti.nb * LY::WB + (c0 >> 7)) * 64 + (cc & 63);
                        }
                        sc = sa * sb0;
                        return ti.nb * W_ROWS + c0;
                    };
                    if (P.epilogue == kEpiF32) {
#pragma unroll
                        for (int rd = 0; rd < NR; ++rd) {
                            uint32_t v[GPR][16];
                            load_round(rd, v);
                            if (rd == NR - 1) release();
                            float sc;
                            const int col = round_col(rd, sc);
                            // 64 FP32 = two rows of 128 bytes: chunk c = columns 4c .. 4c + 3
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                uint4 x[8];
#pragma unroll
                                for (int c = 0; c < 8; ++c) {
                                    const int g = (hh * 32 + 4 * c) >> 4, e = (4 * c) & 15;
                                    x[c] = make_uint4(__float_as_uint(__uint_as_float(v[g][e]) * sc),
                                                      __float_as_uint(__uint_as_float(v[g][e + 1]) * sc),
                                                      __float_as_uint(__uint_as_float(v[g][e + 2]) * sc),
                                                      __float_as_uint(__uint_as_float(v[g][e + 3]) * sc));
                                }
                                store_rows128(x, reinterpret_cast<uint8_t*>(static_cast<float*>(P.out) + po * P.N + col + hh * 32),
                                              valid, lane);
                            }
                        }
                    } else {
                        // bf16: every round is packed (64 columns = 128 bytes: chunk c = columns 8c .. 8c + 7)
                        // as soon as it is loaded, and the accumulator is freed once the last round is
                        // in registers, before any transpose or store
                        uint4 x[NR][8];
#pragma unroll
                        for (int rd = 0; rd < NR; ++rd) {
                            uint32_t v[GPR][16];
                            load_round(rd, v);
                            if (rd == NR - 1) release();
                            float sc;
                            round_col(rd, sc);
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                const int g = c >> 1, e = (c & 1) * 8;
                                x[rd][c] = make_uint4(pack_bf16x2(__uint_as_float(v[g][e]) * sc, __uint_as_float(v[g][e + 1]) * sc),
                                                      pack_bf16x2(__uint_as_float(v[g][e + 2]) * sc, __uint_as_float(v[g][e + 3]) * sc),
                                                      pack_bf16x2(__uint_as_float(v[g][e + 4]) * sc, __uint_as_float(v[g][e + 5]) * sc),
                                                      pack_bf16x2(__uint_as_float(v[g][e + 6]) * sc, __uint_as_float(v[g][e + 7]) * sc));
                            }
                        }
#pragma unroll
                        for (int rd = 0; rd < NR; ++rd) {
                            float sc;
                            const int col = round_col(rd, sc);
                            store_rows128(x[rd], reinterpret_cast<uint8_t*>(static_cast<uint16_t*>(P.out) + po * P.N + col), valid, lane);
                        }
                    }
                } else {
                    release();
                }
            } else {
                // ---- TMEM lane = weight row m of block nb; columns = token slots of the tile
                const int m = q * 32 + lane;
                uint32_t v[32];
                ptx::tmem_ld16(tbase, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                ptx::tmem_ld16(tbase + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                ptx::tmem_ld_wait();
                const int nv = ti.rows;
                if (P.epilogue == kEpiSwiGLU) {
                    // interleaved gate/up block: lanes 0..63 gate rows, 64..127 the matching up rows
                    SwapXchg& xg = *reinterpret_cast<SwapXchg*>(smem + LY::TAIL_OFF + sizeof(Tail<kMode>));
                    const float sg = sa * sb0, su = sa * sb1;
                    const uint32_t xph = xt & 1;
                    ++xt;
                    bool xok = true;
                    if (q >= 2) {
                        xok = ptx::mbar_wait(&st.xchg_empty, xph ^ 1);
                        if (xok) {
#pragma unroll
                            for (int t = 0; t < 32; ++t)
                                if (t < nv) xg.u[m - 64][t] = __uint_as_float(v[t]) * su;
                        }
                        ptx::mbar_arrive(&st.xchg_full);
                    } else {
                        xok = ptx::mbar_wait(&st.xchg_full, xph);
                    }
                    if (!xok) set_abort(st, a.status);
                    if (q < 2 && xok) {
                        const float S = S_h;
                        const float inv_six_s = 1.0f / (6.0f * S);
#pragma unroll
                        for (int t = 0; t < 32; ++t) {
                            if (t < nv) {  // warp-uniform
                                const float h = silu(__uint_as_float(v[t]) * sg) * xg.u[m][t];
                                float amax = fabsf(h);
#pragma unroll
                                for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
                                const uint32_t sf = ptx::cvt_e4m3x2(amax * inv_six_s, 0.0f) & 0xFFu;
                                const float dsf = ue4m3_to_f32(sf);
                                uint32_t code = 0;
                                if (dsf != 0.0f) code = ptx::cvt_e2m1x2(h * __frcp_rn(dsf * S), 0.0f) & 15u;
                                const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, code, 1);
                                const int64_t p = ti.row0 + t;
                                if ((lane & 1) == 0)
                                    static_cast<uint8_t*>(P.out)[p * (I / 2) + ti.nb * 32 + m / 2] =
                                        static_cast<uint8_t>(code | (other << 4));
                                if ((lane & 15) == 0) {
                                    if (P.out_sf_tiled)
                                        hsf_tile[t * 16 + m / 16] = static_cast<uint8_t>(sf);
                                    else
                                        P.out_sf[p * (I / 16) + ti.nb * 4 + m / 16] = static_cast<uint8_t>(sf);
                                }
                            }
                        }
                    }
                    if (q < 2) ptx::mbar_arrive(&st.xchg_empty);
                } else {
                    int col;
                    float sb;
                    if (P.gate_up) {
                        const int upper = m >= 64;
                        col = (upper ? P.N / 2 : 0) + ti.nb * 64 + (m & 63);
                        sb = upper ? sb1 : sb0;
                    } else {
                        col = ti.nb * W_ROWS + m;
                        sb = sb0;
                    }
                    const float s = sa * sb;
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        if (t < nv) {
                            const int64_t p = __shfl_sync(0xFFFFFFFFu, po, t);  // warp-uniform t
                            const float val = __uint_as_float(v[t]) * s;
                            if (P.epilogue == kEpiF32)
                                static_cast<float*>(P.out)[p * P.N + col] = val;
                            else
                                static_cast<uint16_t*>(P.out)[p * P.N + col] = static_cast<uint16_t>(f32_to_bf16(val));
                        }
                    }
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(&st.acc_empty[as]);
            }
            if (a.nphase > 1 && ti.ph == 0) {
                // publish this warp's part of h for the down GEMM of the same token block: the warp
                // barrier orders the lanes' stores before lane 0's (cumulative) fence and count
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    atomicAdd(a.ready + ti.tbg, 1);
                }
            }
            }  // weight blocks of a unit
        }
    }

    // ---- teardown
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        ptx::tmem_dealloc(tmem, LY::TMEM_COLS);
    }
    ptx::griddep_launch_dependents();  // the next launch may start its prologue on this SM
}

int gemm_schedule_rows(int schedule)
{
    switch (schedule) {
        case kSchedWeightsOnM: return Cfg<kModeSwap>::ACT_ROWS;
        case kSchedWide: return Cfg<kModeWide>::ACT_ROWS;
        case kSchedWideNarrow: return Cfg<kModeWideNarrow>::ACT_ROWS;
        case kSchedWideRows: return Cfg<kModeWideRows>::ACT_ROWS;
        case kSchedWeightsResident: return Cfg<kModeWRes>::ACT_ROWS;
        default: return Cfg<kModeActM>::ACT_ROWS;
    }
}

template <int kMode>
static cudaError_t launch_t(const GemmArgs& a, int64_t p_max, int sms, cudaStream_t stream)
{
    using C = Cfg<kMode>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_grouped_gemm_nvf4<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem_bytes<kMode>()));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    CUtensorMap tmap[2];
    for (int i = 0; i < a.nphase; ++i) {
        const GemmProblem& P = a.p[i];
        // codes prepacked K-slab-major: [G][ceil(K/256)][N][128 bytes]; a tile's K-stage is one
        // contiguous run of W_ROWS x 128 bytes
        const uint64_t slabs = static_cast<uint64_t>(a.G) * ((P.K + 255) / 256);
        CUresult cr = encode_tmap_3d_u8(&tmap[i], P.b_codes, BK_BYTES, static_cast<uint64_t>(P.N), slabs, BK_BYTES, C::W_ROWS);
        if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    if (a.nphase == 1) tmap[1] = tmap[0];
    // contiguous activation rows of a phase (no gather index) with scales in token-block tiles and
    // whole 256-value K-stages come as TMA boxes of 128 rows x 128 bytes (token-block units with two
    // MMA threads); a phase whose codes a box cannot address keeps the per-row copies
    GemmArgs b = a;
    CUtensorMap tmap_a[2] = {tmap[0], tmap[0]};
    for (int i = 0; i < 2; ++i) {
        b.a_tma[i] = 0;
        if (!C::SPLIT || i >= a.nphase || a.p[i].a_row || !a.p[i].a_sf_tiled || a.route.topk_ids || a.p[i].K % 256) continue;
        const GemmProblem& P = a.p[i];
        if (encode_tmap_3d_u8(&tmap_a[i], P.a_codes, static_cast<uint64_t>(P.K / 2), static_cast<uint64_t>(p_max), 1,
                              BK_BYTES, C::ACT_ROWS) == CUDA_SUCCESS)
            b.a_tma[i] = 1;
        else
            tmap_a[i] = tmap[0];
    }
    const int64_t blocks_ub = (p_max + C::ACT_ROWS - 1) / C::ACT_ROWS + a.G;
    const int64_t tiles_ub = blocks_ub * (C::ROWS ? 1 : a.p[0].N / C::W_ROWS);
    const int grid = static_cast<int>(tiles_ub < sms ? (tiles_ub < 1 ? 1 : tiles_ub) : sms);
    // Two phases: CTAs wait on one another's results, so all of them must become resident. The
    // grid is at most one CTA per SM and a CTA needs most of an SM's shared memory, so the whole
    // grid is resident once earlier kernels on the SMs have drained (they never wait on this one);
    // the waits are bounded in any case and report a timeout in the status word.
    return launch_pdl(k_grouped_gemm_nvf4<kMode>, dim3(grid), dim3(Lay<kMode>::THREADS), smem_bytes<kMode>(), stream,
                      tmap[0], tmap[1], tmap_a[0], tmap_a[1], b);
}

bool gemm_rows_pays(int64_t p_max, int sms)
{
    // Token-block units carry six (gate/up) or eight (down) weight blocks each, so with few 128-row
    // blocks per SM the last units leave SMs idle longer. With one MMA thread that outweighed the
    // saved scale copies below about eight blocks per SM (4k tokens: 305 vs 285 us). Their two MMA
    // threads and TMA activation boxes now win from about one block per SM: 4k tokens 217 vs 245 us,
    // 2,048 tokens 240 vs 262 us for the expert GEMMs.
    return p_max >= 1LL * sms * Cfg<kModeWideRows>::ACT_ROWS;
}

bool gemm_wide_fits(const GemmArgs& a)
{
    return a.p[0].N % Cfg<kModeWide>::W_ROWS == 0 && (a.nphase < 2 || a.p[1].N % Cfg<kModeWide>::W_ROWS == 0);
}

cudaError_t launch_grouped_gemm(const GemmArgs& a, int64_t p_max, int schedule, int sms, cudaStream_t stream)
{
    if ((schedule == kSchedWide || schedule == kSchedWideNarrow || schedule == kSchedWideRows) && !gemm_wide_fits(a))
        schedule = kSchedActOnM;
    if (schedule == kSchedWeightsResident &&
        (a.p[0].K > Cfg<kModeWRes>::MAX_K || (a.nphase > 1 && a.p[1].K > Cfg<kModeWRes>::MAX_K)))
        schedule = kSchedActOnM;  // the resident region holds K <= 2048
    if (schedule == kSchedAuto) schedule = p_max <= 64 ? kSchedWeightsOnM : kSchedActOnM;
    switch (schedule) {
        case kSchedWeightsOnM: return launch_t<kModeSwap>(a, p_max, sms, stream);
        case kSchedWide: return launch_t<kModeWide>(a, p_max, sms, stream);
        case kSchedWideNarrow: return launch_t<kModeWideNarrow>(a, p_max, sms, stream);
        case kSchedWideRows:
            if (a.p[0].K <= Cfg<kModeWideRows>::MAX_K && (a.nphase < 2 || a.p[1].K <= Cfg<kModeWideRows>::MAX_K))
                return launch_t<kModeWideRows>(a, p_max, sms, stream);
            return launch_t<kModeWide>(a, p_max, sms, stream);
        case kSchedWeightsResident: return launch_t<kModeWRes>(a, p_max, sms, stream);
        default: return launch_t<kModeActM>(a, p_max, sms, stream);
    }
}

}  // namespace moe
