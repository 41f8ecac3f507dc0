/*
 * moe_nvfp4.h -- C ABI of libmoe_nvfp4.so: the forward pass of a routed mixture-of-experts layer
 * in NVIDIA's NVFP4 format with NVFP4 activations (W4A4), on one sm_103a GPU.
 *
 * The layer (shape of Qwen3.8-Flash-Next's MoE: hidden H = 2048, E = 512 routed experts, k = 10
 * routed + 1 shared expert per token, SwiGLU experts of width I = 768):
 *
 *   logits  = x W_r^T                      (bf16 inputs, FP32 accumulation; + optional bias)
 *   ids, w  = top-k of softmax_FP32(logits), ties to the lowest expert id, w renormalised to sum 1
 *   g       = sigmoid(x w_sg)              (w_sg = row E of W_r: the shared-expert gate)
 *   xq      = NVFP4(x)                     (E2M1 codes, UE4M3 scale per 16 along H, FP32 tensor scale)
 *   rows    = the (token, expert) pairs grouped by expert id (stable), then the shared expert
 *   h_r     = NVFP4_static( silu(xq W_gate[e]^T) * (xq W_up[e]^T) )   per row r of expert e
 *   y_r     = h_r W_down[e]^T
 *   out_t   = bf16( [residual_t +] sum_j w_tj y_(t,j) + g_t y_shared,t )   (FP32 accumulation)
 *
 * Sources for the format and the shape: the article "capy-flash runs a 125B MoE in full NVFP4 on
 * two 16 GB GPUs ..." (richland.au), section "What shipped": E2M1 codes, UE4M3 block scales and an
 * FP32 per-expert scale; 512 experts, 10 routed + 1 shared per layer. The capy-flash README v0.5.4,
 * "What it does": activations are quantized to NVFP4 on the GPU (W4A4). The same article, "Why it
 * matters": partial sums accumulate in FP32 throughout. The remaining steps (softmax top-k with
 * renormalised weights, SwiGLU, static requantisation of the intermediate, sigmoid-gated shared
 * expert) are this library's layer definition; the pages print no formula for them.
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers owned by the caller unless a parameter says otherwise. The
 *     library never allocates device memory and keeps no state between calls (except the
 *     per-process driver entry point it looks up once).
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - NVFP4 tensors, row-major ("ModelOpt layout"): codes [rows][K/2] bytes, two E2M1 codes per
 *     byte, the even-K element in the low nibble; block scales [rows][K/16] UE4M3 bytes; one FP32
 *     tensor scale. Value = e2m1(code) * ue4m3(sf) * S.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *     They return MOE_OK after a successful launch; argument errors are detected on the host
 *     before any launch and return an error code (moe_last_error_detail() gives the numbers).
 *   - Scratch comes from a caller workspace of moe_workspace_bytes() bytes (256-byte aligned).
 *     Its first 256 bytes (status word and launch counters) must be zero before its first use;
 *     the calls leave the counters at zero. One workspace serves one stream at a time.
 *   - An empty batch (T = 0) is valid. moe_route_topk, moe_combine, moe_layer_forward and
 *     moe_layer_forward_host then return MOE_OK after checking the shape alone: they read and write
 *     nothing, so their pointers may be NULL. moe_permute still writes its offsets (all zero), and
 *     moe_layer_forward_profiled given events checks its arguments as for T > 0 and records each event.
 *     Kernels record device-side failures (a bounded wait that ran out) in a status word in the
 *     workspace; moe_read_device_status() synchronises `stream` and returns it.
 *   - Shapes: H and I multiples of 128; 1 <= k <= min(E, 32); 1 <= E <= 1024; T >= 0.
 */
#ifndef MOE_NVFP4_H
#define MOE_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,          /* null pointer, negative size, bad enum value */
    MOE_ERR_UNSUPPORTED_SHAPE = 2,    /* a shape outside the limits above */
    MOE_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes < the size the call needs */
    MOE_ERR_MISALIGNED = 4,           /* a pointer below its required alignment */
    MOE_ERR_CUDA = 5,                 /* a CUDA runtime / driver call or a launch failed */
    MOE_ERR_DEVICE_TIMEOUT = 6,       /* a kernel's bounded wait ran out (status word) */
    MOE_ERR_UNSUPPORTED_DEVICE = 7    /* the current device is not sm_103 */
} moe_status_t;

typedef void* moe_stream_t; /* cudaStream_t */

/* NVFP4 weights of G experts, each an [N][K] matrix, in the PREPACKED layout that
 * moe_prepack_nvfp4() writes (see there). gscale: [G][nscale] FP32 per-expert tensor scales. */
typedef struct {
    const uint8_t* codes; /* [G][ceil(K/256)][N][128] K-slabs, rows in prepacked order */
    const uint8_t* sf;    /* [G][N/128][K/64][512] scale-factor tiles */
    const float* gscale;  /* [G][nscale] */
} moe_nvfp4_bank_t;

/* One MoE layer. The shared expert is expert index E of both banks. */
typedef struct {
    int H, E, k, I;
    const uint16_t* w_router;   /* bf16 [E+1][H]; row E = shared-expert gate vector */
    const float* logit_bias;    /* nullable, FP32 [E], 16-byte aligned, added to the routed logits */
    moe_nvfp4_bank_t w_gate_up; /* G = E+1, N = 2I, K = H, prepacked with gate/up interleave; gscale [E+1][2] (gate, up) */
    moe_nvfp4_bank_t w_down;    /* G = E+1, N = H, K = I, prepacked plain; gscale [E+1] */
    const float* s_mid;         /* FP32 [E+1]: static tensor scale of the intermediate h per expert */
} moe_layer_t;

/* Epilogues of moe_grouped_gemm_nvfp4, optionally OR-ed with one schedule flag. */
enum {
    MOE_EPI_F32 = 0,         /* out: FP32 [P][N] */
    MOE_EPI_BF16 = 1,        /* out: bf16 [P][N] */
    MOE_EPI_SWIGLU_NVFP4 = 2, /* gate/up bank; out: h codes [P][N/4], out_sf [P][N/32], scale epi_scale[g] */
    /* Tile schedule (default: weights on M when p_max <= 64, else activations on M). Results agree
     * to FP32 summation order. */
    MOE_GEMM_SCHED_ACT_ON_M = 0x100,     /* 128 token rows x 128 weight rows per tile */
    MOE_GEMM_SCHED_WEIGHTS_ON_M = 0x200, /* 128 weight rows x 32 token rows per tile (small groups) */
    MOE_GEMM_SCHED_WIDE = 0x400,         /* 128 token rows x 256 weight rows per tile (N % 256 == 0,
                                          * else activations on M) */
    MOE_GEMM_SCHED_WIDE_ROWS = 0x800,    /* wide tiles, each CTA taking a whole 128-row token block
                                          * through every weight block (the activation scales stay
                                          * in tensor memory; two threads issue the MMAs, 128 weight
                                          * rows each); K <= 2048, else wide */
    MOE_GEMM_SCHED_WEIGHTS_RESIDENT = 0x1000 /* one group's 128-row weight block (all of K) kept in shared
                                          * memory, its scales in tensor memory, while up to 16 of the
                                          * group's 128-row token blocks stream past it into two
                                          * alternating accumulators; K <= 2048, else activations on M */
};

/* ---------------------------------------------------------------------------------------------
 * moe_quantize_nvfp4 -- NVFP4 encoding of activations (W4A4: "What it does", capy-flash README).
 *   x: bf16 [rows][K], K % 16 == 0. s_in: nullable device FP32 scalar; when NULL the tensor scale
 *   is S = amax(|x|) / (6 * 448) (S = 1 when x is all zero), written to *s_out; when given, S =
 *   *s_in (static scale) and is copied to *s_out. Per 16-element block: sf = UE4M3 nearest-even of
 *   amax_b / (6 S) saturating at 448; each element: E2M1 nearest-even of x / (ue4m3(sf) S),
 *   saturating at 6, sign kept; a block whose sf decodes to 0 has all codes 0.
 *   codes: [rows][K/2]; sf: [rows][K/16]; s_out: FP32 scalar. ws: >= 256 bytes.
 *   Results are bit-exact (every FP32 step is rounded to nearest, no contraction).
 * moe_quantize_nvfp4_f32 -- the same from FP32 input (used to quantize weights).
 * ------------------------------------------------------------------------------------------- */
moe_status_t moe_quantize_nvfp4(const uint16_t* x, int64_t rows, int64_t K, const float* s_in,
                                uint8_t* codes, uint8_t* sf, float* s_out, void* ws, size_t ws_bytes,
                                moe_stream_t stream);
moe_status_t moe_quantize_nvfp4_f32(const float* x, int64_t rows, int64_t K, const float* s_in,
                                    uint8_t* codes, uint8_t* sf, float* s_out, void* ws,
                                    size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * moe_route_topk -- router GEMM, FP32 softmax, top-k with renormalised weights, shared gate.
 *   The capy-flash README v0.5.4 ("Measured") notes that the summation order of the router can
 *   flip exact ties; here ties are broken by the lowest expert id. A NaN logit ranks below every
 *   number, so the ids are always in [0, E).
 *   x: bf16 [T][H]; uses L->w_router, L->logit_bias, L->H, L->E, L->k.
 *   topk_ids: int32 [T][k] (routing order: weight non-increasing); topk_w: FP32 [T][k];
 *   shared_g: nullable FP32 [T]; logits_out: nullable FP32 [T][E] (bias included).
 *   With E = 512, k <= 16 and T >= 12288 the logits, top-k, weights and shared gate come from one
 *   launch that holds all 512 logits of 128 tokens per CTA; the shared-gate logit is then a
 *   sequential FP32 sum (the routed logits stay tensor-core sums).
 *   ws: >= moe_workspace_bytes(H, E, k, I, T).
 * ------------------------------------------------------------------------------------------- */
moe_status_t moe_route_topk(const uint16_t* x, int T, const moe_layer_t* L, int32_t* topk_ids,
                            float* topk_w, float* shared_g, float* logits_out, void* ws,
                            size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * moe_permute -- stable counting sort of the T*k assignments f = t*k + j by expert id.
 *   The layer's step "permute tokens by expert id" between routing and the grouped GEMMs: the
 *   pages (article "What shipped": 10 routed + 1 shared expert per token) give no order, so this
 *   library takes the plainest deterministic one -- stable, rows of one expert in ascending f --
 *   and appends the shared expert as group E with one row per token.
 *   expert_offsets: int32 [E+2]: rows of expert e are [off[e], off[e+1]) (e < E); the shared
 *   expert's group is [off[E], off[E+1]) = [T*k, T*k + T) when with_shared, else empty.
 *   perm_src: int32 [T*k], perm_src[p] = f; src_perm: int32 [T*k], src_perm[f] = p;
 *   row_token: nullable int32 [T*k + T*with_shared], the token of every permuted row (f / k, then
 *   t for the shared rows) -- the gather index of the gate/up GEMM. Bit-exact.
 *   ws: >= moe_workspace_bytes(any H, E, k, any I, T).
 * ------------------------------------------------------------------------------------------- */
moe_status_t moe_permute(const int32_t* topk_ids, int T, int k, int E, int with_shared,
                         int32_t* expert_offsets, int32_t* perm_src, int32_t* src_perm,
                         int32_t* row_token, void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * moe_prepack_nvfp4 -- rewrite G row-major NVFP4 matrices [N][K] into the layout the grouped GEMM
 *   streams with TMA: codes become K-slab-major [G][ceil(K/256)][N][128 bytes] (slab s = bytes
 *   128 s .. 128 s + 127 of every row, zero past K/2; codes_out holds G * N * ceil(K/256) * 128
 *   bytes), so one TMA box of rows is one contiguous run; with gate_up_interleave = 1 the rows are
 *   reordered in blocks of 128 = 64 gate rows n..n+63 followed by the 64 up rows N/2+n..N/2+n+63.
 *   Block scales become 512-byte tiles [G][N/128][K/64]: tile byte (r % 32) * 16 + (r / 32) * 4 + j
 *   holds the scale of row r (of the 128) for K-block 4 * (tile index) + j.
 *   N % 128 == 0, K % 64 == 0; outputs must not alias inputs.
 * ------------------------------------------------------------------------------------------- */
moe_status_t moe_prepack_nvfp4(const uint8_t* codes, const uint8_t* sf, int G, int N, int K,
                               int gate_up_interleave, uint8_t* codes_out, uint8_t* sf_out,
                               moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * moe_grouped_gemm_nvfp4 -- block-scaled grouped GEMM on the tcgen05 tensor cores
 *   (kind::mxf4nvf4: E2M1 x E2M1 products, UE4M3 scale per 16 along K, FP32 accumulation in TMEM).
 *   The expert GEMMs of the layer: NVFP4 weights "as published" with E2M1 codes, UE4M3 block
 *   scales and an FP32 per-expert scale (article, "What shipped") against NVFP4 activations (W4A4,
 *   capy-flash README v0.5.4, "What it does"); accumulation in FP32 ("Why it matters"). The block
 *   length of 16 along K and the SwiGLU + static-scale requantisation of the intermediate are this
 *   library's readings (the pages print no formula).
 *   For every group g < G and row p in [group_offsets[g], group_offsets[g+1]):
 *     acc[p][n] = sum_k A_hat[src(p)][k] * B_hat[g][n][k],  src(p) = a_row_index ? a_row_index[p] : p
 *   A: codes [*][K/2], sf [*][K/16] (row-major), tensor scale a_scale[a_scale_per_group ? g : 0].
 *   B: a prepacked bank with N columns (natural column order n of the unpacked matrix).
 *   Epilogues:
 *     MOE_EPI_F32 / MOE_EPI_BF16: out[p][n] = acc * a_scale * gscale[g][half]; half = n >= N/2
 *        for a gate/up bank (nscale 2, interleaved prepack), else 0.
 *     MOE_EPI_SWIGLU_NVFP4 (gate/up bank): h[p][j] = silu(gate) * up (FP32), j < N/2, encoded
 *        like moe_quantize_nvfp4 with the static scale epi_scale[g]: out = codes [P][N/4],
 *        out_sf = [P][N/32].
 *   gate_up: 1 when b is a gate/up bank (nscale 2, interleaved prepack), 0 for a plain bank.
 *   N % 128 == 0, K % 64 == 0, K <= 16384. P = group_offsets[G] (read on the device);
 *   p_max: an upper bound of P that the host knows (sizes the grid).
 *   ws: >= 256 bytes (status word).
 * ------------------------------------------------------------------------------------------- */
moe_status_t moe_grouped_gemm_nvfp4(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_scale,
                                    int a_scale_per_group, const int32_t* a_row_index,
                                    const int32_t* group_offsets, int G, int64_t p_max,
                                    const moe_nvfp4_bank_t* b, int N, int K, int gate_up, int epilogue,
                                    const float* epi_scale, void* out, uint8_t* out_sf, void* ws,
                                    size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * moe_combine -- weighted un-permute with FP32 accumulation ("Why it matters": FP32 partials):
 *   out[t] = bf16( [residual[t] +] sum_j topk_w[t][j] * y[src_perm[t*k+j]]
 *                  + (shared_g ? shared_g[t] * y[T*k + t] : 0) )
 *   y: bf16 [T*k (+T)][H]; residual nullable bf16 [T][H]; out bf16 [T][H]. Each product is rounded
 *   to FP32 before it is added (the README's rounding-order note: a product, then a sum).
 * ------------------------------------------------------------------------------------------- */
moe_status_t moe_combine(const uint16_t* y, const float* topk_w, const float* shared_g,
                         const int32_t* src_perm, int T, int k, int H, const uint16_t* residual,
                         uint16_t* out, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * moe_layer_forward -- the whole layer (all steps above) on `stream`.
 *   x: bf16 [T][H]; residual: nullable bf16 [T][H] (added to the output: a stack of MoE layers);
 *   out: bf16 [T][H], must not alias x. ws: >= moe_workspace_bytes(H, E, k, I, T).
 * ------------------------------------------------------------------------------------------- */
moe_status_t moe_layer_forward(const moe_layer_t* L, const uint16_t* x, int T, const uint16_t* residual,
                               uint16_t* out, void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * moe_layer_forward_profiled -- moe_layer_forward that also records caller-created CUDA events
 *   (cudaEvent_t handles) on `stream` at the stage boundaries: events[0] before the activation
 *   quantizer, [1] after it, [2] after routing (logits + top-k), [3] after the permutation, [4]
 *   after the expert GEMMs (gate/up + SwiGLU + requantisation + down, one launch), [5] after the
 *   combine. For small batches (T <= 64 and T*k <= 512) quantisation, routing and permutation run
 *   as one launch between events [0] and [1]; [2] and [3] then follow [1] directly. For large
 *   batches with E = 512 and k <= 16 (T >= 12288) routing runs first and also takes x's maximum:
 *   [1] follows routing and [2] the quantizer (moe_layer_workspace_view reports route_first = 1).
 *   n_events: 0 (plain forward) or 6. The library creates and destroys no event.
 * ------------------------------------------------------------------------------------------- */
moe_status_t moe_layer_forward_profiled(const moe_layer_t* L, const uint16_t* x, int T, const uint16_t* residual,
                                        uint16_t* out, void* ws, size_t ws_bytes, moe_stream_t stream,
                                        void* const* events, int n_events);

/* ---------------------------------------------------------------------------------------------
 * moe_layer_forward_host -- moe_layer_forward for a caller whose tokens live in HOST memory: the
 *   call enqueues on `stream` the copy of x (and residual) into device staging inside the
 *   workspace, the whole layer, and the copy of the result back to `out`.
 *   x: host bf16 [T][H]; residual: nullable host bf16 [T][H]; out: host bf16 [T][H], must not
 *   overlap x or residual. Page-locked host memory (cudaHostAlloc / cudaHostRegister) keeps the
 *   call asynchronous; pageable memory also works, with the copies then behaving as
 *   cudaMemcpyAsync does for pageable memory (staged, partly synchronous). The call returns once
 *   everything is enqueued: `out` holds the result when `stream` has passed this point (for
 *   example after cudaStreamSynchronize), and x / residual must stay unchanged until then.
 *   A device pointer for x, residual or out returns MOE_ERR_INVALID_ARG.
 *   ws: >= moe_workspace_bytes_host(H, E, k, I, T) (the layer's workspace followed by three
 *   256-byte-aligned staging buffers of T*H bf16).
 * ------------------------------------------------------------------------------------------- */
moe_status_t moe_layer_forward_host(const moe_layer_t* L, const uint16_t* x, int T, const uint16_t* residual,
                                    uint16_t* out, void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * moe_route_topk_noalloc -- moe_route_topk for callers that cannot give the library scratch
 *   memory: an application whose device memory is owned by another allocator and may not grow
 *   by extra cudaMalloc calls, or a decode loop that cannot afford cudaMalloc's implicit device
 *   synchronisation. The capy-flash pages have no counterpart of this call; it is a convenience
 *   of this library.
 *   Same arguments and results as moe_route_topk, without the workspace. The logits scratch is a
 *   fixed array inside the library (64 tokens x 1025 FP32 = 262,400 bytes of device memory on
 *   every GPU that loads the library, held until the process exits); it allocates nothing.
 *   Limits: T <= 64, E <= 1024; larger calls return MOE_ERR_UNSUPPORTED_SHAPE (use
 *   moe_route_topk). The first call with T > 0 on a device looks up the array's device address (a
 *   host-side set-up step); make that first call before capturing any stream. The checks run in
 *   moe_route_topk's order, so an empty batch (T = 0) returns MOE_OK with NULL buffers allowed. Every call shares the one
 *   array: calls that overlap on the GPU (other streams or host threads) race on it.
 * ------------------------------------------------------------------------------------------- */
moe_status_t moe_route_topk_noalloc(const uint16_t* x, int T, const moe_layer_t* L, int32_t* topk_ids,
                                    float* topk_w, float* shared_g, float* logits_out, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * moe_layer_workspace_view -- where moe_layer_forward leaves the layer's intermediate results in
 *   its workspace, so a caller can inspect them after the call (for example to check each step
 *   against a reference implementation). The pages have no counterpart; the results themselves
 *   are the steps listed at the top of this header. Every field is a BYTE OFFSET from the start
 *   of the workspace, valid for a forward of T tokens through a layer of L's shape on the current
 *   device, once `stream` has passed that forward and until the next call that uses the workspace:
 *     x_scale         FP32 scalar: the tensor scale S_x of x
 *     x_codes, x_sf   NVFP4 x: codes u8 [T][H/2], block scales u8 [T][H/16]
 *     logits          FP32 [T][logits_ld]: column e < E = the routed logit (bias included),
 *                     column E = the shared-gate logit
 *     topk_ids/_w     int32 / FP32 [T][k] in routing order; shared_g FP32 [T]
 *     expert_offsets  int32 [E+2]; perm_src, src_perm int32 [T*k]; row_token int32 [T*k + T]
 *                     (as moe_permute) -- only when permutation_in_workspace is 1; for small
 *                     batches the expert GEMMs build the permutation in on-chip memory instead
 *                     (permutation_in_workspace 0) and these bytes are not written
 *     h_codes         the requantised intermediate, u8 [T*k + T][I/2], rows in permuted order
 *                     (expert groups ascending, the shared expert's T rows last)
 *     h_sf            its block scales in 512-byte tiles [token block][I/64][512]: the rows of
 *                     each expert group are cut into blocks of h_block_rows (the last one ragged),
 *                     numbered across the groups in order; row r of a block, scale column c is
 *                     byte (r % 32) * 16 + (r / 32) * 4 + c % 4 of tile c / 4
 *     y               bf16 [T*k + T][H]: the down projection of row (t, j) at row t*k + j (the
 *                     assignment order), of the shared expert for token t at row T*k + t
 *     route_first     1 when the forward routes before it encodes x (the fused router of large
 *                     batches), else 0
 *   bytes = moe_workspace_bytes(H, E, k, I, T). The view depends on the device (its SM count
 *   picks the tile schedule), so query it on the device that runs the forward.
 * ------------------------------------------------------------------------------------------- */
typedef struct {
    int64_t bytes;
    int64_t x_scale, x_codes, x_sf;
    int64_t logits, logits_ld;
    int64_t topk_ids, topk_w, shared_g;
    int64_t permutation_in_workspace, expert_offsets, perm_src, src_perm, row_token;
    int64_t h_codes, h_sf, h_block_rows;
    int64_t y;
    int64_t route_first;
} moe_layer_view_t;

moe_status_t moe_layer_workspace_view(const moe_layer_t* L, int T, moe_layer_view_t* view);

/* ---------------------------------------------------------------------------------------------
 * moe_set_wait_test_hook -- test hook of the failure path (the pages' engine fails one request,
 *   not the server: capy-flash README v0.7.7, "What's new"). Every device-side wait of the library
 *   is bounded; this makes one of them run out on purpose, with no fault: the expert GEMMs' wait
 *   for a token block's intermediate then gives up after wait_limit_us microseconds (0: the
 *   default, 1 s) and needs ready_extra more completions than exist (0: the real count), so
 *   with ready_extra > 0 every down tile of moe_layer_forward times out; the launch stops, frees
 *   its tensor memory and records MOE_ERR_DEVICE_TIMEOUT for moe_read_device_status(). Another
 *   call with (0, 0) restores normal operation. The values are written into the workspace header
 *   in stream order (a one-thread kernel on `stream`).
 * ------------------------------------------------------------------------------------------- */
moe_status_t moe_set_wait_test_hook(void* ws, unsigned wait_limit_us, int ready_extra, moe_stream_t stream);

/* Workspace bytes for any call above with these sizes (T tokens). */
size_t moe_workspace_bytes(int H, int E, int k, int I, int T);

/* Workspace bytes for moe_layer_forward_host with these sizes (T tokens). */
size_t moe_workspace_bytes_host(int H, int E, int k, int I, int T);

/* Synchronise `stream`, read and clear the device status word of `ws`: MOE_OK or
 * MOE_ERR_DEVICE_TIMEOUT. */
moe_status_t moe_read_device_status(void* ws, moe_stream_t stream);

const char* moe_status_string(moe_status_t s);

/* Thread-local text of the last host-side error, with the offending numbers. */
const char* moe_last_error_detail(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_NVFP4_H */
