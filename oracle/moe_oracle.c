/*
 * moe_oracle.c -- plain, slow, CPU reference of the NVFP4 (W4A4) routed-MoE layer forward.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this library. The GPU library never links or calls it, and it shares no code, header,
 * table or constant generator with the GPU library.
 *
 * What the layer is, as the capy-flash pages state it:
 *   - "capy-flash runs a 125B MoE in full NVFP4 ..." (richland.au), section "What shipped":
 *     a 48-layer MoE with 512 experts, 10 routed + 1 shared per layer; NVFP4 weights made of
 *     E2M1 codes, UE4M3 block scales and an FP32 per-expert scale.
 *   - capy-flash README v0.5.4 (spark.entire.vc), "What it does": activations are quantized to
 *     NVFP4 on the GPU (W4A4) before they meet the NVFP4 expert weights.
 *   - same article, "Why it matters": partial sums are accumulated in FP32 throughout.
 * The rest of the layer (FP32 softmax, top-k with renormalised weights and lowest-index ties,
 * SwiGLU, requantisation of the intermediate, sigmoid-gated shared expert, weighted combine)
 * is the layer definition this library implements; the pages print no formula for it.
 * Every step below is that plain definition, evaluated with FP64 accumulation.
 *
 * Readings taken where the pages are silent (each is repeated in the design notes):
 *   R1 block = 16 consecutive elements along K (the reduction dimension), one UE4M3 scale each.
 *   R2 tensor scale S = amax(|X|) / (6 * 448) computed in FP32; S = 1 when amax == 0.
 *   R3 block scale = UE4M3 nearest-even (saturating at 448) of amax_b / (6 * S), in FP32 ops.
 *   R4 element code = E2M1 nearest-even (saturating at 6) of x / (dec(sf) * S), FP32 ops;
 *      the sign bit is kept, so a negative value that rounds to zero encodes 0x8;
 *      a block whose scale decodes to 0 encodes all codes as 0x0.
 *   R5 packing: two codes per byte, the even-K element in the low nibble.
 *   R6 routed experts are selected on the logits (softmax is monotone) by (value desc, index asc).
 *   R7 the shared expert is group E of the grouped GEMMs, one row per token.
 *   R8 the layer output is rounded once, from FP64 to bf16 (nearest-even).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (no fast-math; FP32 steps stay FP32).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------------ */
/* Formats                                                                                      */
/* ------------------------------------------------------------------------------------------ */

/* E2M1 magnitudes indexed by the 3 low bits of a code (1 sign, 2 exponent, 1 mantissa bit). */
static const double kE2M1Mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(int code)
{
    double m = kE2M1Mag[code & 7];
    return (code & 8) ? -m : m;
}

/* UE4M3: unsigned, 4 exponent bits (bias 7), 3 mantissa bits; e == 0 is subnormal m * 2^-9;
 * code 0x7F is NaN and is never produced; 0x7E = 448 is the largest finite value. */
double orc_ue4m3_value(int code)
{
    int e = (code >> 3) & 15;
    int m = code & 7;
    if ((code & 0x80) || code == 0x7F) return NAN;
    if (e == 0) return ldexp((double)m, -9);
    return ldexp(1.0 + m / 8.0, e - 7);
}

/* Nearest UE4M3 value to q >= 0; ties go to the even code (even mantissa); q >= 448 gives 448.
 * Written as a search over all finite codes, which is the definition of round-to-nearest. */
uint8_t orc_ue4m3_encode(float q)
{
    if (!(q > 0.0f)) return 0;
    if (q >= 448.0f) return 0x7E;
    int best = 0;
    double bestd = fabs((double)q);
    for (int c = 1; c <= 0x7E; ++c) {
        double d = fabs((double)q - orc_ue4m3_value(c));
        if (d < bestd || (d == bestd && (c & 1) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)best;
}

/* Nearest E2M1 value to v; ties go to the even code; |v| > 6 gives 6; the sign bit is kept. */
uint8_t orc_e2m1_encode(float v)
{
    double a = fabs((double)v);
    int best = 0;
    double bestd = a;
    for (int m = 1; m < 8; ++m) {
        double d = fabs(a - kE2M1Mag[m]);
        if (d < bestd || (d == bestd && (m & 1) == 0)) {
            best = m;
            bestd = d;
        }
    }
    return (uint8_t)((signbit(v) ? 8 : 0) | best);
}

/* bf16 nearest-even rounding of a double (R8): keep 8 significant bits. */
double orc_round_bf16(double v)
{
    if (v == 0.0 || !isfinite(v)) return v;
    int e;
    double m = frexp(v, &e); /* v = m * 2^e, 0.5 <= |m| < 1 */
    return ldexp(nearbyint(ldexp(m, 8)), e - 8);
}

/* ------------------------------------------------------------------------------------------ */
/* NVFP4 encode / decode (R1-R5)                                                                */
/* ------------------------------------------------------------------------------------------ */

/* Tensor scale of a whole tensor (R2). */
float orc_tensor_scale(const float* x, int64_t n)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) return 1.0f;
    return amax / 2688.0f;
}

/* Encode x[rows][K] with tensor scale S. codes: [rows][K/2], sf: [rows][K/16]. */
static void encode_with_scale(const float* x, int64_t rows, int64_t K, float S, uint8_t* codes,
                              uint8_t* sf)
{
    const float six_s = 6.0f * S;
    const int64_t nb = K / 16;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float* blk = x + r * K + b * 16;
            float amax_b = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float a = fabsf(blk[i]);
                if (a > amax_b) amax_b = a;
            }
            float q = amax_b / six_s;
            uint8_t s = orc_ue4m3_encode(q);
            sf[r * nb + b] = s;
            double dsf = orc_ue4m3_value(s);
            float d = (float)dsf * S;
            uint8_t* out = codes + r * (K / 2) + b * 8;
            for (int i = 0; i < 16; i += 2) {
                uint8_t c0 = 0, c1 = 0;
                if (dsf != 0.0) {
                    c0 = orc_e2m1_encode(blk[i] / d);
                    c1 = orc_e2m1_encode(blk[i + 1] / d);
                }
                out[i / 2] = (uint8_t)(c0 | (c1 << 4));
            }
        }
    }
}

/* Quantize x[rows][K] (K % 16 == 0). s_in > 0: static scale; otherwise S from the tensor (R2).
 * Returns 0, or -1 on a bad shape. */
int orc_quantize_nvfp4(const float* x, int64_t rows, int64_t K, float s_in, uint8_t* codes,
                       uint8_t* sf, float* s_out)
{
    if (rows < 0 || K <= 0 || K % 16 != 0) return -1;
    float S = (s_in > 0.0f) ? s_in : orc_tensor_scale(x, rows * K);
    if (s_out) *s_out = S;
    encode_with_scale(x, rows, K, S, codes, sf);
    return 0;
}

/* x_hat = e2m1(code) * dec(sf) * S, exactly, in FP64. */
void orc_dequantize_nvfp4(const uint8_t* codes, const uint8_t* sf, float S, int64_t rows, int64_t K,
                          double* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = codes[r * (K / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            out[r * K + k] = orc_e2m1_value(code) * orc_ue4m3_value(sf[r * (K / 16) + k / 16]) * (double)S;
        }
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Router: logits, FP64 softmax, top-k, renormalised weights, shared gate (R6)                  */
/* ------------------------------------------------------------------------------------------ */

/* Routing decision from given logits (R6): softmax over all E logits in FP64, the top k by
 * (logit desc, index asc), their probabilities renormalised to sum 1; the shared gate is the
 * sigmoid of the gate logit. logits: [T][E]; gate_logit: nullable [T].
 * Outputs: topk_ids [T][k] in routing order, topk_w [T][k], shared_g [T] (if gate_logit). */
void orc_route_from_logits(const double* logits, const double* gate_logit, int T, int E, int k,
                           int32_t* topk_ids, double* topk_w, double* shared_g)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (int t = 0; t < T; ++t) {
        const double* l = logits + (int64_t)t * E;
        unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
        /* softmax over all E experts */
        double mx = l[0];
        for (int e = 1; e < E; ++e)
            if (l[e] > mx) mx = l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += exp(l[e] - mx);
        /* top-k by (logit desc, index asc): a strict '>' keeps the lowest index on ties */
        double psum = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;
            }
            taken[best] = 1;
            topk_ids[(int64_t)t * k + j] = best;
            double p = exp(l[best] - mx) / z;
            topk_w[(int64_t)t * k + j] = p;
            psum += p;
        }
        for (int j = 0; j < k; ++j) topk_w[(int64_t)t * k + j] /= psum;
        if (gate_logit) shared_g[t] = 1.0 / (1.0 + exp(-gate_logit[t]));
        free(taken);
    }
}

/* x: [T][H]; w_router: [E + has_shared][H] (the last row is the shared-expert gate when
 * has_shared); bias: nullable [E], added to the routed logits.
 * Outputs: topk_ids [T][k] in routing order, topk_w [T][k], shared_g [T] (if has_shared),
 * logits [T][E] (nullable). The logits are FP64 dot products of the bf16 values; the routing
 * decision is orc_route_from_logits on them. */
void orc_router(const float* x, const float* w_router, const double* bias, int T, int H, int E,
                int k, int has_shared, int32_t* topk_ids, double* topk_w, double* shared_g,
                double* logits)
{
    double* l = (double*)malloc(sizeof(double) * (size_t)T * (size_t)E);
    double* lg = has_shared ? (double*)malloc(sizeof(double) * (size_t)T) : NULL;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; ++t) {
        const float* xt = x + (int64_t)t * H;
        for (int e = 0; e < E + (has_shared ? 1 : 0); ++e) {
            const float* we = w_router + (int64_t)e * H;
            double s = 0.0;
            for (int h = 0; h < H; ++h) s += (double)xt[h] * (double)we[h];
            if (e == E) {
                lg[t] = s;
            } else {
                l[(int64_t)t * E + e] = s + (bias ? bias[e] : 0.0);
                if (logits) logits[(int64_t)t * E + e] = l[(int64_t)t * E + e];
            }
        }
    }
    orc_route_from_logits(l, lg, T, E, k, topk_ids, topk_w, shared_g);
    free(l);
    free(lg);
}

/* ------------------------------------------------------------------------------------------ */
/* Permutation: stable counting sort of the flat assignments f = t*k + j by expert id          */
/* ------------------------------------------------------------------------------------------ */

/* offsets: [E+2]; offsets[e]..offsets[e+1] are the rows of expert e (e < E); the shared group
 * (R7) is offsets[E]..offsets[E+1] = T*k .. T*k + T when with_shared, else empty.
 * perm_src[p] = f (the assignment held by permuted row p), src_perm[f] = p. Returns 0 or -1. */
int orc_permute(const int32_t* topk_ids, int T, int k, int E, int with_shared, int32_t* offsets,
                int32_t* perm_src, int32_t* src_perm)
{
    int64_t n = (int64_t)T * k;
    int64_t* cursor = (int64_t*)calloc((size_t)E + 1, sizeof(int64_t));
    for (int64_t f = 0; f < n; ++f) {
        int32_t e = topk_ids[f];
        if (e < 0 || e >= E) {
            free(cursor);
            return -1;
        }
        cursor[e + 1] += 1;
    }
    for (int e = 0; e < E; ++e) cursor[e + 1] += cursor[e];
    for (int e = 0; e <= E; ++e) offsets[e] = (int32_t)cursor[e];
    offsets[E + 1] = (int32_t)(n + (with_shared ? T : 0));
    for (int64_t f = 0; f < n; ++f) { /* ascending f: stable */
        int64_t p = cursor[topk_ids[f]]++;
        perm_src[p] = (int32_t)f;
        src_perm[f] = (int32_t)p;
    }
    free(cursor);
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Grouped GEMM over dequantized NVFP4 operands, FP64 accumulation                              */
/* ------------------------------------------------------------------------------------------ */

/* For every group g and row p in [offsets[g], offsets[g+1]):
 *   out[p][n] = sum_k  A_hat[src(p)][k] * B_hat[g][n][k]
 * A: codes [*][K/2], sf [*][K/16], tensor scale a_scale[a_scale_per_group ? g : 0];
 *    src(p) = a_row ? a_row[p] : p.
 * B: codes [G][N][K/2], sf [G][N][K/16], scales b_scale[G][b_nscale]; with b_nscale == 2 the
 *    columns n < N/2 use b_scale[g][0] and the others b_scale[g][1] (gate | up halves).
 * out: [offsets[G]][N] (rows outside every group are left untouched). */
void orc_grouped_gemm(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_scale,
                      int a_scale_per_group, const int32_t* a_row, const int32_t* offsets, int G,
                      const uint8_t* b_codes, const uint8_t* b_sf, const float* b_scale, int b_nscale,
                      int N, int K, double* out)
{
    double* bhat = (double*)malloc(sizeof(double) * (size_t)N * (size_t)K);
    double* arow = NULL;
    for (int g = 0; g < G; ++g) {
        int64_t p0 = offsets[g], p1 = offsets[g + 1];
        if (p1 <= p0) continue;
        const uint8_t* bc = b_codes + (int64_t)g * N * (K / 2);
        const uint8_t* bs = b_sf + (int64_t)g * N * (K / 16);
        /* dequantize this group's B with its per-column-half scale */
        for (int h = 0; h < b_nscale; ++h) {
            int64_t n0 = (int64_t)h * N / b_nscale, n1 = (int64_t)(h + 1) * N / b_nscale;
            orc_dequantize_nvfp4(bc + n0 * (K / 2), bs + n0 * (K / 16), b_scale[(int64_t)g * b_nscale + h],
                                 n1 - n0, K, bhat + n0 * K);
        }
        float sa = a_scale[a_scale_per_group ? g : 0];
#pragma omp parallel private(arow)
        {
            arow = (double*)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
            for (int64_t p = p0; p < p1; ++p) {
                int64_t src = a_row ? a_row[p] : p;
                orc_dequantize_nvfp4(a_codes + src * (K / 2), a_sf + src * (K / 16), sa, 1, K, arow);
                for (int64_t n = 0; n < N; ++n) {
                    const double* bn = bhat + n * K;
                    double s = 0.0;
                    for (int64_t kk = 0; kk < K; ++kk) s += arow[kk] * bn[kk];
                    out[p * N + n] = s;
                }
            }
            free(arow);
        }
    }
    free(bhat);
}

/* ------------------------------------------------------------------------------------------ */
/* SwiGLU and combine                                                                           */
/* ------------------------------------------------------------------------------------------ */

/* gu: [P][2I] with gate in columns [0, I) and up in [I, 2I); h = silu(gate) * up in FP64,
 * rounded to FP32 (the precision the intermediate is requantized from). */
void orc_swiglu(const double* gu, int64_t P, int64_t I, float* h)
{
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < P; ++p) {
        for (int64_t n = 0; n < I; ++n) {
            double g = gu[p * 2 * I + n];
            double u = gu[p * 2 * I + I + n];
            h[p * I + n] = (float)(g / (1.0 + exp(-g)) * u);
        }
    }
}

/* out[t] = [residual[t] +] sum_j topk_w[t][j] * y[src_perm[t*k+j]] + shared_g[t] * y[shared_row0 + t]
 * in FP64; out_f64 keeps the unrounded value, out_bf16 the bf16 value (R8) as a double.
 * y rows are permuted rows; shared_g nullable (no shared expert); residual nullable. */
void orc_combine(const double* y, int T, int k, int64_t H, const double* topk_w,
                 const double* shared_g, int64_t shared_row0, const int32_t* src_perm,
                 const float* residual, double* out_f64, double* out_bf16)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int64_t c = 0; c < H; ++c) {
            double s = residual ? (double)residual[(int64_t)t * H + c] : 0.0;
            for (int j = 0; j < k; ++j) {
                int64_t p = src_perm[(int64_t)t * k + j];
                s += topk_w[(int64_t)t * k + j] * y[p * H + c];
            }
            if (shared_g) s += shared_g[t] * y[(shared_row0 + t) * H + c];
            if (out_f64) out_f64[(int64_t)t * H + c] = s;
            if (out_bf16) out_bf16[(int64_t)t * H + c] = orc_round_bf16(s);
        }
    }
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
