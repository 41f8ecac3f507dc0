// common.cuh -- shared device helpers of libmoe_nvfp4: workspace header, status codes, bf16 and
// NVFP4 element conversions.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

#include "ptx.cuh"

namespace moe {

// Device status bits (the status word of the workspace header).
enum : int {
    kDevOk = 0,
    kDevTimeoutGemm = 1,   // a bounded wait in the grouped GEMM ran out
    kDevBadExpertId = 2,   // moe_permute met an id outside [0, E)
    kDevTimeoutRouter = 4, // a bounded wait in the tensor-core router ran out
    kDevTimeoutCombine = 8, // a bounded wait in the streaming combine ran out
};

// First 256 bytes of every workspace.
struct WsHeader {
    int status;            // OR of kDev* bits
    unsigned amax_bits;    // bit pattern of amax(|x|) (non-negative floats order like integers)
    float s_x;             // tensor scale of the layer input
    unsigned ticket;       // CTAs of the one-launch front half that finished (zero between calls)
    int gemm_tiles;        // tile counter of a standalone grouped GEMM (cleared before its launch)
    unsigned perm_ticket;  // row-scan CTAs of the permutation that finished (zero between calls)
    // test hook of the expert GEMMs' wait for a token block's intermediate (both zero in normal
    // use): a wait limit in microseconds instead of the default, and an amount added to the count
    // that wait needs, so a test can make the wait run out without any fault
    unsigned test_wait_us;
    int test_ready_extra;
    int pad[56];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// Round to nearest even (finite inputs).
__device__ __forceinline__ uint32_t f32_to_bf16(float f)
{
    uint32_t u = __float_as_uint(f);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return u >> 16;
}

// Two floats as packed bf16 (round to nearest even; lo in bits 0..15) by one conversion instruction.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Exact value of a UE4M3 byte (code < 0x7F): e == 0 -> m * 2^-9, else 2^(e-7) * (1 + m/8).
__device__ __forceinline__ float ue4m3_to_f32(uint32_t c)
{
    const uint32_t e = (c >> 3) & 15u, m = c & 7u;
    return e == 0 ? static_cast<float>(m) * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// NVFP4 encoding of one 16-element block with tensor scale S (six_s = 6 * S, rounded to FP32):
// sf = UE4M3 nearest-even of amax / six_s (saturating at 448); codes = E2M1 nearest-even of
// v / (ue4m3(sf) * S) (saturating at 6, sign kept); all codes 0 when the scale decodes to 0.
// Every FP32 operation is a separately rounded IEEE operation, so the result does not depend on
// contraction or on the order of the max. Returns sf; writes 8 code bytes (element 2i in the low
// nibble of byte i) to lo (elements 0..7) and hi (8..15).
__device__ __forceinline__ uint32_t nvfp4_encode16(const float (&v)[16], float S, float six_s, uint32_t& lo,
                                                   uint32_t& hi)
{
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const float q = __fdiv_rn(amax, six_s);
    const uint32_t sf = ptx::cvt_e4m3x2(q, 0.0f) & 0xFFu;
    const float dsf = ue4m3_to_f32(sf);
    lo = 0u;
    hi = 0u;
    if (dsf != 0.0f) {
        const float d = __fmul_rn(dsf, S);
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            lo |= ptx::cvt_e2m1x2(__fdiv_rn(v[i], d), __fdiv_rn(v[i + 1], d)) << (4 * i);
            hi |= ptx::cvt_e2m1x2(__fdiv_rn(v[8 + i], d), __fdiv_rn(v[8 + i + 1], d)) << (4 * i);
        }
    }
    return sf;
}

__device__ __forceinline__ void record_status(int* status, int bits)
{
    if (status) atomicOr(status, bits);
}

}  // namespace moe
