// topk.cuh -- warp-level pieces of the FP32 top-k (lowest expert id first on equal logits).
#pragma once
#include <cstdint>

namespace moe {

// Order-preserving key of a logit: a larger logit has a larger key; every logit, -inf included, has
// a key >= 1, and NaN ranks with -inf (so the selected ids always lie in [0, E)).
__device__ __forceinline__ uint32_t order_key(float v)
{
    if (v != v) v = -INFINITY;
    if (v == 0.0f) v = 0.0f;  // -0 ties with +0
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// A lane's four largest keys not yet taken (bit i of `taken` set: slot i is gone), largest first
// (equal keys: lowest slot first); unused entries hold 0. The keys stay read-only so the array lives
// in registers.
struct Top4 {
    uint32_t k[4];
    int s[4];
};

__device__ __forceinline__ void lane_top4(const uint32_t (&key)[32], uint32_t taken, Top4& c)
{
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        c.k[q] = 0u;
        c.s[q] = 31;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        uint32_t kv = ((taken >> i) & 1u) ? 0u : key[i];
        int sv = i;
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // insertion: a strictly larger key moves ahead
            const bool gt = kv > c.k[q];
            const uint32_t tk = gt ? c.k[q] : kv;
            const int ts = gt ? c.s[q] : sv;
            c.k[q] = gt ? kv : c.k[q];
            c.s[q] = gt ? sv : c.s[q];
            kv = tk;
            sv = ts;
        }
    }
}

// One warp: the k (<= 32) largest of the E (<= 1024) logits l[0..E) in (logit desc, id asc)
// order. Lane l holds logits l, l + 32, ... as keys plus a cache of its four largest; a round takes
// the warp's largest cached key with one reduction and the lowest id holding it with a second, and
// only the winning lane pops its cache (rebuilding it from its remaining keys when it runs empty).
// Lane j < k returns the j-th logit and id; every lane returns the largest logit in l0.
__device__ __forceinline__ void warp_topk(const float* l, int E, int k, float& sel_l, int& sel_i, float& l0)
{
    const int lane = threadIdx.x & 31;
    uint32_t key[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int ee = i * 32 + lane;
        key[i] = ee < E ? order_key(__ldcg(l + ee)) : 0u;
    }
    Top4 c;
    uint32_t taken = 0;
    lane_top4(key, taken, c);
    sel_l = 0.0f;
    sel_i = 0;
    uint32_t k0 = 0;
    for (int j = 0; j < k; ++j) {
        const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, c.k[0]);
        const int widx = static_cast<int>(__reduce_min_sync(
            0xFFFFFFFFu, c.k[0] == wmax ? static_cast<unsigned>(c.s[0] * 32 + lane) : 0x7FFFFFFFu));
        if (j == 0) k0 = wmax;
        if (lane == j) {
            sel_l = key_value(wmax);
            sel_i = widx;
        }
        if ((widx & 31) == lane) {
            taken |= 1u << c.s[0];
#pragma unroll
            for (int q = 0; q < 3; ++q) {
                c.k[q] = c.k[q + 1];
                c.s[q] = c.s[q + 1];
            }
            c.k[3] = 0u;
            c.s[3] = 31;
            if (c.k[0] == 0u) lane_top4(key, taken, c);
        }
    }
    l0 = key_value(k0);
}

// Capacity of the candidate list of warp_topk_threshold, per warp.
constexpr int kTopkCand = 64;

// One warp, the same selection as warp_topk in a few straight-line steps, for E <= 32 * kNper and
// k <= 32. Lane l holds logits l, l + 32, ... as keys; tau = the k-th largest of the 32 lane maxima
// (lowest lane first on ties). At least k logits reach tau (those k maxima), so every logit of the
// top k does: the candidates are the keys >= tau, compacted into cand[] (kTopkCand entries of
// shared memory per warp) in lane order by a warp prefix sum. Each candidate's place is the number
// of candidates ahead of it in (key desc, id asc) order; the first k places are the result, written
// to out[] (k entries of shared memory). Returns false, with nothing selected, when more than
// kTopkCand logits reach tau (many equal logits): the caller then runs warp_topk.
template <int kNper>
__device__ __forceinline__ bool warp_topk_threshold(const float* l, int E, int k, uint2* cand, uint2* out,
                                                    float& sel_l, int& sel_i, float& l0)
{
    const int lane = threadIdx.x & 31;
    uint32_t key[kNper];
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < kNper; ++i) {
        const int ee = i * 32 + lane;
        key[i] = ee < E ? order_key(__ldcg(l + ee)) : 0u;
        m = max(m, key[i]);
    }
    int rank = 0;  // of this lane's maximum among the 32
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const uint32_t mj = __shfl_sync(0xFFFFFFFFu, m, j);
        rank += (mj > m) | ((mj == m) & (j < lane));
    }
    const unsigned at_k = __ballot_sync(0xFFFFFFFFu, rank == k - 1);
    const uint32_t tau = __shfl_sync(0xFFFFFFFFu, m, __ffs(at_k) - 1);
    int c = 0;
#pragma unroll
    for (int i = 0; i < kNper; ++i) c += key[i] >= tau;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
    }
    const int C = __shfl_sync(0xFFFFFFFFu, incl, 31);
    if (C > kTopkCand) return false;
    int pos = incl - c;
#pragma unroll
    for (int i = 0; i < kNper; ++i)
        if (key[i] >= tau) cand[pos++] = make_uint2(key[i], static_cast<uint32_t>(i * 32 + lane));
    __syncwarp();
    for (int j = lane; j < C; j += 32) {
        const uint2 me = cand[j];
        int r = 0;
        for (int q = 0; q < C; ++q) {
            const uint2 o = cand[q];
            r += (o.x > me.x) | ((o.x == me.x) & (o.y < me.y));
        }
        if (r < k) out[r] = me;
    }
    __syncwarp();
    const uint2 s = out[lane < k ? lane : 0];
    sel_l = lane < k ? key_value(s.x) : 0.0f;
    sel_i = lane < k ? static_cast<int>(s.y) : 0;
    l0 = key_value(out[0].x);
    __syncwarp();
    return true;
}

// Renormalised routing weight of lane j < k: the softmax over the selected logits (the full
// softmax denominator cancels); l0 is the largest selected logit.
__device__ __forceinline__ float warp_topk_weight(float sel_l, float l0, int k)
{
    const int lane = threadIdx.x & 31;
    const float p = lane < k ? expf(sel_l - l0) : 0.0f;
    float sum = p;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    return p / sum;
}

}  // namespace moe
