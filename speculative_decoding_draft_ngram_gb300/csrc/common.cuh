// Internal device helpers of libspecng (sm_103a).  Not part of the C ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/specng.h"

namespace specng {

// ---------------------------------------------------------------- status

__device__ __forceinline__ void raise_status(unsigned* status, unsigned bit) {
    if (status != nullptr) atomicOr(status, bit);
}

// ---------------------------------------------------------------- Philox
// Philox4x32-10 as defined by Salmon, Moraes, Dror and Shaw, "Parallel random
// numbers: as easy as 1, 2, 3" (SC'11): per round the two multiplier products
// of counter words 0 and 2 are taken hi/lo, the high halves are xored with
// the other two words and the key, and the key advances by the Weyl
// increments between rounds.

constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(kPhiloxM0, c.x);
        const uint32_t lo0 = kPhiloxM0 * c.x;
        const uint32_t hi1 = __umulhi(kPhiloxM1, c.z);
        const uint32_t lo1 = kPhiloxM1 * c.z;
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += kPhiloxW0;
        k1 += kPhiloxW1;
    }
    return c;
}

// Counter layout of the sampler's noise.
constexpr uint32_t kPurposeGumbel = 0u;
constexpr uint32_t kPurposeAccept = 1u;

struct NoiseKey {
    uint32_t k0, k1, step, seq;
};

// The four Philox words that serve vocab ids 4*blk .. 4*blk+3 of row pos.
__device__ __forceinline__ uint4 gumbel_block(const NoiseKey& nk, uint32_t blk, uint32_t pos) {
    return philox4x32_10(make_uint4(blk, pos | (kPurposeGumbel << 16), nk.step, nk.seq), nk.k0, nk.k1);
}

__device__ __forceinline__ uint32_t pick_word(const uint4& w, uint32_t lane) {
    return lane == 0 ? w.x : lane == 1 ? w.y : lane == 2 ? w.z : w.w;
}

// u = (2 (w >> 9) + 1) 2^-24: exact in fp32 and fp64, strictly inside (0, 1).
__device__ __forceinline__ uint32_t uniform_numerator(uint32_t w) { return ((w >> 9) << 1) | 1u; }

__device__ __forceinline__ float gumbel_f32(uint32_t w) {
    const float u = static_cast<float>(uniform_numerator(w)) * 0x1p-24f;
    const float e = u > 0.5f ? -log1pf(u - 1.0f) : -logf(u);
    return -logf(e);
}

__device__ __forceinline__ double gumbel_f64(uint32_t w) {
    const double u = static_cast<double>(uniform_numerator(w)) * 0x1p-24;
    const double e = u > 0.5 ? -log1p(u - 1.0) : -log(u);
    return -log(e);
}

__device__ __forceinline__ double accept_uniform_f64(const NoiseKey& nk, uint32_t i) {
    const uint4 w = philox4x32_10(make_uint4(0u, i | (kPurposeAccept << 16), nk.step, nk.seq), nk.k0, nk.k1);
    return static_cast<double>(uniform_numerator(w.x)) * 0x1p-24;
}

// Upper bound of a Gumbel draw on the 2^-24 grid (-ln(-ln(1 - 2^-24)) = 16.6355),
// with slack for fp32 rounding.
constexpr float kGumbelMax = 16.7f;

// Candidates whose fp32 score is below (best - delta) cannot win once the
// final choice is re-scored in fp64: delta is far above the fp32 error of a
// score (a few ulps of |score| plus the logarithms' error).
__device__ __forceinline__ float cand_delta(float s) { return 1e-4f + fabsf(s) * 1e-6f; }

// ---------------------------------------------------------------- numerics

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kLog2e = 1.4426950408889634f;

// Order used by every candidate merge: higher score first, lower id on ties.
__device__ __forceinline__ bool better(float s, int id, float t, int jd) {
    return s > t || (s == t && static_cast<unsigned>(id) < static_cast<unsigned>(jd));
}
__device__ __forceinline__ bool better64(double s, int id, double t, int jd) {
    return s > t || (s == t && static_cast<unsigned>(id) < static_cast<unsigned>(jd));
}

struct Top2 {
    float s1, s2;
    int i1, i2;
};

__device__ __forceinline__ Top2 top2_empty() { return Top2{-INFINITY, -INFINITY, -1, -1}; }

__device__ __forceinline__ void top2_push(Top2& t, float s, int id) {
    if (better(s, id, t.s1, t.i1)) {
        t.s2 = t.s1; t.i2 = t.i1; t.s1 = s; t.i1 = id;
    } else if (better(s, id, t.s2, t.i2)) {
        t.s2 = s; t.i2 = id;
    }
}

__device__ __forceinline__ Top2 top2_merge(const Top2& a, const Top2& b) {
    Top2 r;
    if (better(b.s1, b.i1, a.s1, a.i1)) {
        r.s1 = b.s1; r.i1 = b.i1;
        if (better(a.s1, a.i1, b.s2, b.i2)) { r.s2 = a.s1; r.i2 = a.i1; } else { r.s2 = b.s2; r.i2 = b.i2; }
    } else {
        r.s1 = a.s1; r.i1 = a.i1;
        if (better(b.s1, b.i1, a.s2, a.i2)) { r.s2 = b.s1; r.i2 = b.i1; } else { r.s2 = a.s2; r.i2 = a.i2; }
    }
    return r;
}

__device__ __forceinline__ Top2 top2_shfl_xor(const Top2& t, int off) {
    Top2 o;
    o.s1 = __shfl_xor_sync(0xffffffffu, t.s1, off);
    o.s2 = __shfl_xor_sync(0xffffffffu, t.s2, off);
    o.i1 = __shfl_xor_sync(0xffffffffu, t.i1, off);
    o.i2 = __shfl_xor_sync(0xffffffffu, t.i2, off);
    return o;
}

__device__ __forceinline__ Top2 top2_warp_reduce(Top2 t) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t = top2_merge(t, top2_shfl_xor(t, off));
    return t;
}

// Streaming 16-byte load: read once, do not keep in L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
}

// ---------------------------------------------------------------- hashing
// splitmix64 finaliser (Steele, Lea, Flood, "Fast splittable pseudorandom
// number generators", OOPSLA 2014): a bijective 64-bit mixer.
__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

}  // namespace specng
