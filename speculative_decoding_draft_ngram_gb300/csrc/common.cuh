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

// ---------------------------------------------------------------- checked build
// Compiled with SPECNG_CHECKED, every index that is computed from data (a
// vocabulary id, a history position, a draft slot, a logit element) is
// checked against its array before use: one outside [0, n) sets
// CHECKED_OOB and is clamped into range, so the access stays inside the
// array and nothing traps.  In the normal build chk() returns its argument.
#ifdef SPECNG_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

template <typename I>
__device__ __forceinline__ I chk(I idx, I n, unsigned* status) {
    if constexpr (kChecked) {
        if (idx < I(0) || idx >= n) {
            raise_status(status, SPECNG_DEV_CHECKED_OOB);
            return idx < I(0) ? I(0) : (n > I(0) ? n - I(1) : I(0));
        }
    }
    return idx;
}

// ---------------------------------------------------------------- launch chaining
// Programmatic dependent launch (sm_90+): a kernel launched with the
// programmatic-serialisation attribute may start before the previous kernel
// of its stream has finished.  It does the work that depends on nothing the
// previous kernel writes, then waits in pdl_wait() until that kernel has
// completed and its writes are visible.  pdl_trigger() lets the next kernel
// launch early (its own pdl_wait() still waits for this kernel's completion).
// Both are no-ops for a kernel launched without the attribute.

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `kernel` on stream s with programmatic stream serialisation.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                  Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
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

// Philox4x32-10 for counters that differ only in word 0 (the vocab block):
// with words 1..3 fixed, round 1's second product and round 2's first
// product do not depend on word 0, so they are computed once per row.
struct RowPhilox {
    uint32_t c3k1;     // c3 ^ k1 (round 1)
    uint32_t e2;       // lo(M1 c2) ^ (k0 + W0) (round 2)
    uint32_t f2;       // hi(M0 c0') ^ (k1 + W1) (round 2)
    uint32_t d2;       // lo(M0 c0') (round 2, output word 3)
    uint32_t k0, k1;   // original key
};

__device__ __forceinline__ RowPhilox row_philox(const NoiseKey& nk, uint32_t pos) {
    const uint32_t c1 = pos | (kPurposeGumbel << 16), c2 = nk.step, c3 = nk.seq;
    const uint32_t hi1 = __umulhi(kPhiloxM1, c2), lo1 = kPhiloxM1 * c2;
    const uint32_t c0p = hi1 ^ c1 ^ nk.k0;  // round-1 output word 0
    RowPhilox r;
    r.c3k1 = c3 ^ nk.k1;
    r.e2 = lo1 ^ (nk.k0 + kPhiloxW0);
    r.f2 = __umulhi(kPhiloxM0, c0p) ^ (nk.k1 + kPhiloxW1);
    r.d2 = kPhiloxM0 * c0p;
    r.k0 = nk.k0;
    r.k1 = nk.k1;
    return r;
}

// Same words as gumbel_block(nk, blk, pos) for the row that rp describes.
__device__ __forceinline__ uint4 gumbel_block_row(const RowPhilox& rp, uint32_t blk) {
    // round 1
    const uint64_t q0 = static_cast<uint64_t>(kPhiloxM0) * blk;
    const uint32_t hi0 = static_cast<uint32_t>(q0 >> 32), lo0 = static_cast<uint32_t>(q0);
    const uint32_t c2p = hi0 ^ rp.c3k1;
    // round 2 (c0' and c1' are row constants folded into e2 / f2 / d2)
    const uint64_t q1 = static_cast<uint64_t>(kPhiloxM1) * c2p;
    const uint32_t hi1 = static_cast<uint32_t>(q1 >> 32), lo1 = static_cast<uint32_t>(q1);
    uint4 c = make_uint4(hi1 ^ rp.e2, lo1, rp.f2 ^ lo0, rp.d2);
    uint32_t k0 = rp.k0 + 2u * kPhiloxW0, k1 = rp.k1 + 2u * kPhiloxW1;
#pragma unroll
    for (int r = 2; r < 10; ++r) {
        // one 32 x 32 -> 64-bit product per multiplier gives both halves
        const uint64_t p0 = static_cast<uint64_t>(kPhiloxM0) * c.x;
        const uint64_t p1 = static_cast<uint64_t>(kPhiloxM1) * c.z;
        c = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ c.y ^ k0, static_cast<uint32_t>(p1),
                       static_cast<uint32_t>(p0 >> 32) ^ c.w ^ k1, static_cast<uint32_t>(p0));
        k0 += kPhiloxW0;
        k1 += kPhiloxW1;
    }
    return c;
}

__device__ __forceinline__ uint32_t pick_word(const uint4& w, uint32_t lane) {
    return lane == 0 ? w.x : lane == 1 ? w.y : lane == 2 ? w.z : w.w;
}

// u = (2 (w >> 9) + 1) 2^-24: exact in fp32 and fp64, strictly inside (0, 1).
__device__ __forceinline__ uint32_t uniform_numerator(uint32_t w) { return ((w >> 9) << 1) | 1u; }

// Exp(1) variate -ln u of a Philox word; -log1p(u - 1) above 1/2, where u - 1
// is exact, keeps small values (the large Gumbel values) accurate.
__device__ __forceinline__ float exp_of_word(uint32_t w) {
    const float u = static_cast<float>(uniform_numerator(w)) * 0x1p-24f;
    return u > 0.5f ? -log1pf(u - 1.0f) : -logf(u);
}
__device__ __forceinline__ double exp_of_word_f64(uint32_t w) {
    const double u = static_cast<double>(uniform_numerator(w)) * 0x1p-24;
    return u > 0.5 ? -log1p(u - 1.0) : -log(u);
}

__device__ __forceinline__ double accept_uniform_f64(const NoiseKey& nk, uint32_t i) {
    const uint4 w = philox4x32_10(make_uint4(0u, i | (kPurposeAccept << 16), nk.step, nk.seq), nk.k0, nk.k1);
    return static_cast<double>(uniform_numerator(w.x)) * 0x1p-24;
}

// ---------------------------------------------------------------- sampling noise
// The sampler's noise is g_v = -ln E_v with E_v i.i.d. Exp(1), drawn per block
// of 256 vocab ids through the Renyi representation of exponential order
// statistics: one block draw gives the block minimum M ~ Exp(256) (word 0,
// scaled by 2^-8) and the slot I of the id holding it (word 1, low 8 bits,
// uniform); every other id adds its own Exp(1) draw F_v, E_v = M + F_v.  Any
// score of the block is therefore at most log w_v - ln M, which prunes whole
// blocks before a single per-id draw is made.

constexpr uint32_t kPurposeBlock = 2u;
constexpr int kNoiseBlockShift = 8;
constexpr uint32_t kNoiseBlockMask = (1u << kNoiseBlockShift) - 1u;

__device__ __forceinline__ uint4 block_words(const NoiseKey& nk, uint32_t blk, uint32_t pos) {
    return philox4x32_10(make_uint4(blk, pos | (kPurposeBlock << 16), nk.step, nk.seq), nk.k0, nk.k1);
}

struct BlockNoise {
    float M, lnM;  // block minimum and its logarithm (fp32)
    int I;         // slot (v & 255) of the id whose E is M
    int pad;
};


// Screening precision (fp32 scores that only order candidates; every final
// decision between close scores is re-taken in fp64).  -ln u for a Philox
// word: above 1/2, with x = u - 1 (exact) and s = x / (2 + x),
// -ln u = -log1p(x) = -2 atanh(s) = -2 s (1 + s^2/3 + s^4/5 + s^6/7 + s^8/9 + ...),
// |s| <= 1/3, truncated after s^8/9 (relative error below 2e-6); below 1/2,
// -ln u >= ln 2 and the hardware logarithm's error is relative to it.
__device__ __forceinline__ float exp_of_word_fast(uint32_t w) {
    const float u = static_cast<float>(uniform_numerator(w)) * 0x1p-24f;
    if (u > 0.5f) {
        const float x = u - 1.0f;
        const float sv = __fdividef(x, 2.0f + x);
        const float s2 = sv * sv;
        const float poly = fmaf(s2, fmaf(s2, fmaf(s2, fmaf(s2, 1.0f / 9.0f, 1.0f / 7.0f), 0.2f), 1.0f / 3.0f), 1.0f);
        return -2.0f * sv * poly;
    }
    return -__logf(u);
}

// E_v in fp32 for an id of a block with minimum M and argmin slot I (rp: the row's element draws).
__device__ __forceinline__ float noise_exp_f32(const RowPhilox& rp, float M, int I, uint32_t v) {
    if (static_cast<int>(v & kNoiseBlockMask) == I) return M;
    return M + exp_of_word_fast(pick_word(gumbel_block_row(rp, v >> 2), v & 3u));
}

// ln E at screening precision: 3 ulp of |ln E| (hardware logarithm).
__device__ __forceinline__ float ln_fast(float e) { return __logf(e); }

// A block's draw at screening precision (the bound ln M is off by a few ulp at
// most, far inside the slack every comparison with it carries).
__device__ __forceinline__ BlockNoise block_noise(const NoiseKey& nk, uint32_t blk, uint32_t pos) {
    const uint4 w = block_words(nk, blk, pos);
    BlockNoise r;
    r.M = exp_of_word_fast(w.x) * 0x1p-8f;
    r.lnM = ln_fast(r.M);
    r.I = static_cast<int>(w.y & kNoiseBlockMask);
    r.pad = 0;
    return r;
}

// E_v in fp64, the oracle's arithmetic, for the final decisions.
__device__ __forceinline__ double noise_exp_f64(const NoiseKey& nk, uint32_t v, uint32_t pos) {
    const uint4 bw = block_words(nk, v >> kNoiseBlockShift, pos);
    const double M = exp_of_word_f64(bw.x) * 0x1p-8;
    if ((v & kNoiseBlockMask) == (bw.y & kNoiseBlockMask)) return M;
    return M + exp_of_word_f64(pick_word(gumbel_block(nk, v >> 2, pos), v & 3u));
}

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

// ---------------------------------------------------------------- TMA bulk
// 1-D bulk copies global -> shared completing on an mbarrier (sm_90+ PTX).

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Raise the expected transaction bytes of the current phase without arriving.
__device__ __forceinline__ void mbar_add_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0u;
}

// Wait for a phase of an mbarrier, giving up after a bounded number of polls
// (well under a second): a copy that never lands is reported, not waited on.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity) {
    for (int it = 0; it < (1 << 22); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (it >= 32) __nanosleep(64);
    }
    return false;
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
