// spec_verify kernels (sm_103a): the streaming pass over the logit rows, the
// per-sequence decision kernel, and the dense-q residual pass.
//
// Method (SwiftLM page, paragraph on algorithmic equivalence after Leviathan
// et al.; AX Engine page, "Core Technical Architecture & Methods"):
//   row transform  soft cap -> repetition penalty -> temperature
//   p_j = softmax(x_j / T); accept draft i iff u_i q(d_i) <= p(d_i)
//   a = number accepted before the first rejection (<= k_eff, EMA gate)
//   sample at row a: residual max(0, p_a - q_a) on a rejection, p_a (bonus)
//   otherwise, by Gumbel-max argmax_v (log w_v - ln E_v); T = 0: argmax
//   epilogue: tokens, kv_len <- kv_len - k + a, EMA update.
//
// The noise E_v is drawn per block of 256 ids (block minimum M and its slot,
// then E_v = M + F_v for the others; see common.cuh), so a score of a block is
// at most z_max / T - ln M, with z_max the transform of the block's largest
// logit (a bound of the block's transformed logits).
// The streaming pass (bandwidth only) leaves, per row, the segment sums of
// the softmax and every block's z_max; the decision kernel takes the accept
// tests from the sums, and only then samples, at row a alone, reading again
// just the blocks whose bound reaches the best score found.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace specng {

template <bool BF16> struct ElemTraits;
template <> struct ElemTraits<true> { static constexpr int EPV = 8; static constexpr int SIZE = 2; };
template <> struct ElemTraits<false> { static constexpr int EPV = 4; static constexpr int SIZE = 4; };

// One chunk of a row = one 64 KB stage of the streaming ring; the residual
// pass takes 32 KB chunks, one per CTA.
constexpr int kChunkBytes = 65536;
constexpr int kResChunkBytes = 32768;
template <bool BF16>
__host__ __device__ constexpr int chunk_elems() { return kChunkBytes / ElemTraits<BF16>::SIZE; }
template <bool BF16>
__host__ __device__ constexpr int res_chunk_elems() { return kResChunkBytes / ElemTraits<BF16>::SIZE; }

// Noise blocks of a row of V ids.
__host__ __device__ constexpr int noise_blocks(int V) { return (V + (1 << kNoiseBlockShift) - 1) >> kNoiseBlockShift; }

// Workspace records.
struct __align__(8) SegSum {
    float m, s;  // reference (transformed units) and sum of exp((z - m) / T) of a row segment;
                 // s < 0: the segment holds a value that proves the row's accept test rejects
};
struct __align__(32) Partial {
    float m, s;
    Top2 t;      // top-two candidates (fp32 scores)
    int pad[2];
};
struct __align__(16) RowRes {
    float m, S;    // the row's softmax normaliser: lse = m / T + ln S (T > 0)
    int winner, pad;
};
struct __align__(16) SeqRes {
    int a, keff, need_residual, pad;
};

// Per-block scratch of the decision kernel (bound, M, slot, list entry).
constexpr int kBlkScratchBytes = 16;
// Blocks whose scratch the decision kernel keeps in shared memory (64 KB);
// longer rows keep it in the workspace.
constexpr int kSmemBlkCap = 4096;

struct VerifyDev {
    const void* logits;
    int B, K, V, nchunk;      // nchunk: streaming chunks per row
    int nchunk2;              // residual-pass chunks per row
    int nblk;                 // noise blocks per row
    const int32_t* drafts;
    const float* q;
    const int32_t* k;
    const int32_t* hist;
    int64_t hist_stride;
    const int32_t* lens;
    float T, invT, sc;        // temperature, 1/T, log2(e)/T
    double Td;                // (double)T
    float cap, invcap;        // soft cap c and 1/c
    float cap2l;              // 2 log2(e) / c (soft cap inside the sums of exponentials)
    float rep, invrep;        // repetition penalty r and 1/r
    int W;                    // penalty window
    float tau, thresh;
    int gate;
    NoiseKey nk;              // seq filled per row
    int aligned;              // logits (and q) allow 16-byte vector loads
    int32_t* kv_len;
    float* ema;
    int32_t* out_tokens;
    int32_t* out_accept;
    SegSum* part;             // [B (K + 1)][nchunk] segment sums, at each segment's last chunk
    float* bmax;              // [B (K + 1)][nblk] largest raw logit of each noise block
    uint8_t* blkws;           // [B][nblk][16] decision-kernel block scratch (rows past kSmemBlkCap blocks)
    RowRes* rowres;
    SeqRes* seqres;
    unsigned* row_thr;        // best residual score published per row (score_key)
    Partial* part2;
    unsigned* seq_ticket2;
    unsigned* status;
    unsigned* diag;           // SPECNG_DIAG_* counters of the exact (fp64) paths
    // single-kernel schedule
    unsigned long long* row_tix;    // [B (K + 1)] chunks streamed per row: epoch:32 | count:32
    unsigned long long* seq_state;  // [B] rows done / accepted this call: epoch:31 | bits:33
    float* ema_new;                 // [B] updated EMA, copied to ema by the grid's last CTA
    unsigned* grid_tix;             // CTAs finished
    uint32_t epoch;                 // this call's tag, in [1, 2^31)
    int early_exit;                 // rows past a known first rejection are not streamed
    int fused;                      // 1: single-kernel schedule
    int records_given;              // 1: the fused LM-head kernel wrote the records (no streaming pass)
    // gate variants
    int probe;                      // re-probe interval (0: none)
    uint64_t step64;                // the call's decode step (host argument)
    const uint64_t* step_dev;       // device step counter, read instead when not NULL
    int cool;                       // cooling calls after a partial acceptance (0: none)
    int32_t* gate_state;            // [B] cooling counts, in/out (NULL when cool == 0)
    int32_t* cool_new;              // [B] single-kernel schedule: updated counts, copied by the last CTA
};

// Checked-build accessors (plain accesses in the normal build).
__device__ __forceinline__ size_t chk_row(const VerifyDev& P, size_t row) {
    return chk<size_t>(row, static_cast<size_t>(P.B) * (P.K + 1), P.status);
}
__device__ __forceinline__ int chk_id(const VerifyDev& P, int v) { return chk<int>(v, P.V, P.status); }
// History token at position pos of sequence b.
__device__ __forceinline__ int hist_at(const VerifyDev& P, int b, int64_t pos) {
    return P.hist[static_cast<size_t>(chk<int>(b, P.B, P.status)) * P.hist_stride +
                  chk<int64_t>(pos, P.hist_stride, P.status)];
}
// Draft d_{j+1} of sequence b.
__device__ __forceinline__ int draft_at(const VerifyDev& P, int b, int j) {
    return P.drafts[static_cast<size_t>(chk<int>(b, P.B, P.status)) * P.K + chk<int>(j, P.K, P.status)];
}

// Count one run of a rarely taken exact path (see SPECNG_DIAG_*).
__device__ __forceinline__ void count_diag(const VerifyDev& P, int which) {
    if (P.diag != nullptr) atomicAdd(P.diag + which, 1u);
}
// ---------------------------------------------------------------- helpers

template <bool BF16>
__device__ __forceinline__ void unpack(const uint4& r, float* x) {
    if constexpr (BF16) {
        x[0] = bf16lo(r.x); x[1] = bf16hi(r.x); x[2] = bf16lo(r.y); x[3] = bf16hi(r.y);
        x[4] = bf16lo(r.z); x[5] = bf16hi(r.z); x[6] = bf16lo(r.w); x[7] = bf16hi(r.w);
    } else {
        x[0] = __uint_as_float(r.x); x[1] = __uint_as_float(r.y);
        x[2] = __uint_as_float(r.z); x[3] = __uint_as_float(r.w);
    }
}

template <bool BF16>
__device__ __forceinline__ uint4 load_vec(const char* rowp, int e0, int v1, bool aligned) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    if (aligned) return ld_stream16(rowp + static_cast<size_t>(e0) * ElemTraits<BF16>::SIZE);
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
        const int v = e0 + e;
        if (v < v1) {
            if constexpr (BF16) {
                const uint32_t h = reinterpret_cast<const uint16_t*>(rowp)[v];
                w[e >> 1] |= (e & 1) ? (h << 16) : h;
            } else {
                w[e] = reinterpret_cast<const uint32_t*>(rowp)[v];
            }
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <bool BF16>
__device__ __forceinline__ double raw_logit_f64(const void* logits, size_t row, int V, int id);
// Raw logit id of row `row`, index-checked in the checked build.
template <bool BF16>
__device__ __forceinline__ double raw_logit_chk(const VerifyDev& P, size_t row, int id) {
    return raw_logit_f64<BF16>(P.logits, chk_row(P, row), P.V, chk_id(P, id));
}
// Vector load of row elements e0.. below v1 (see load_vec), e0 checked in the checked build.
template <bool BF16>
__device__ __forceinline__ uint4 load_vec(const char* rowp, int e0, int v1, bool aligned);
template <bool BF16>
__device__ __forceinline__ uint4 load_vec_chk(const VerifyDev& P, const char* rowp, int e0, int v1) {
    return load_vec<BF16>(rowp, chk<int>(e0, v1, P.status), v1, P.aligned);
}

template <bool BF16>
__device__ __forceinline__ double raw_logit_f64(const void* logits, size_t row, int V, int id) {
    if constexpr (BF16) {
        const uint16_t h = reinterpret_cast<const uint16_t*>(logits)[row * V + id];
        return static_cast<double>(__uint_as_float(static_cast<uint32_t>(h) << 16));
    } else {
        return static_cast<double>(reinterpret_cast<const float*>(logits)[row * V + id]);
    }
}

template <bool BF16>
__device__ __forceinline__ float elem_of_stage(const uint4* stage, int loc) {
    if constexpr (BF16) {
        return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(stage)[loc]) << 16);
    } else {
        return reinterpret_cast<const float*>(stage)[loc];
    }
}

// fp32 transform of one element: soft cap, then repetition penalty.
template <bool SOFTCAP, bool PENALTY>
__device__ __forceinline__ float transform_f32(float x, bool pen, const VerifyDev& P) {
    float z = x;
    if constexpr (SOFTCAP) z = P.cap * tanhf(x * P.invcap);
    if constexpr (PENALTY) {
        if (pen) z = z > 0.0f ? z * P.invrep : z * P.rep;
    }
    return z;
}

// The soft cap inside the sums of exponentials, from the identity
// c tanh(x / c) = c - 2c / (exp(2x / c) + 1) with the hardware 2^x and
// reciprocal: two special-function operations instead of an accurate tanh.
// Its absolute error is a few 1e-6 of c; the sums only screen the accept
// tests, whose decisions inside a 1e-4 band are taken again.
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
template <bool SOFTCAP>
__device__ __forceinline__ float sum_transform(float x, const VerifyDev& P) {
    if constexpr (!SOFTCAP) {
        return x;
    } else {
        const float e = ex2_approx(x * P.cap2l);  // exp(2x / c)
        return fmaf(-2.0f * P.cap, rcp_approx(e + 1.0f), P.cap);
    }
}
template <bool SOFTCAP>
__device__ __forceinline__ float sum_transform_pen(float x, const VerifyDev& P) {
    const float z = sum_transform<SOFTCAP>(x, P);
    return z > 0.0f ? z * P.invrep : z * P.rep;
}

// fp64 transform, the same definition in the oracle's precision.
template <bool SOFTCAP, bool PENALTY>
__device__ __forceinline__ double transform_f64(double x, bool pen, const VerifyDev& P) {
    double z = x;
    if constexpr (SOFTCAP) {
        const double c = static_cast<double>(P.cap);
        z = c * tanh(x / c);
    }
    if constexpr (PENALTY) {
        if (pen) {
            const double r = static_cast<double>(P.rep);
            z = z > 0.0 ? z / r : z * r;
        }
    }
    return z;
}

// Is id in the penalty window held in shared memory?  Whole warp calls it.
__device__ __forceinline__ bool warp_in_window(int id, const int* s_win, int nw) {
    bool f = false;
    for (int t = threadIdx.x & 31; t < nw; t += 32) f |= (s_win[t] == id);
    return __any_sync(0xffffffffu, f);
}

__device__ __forceinline__ Partial ldcg_partial(const Partial* p) {
    const uint4 a = __ldcg(reinterpret_cast<const uint4*>(p));
    const uint4 b = __ldcg(reinterpret_cast<const uint4*>(p) + 1);
    Partial r;
    r.m = __uint_as_float(a.x);
    r.s = __uint_as_float(a.y);
    r.t.s1 = __uint_as_float(a.z);
    r.t.s2 = __uint_as_float(a.w);
    r.t.i1 = static_cast<int>(b.x);
    r.t.i2 = static_cast<int>(b.y);
    return r;
}

__device__ __forceinline__ void st_partial(Partial* p, float m, float s, const Top2& t) {
    reinterpret_cast<uint4*>(p)[0] =
        make_uint4(__float_as_uint(m), __float_as_uint(s), __float_as_uint(t.s1), __float_as_uint(t.s2));
    reinterpret_cast<uint4*>(p)[1] = make_uint4(static_cast<unsigned>(t.i1), static_cast<unsigned>(t.i2), 0u, 0u);
}

template <typename R>
__device__ __forceinline__ void st_zero(R* p) {
    static_assert(sizeof(R) % 16 == 0, "record size");
#pragma unroll
    for (int i = 0; i < static_cast<int>(sizeof(R) / 16); ++i) reinterpret_cast<uint4*>(p)[i] = make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Order-preserving map of a float score to an unsigned key (0 = "none").
__device__ __forceinline__ unsigned score_key(float f) {
    const unsigned u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_score(unsigned k) {
    if (k == 0u) return -INFINITY;
    return (k & 0x80000000u) ? __uint_as_float(k & 0x7FFFFFFFu) : __uint_as_float(~k);
}

__device__ __forceinline__ unsigned warp_best_key(float best) {
    return __reduce_max_sync(0xffffffffu, best > -INFINITY ? score_key(best) : 0u);
}

// Largest bf16 value <= f, as a packed pair (both halves).  NaN maps to +inf.
__device__ __forceinline__ uint32_t bf16x2_floor(float f) {
    uint32_t u = __float_as_uint(f);
    if (f != f) u = 0x7F800000u;
    uint32_t h = u >> 16;
    if ((u & 0x80000000u) && (u & 0xFFFFu) && (u & 0x7FFFFFFFu) < 0x7F800000u) h += 1u;  // negative: away from 0
    return h | (h << 16);
}

__device__ __forceinline__ __nv_bfloat162 as_bf162(uint32_t w) { return *reinterpret_cast<__nv_bfloat162*>(&w); }
__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Packed maximum of the 8 bf16 values of a 16-byte vector (both halves hold a partial maximum).
__device__ __forceinline__ __nv_bfloat162 bf16x8_max2(const uint4& r) {
    return __hmax2(__hmax2(as_bf162(r.x), as_bf162(r.y)), __hmax2(as_bf162(r.z), as_bf162(r.w)));
}
// The same with NaN propagated (a NaN element makes its half NaN).
__device__ __forceinline__ __nv_bfloat162 bf16x8_max2_nan(const uint4& r) {
    return __hmax2_nan(__hmax2_nan(as_bf162(r.x), as_bf162(r.y)), __hmax2_nan(as_bf162(r.z), as_bf162(r.w)));
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float y;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
    return y;
}

// Bit e set when element e of the vector is >= the (packed) threshold t: the
// high byte of each compared half is gathered with byte permutes, and the four
// 0xFF / 0x00 bytes of a word become four bits by one multiply (the partial
// products of distinct bytes land on distinct bit positions, so nothing
// carries into bits 24..27).
__device__ __forceinline__ unsigned bf16x8_ge_bits(const uint4& r, uint32_t t) {
    const __nv_bfloat162 th = as_bf162(t);
    const unsigned m0 = __hge2_mask(as_bf162(r.x), th), m1 = __hge2_mask(as_bf162(r.y), th);
    const unsigned m2 = __hge2_mask(as_bf162(r.z), th), m3 = __hge2_mask(as_bf162(r.w), th);
    const unsigned b03 = __byte_perm(m0, m1, 0x7531u) & 0x01010101u;  // elements 0..3, one byte each
    const unsigned b47 = __byte_perm(m2, m3, 0x7531u) & 0x01010101u;  // elements 4..7
    return ((b03 * 0x01020408u) >> 24) | (((b47 * 0x01020408u) >> 24) << 4);
}

// Merge (m, s) pairs whose sums are relative to their own maxima.
__device__ __forceinline__ void ms_merge(float& m, float& s, float mo, float so, float sc) {
    const float M = fmaxf(m, mo);
    float r = 0.0f;
    if (m > -INFINITY) r += s * ex2_approx((m - M) * sc);
    if (mo > -INFINITY) r += so * ex2_approx((mo - M) * sc);
    m = M;
    s = r;
}

// Penalty window of row j: the last W tokens of history ++ d_1..d_j, read
// from the history tail and the drafts (shared or global memory).
struct WindowView {
    const int* hwin;    // last nh history tokens
    const int* drafts;  // d_1..d_k
    int nh, W;

    __device__ __forceinline__ int count(int j) const {
        const int total = nh + j;
        return total < W ? total : W;
    }
    __device__ __forceinline__ int token(int j, int t) const {  // t-th token of row j's window
        const int total = nh + j;
        const int idx = total - count(j) + t;
        return idx < nh ? hwin[idx] : drafts[idx - nh];
    }
    // whole warp calls it
    __device__ __forceinline__ bool warp_has(int j, int id) const {
        bool f = false;
        const int n = count(j);
        for (int t = threadIdx.x & 31; t < n; t += 32) f |= token(j, t) == id;
        return __any_sync(0xffffffffu, f);
    }
};

// The EMA's rate a / k_eff in fp64 (correctly rounded, as a division gives it),
// tabulated at compile time: a division in fp64 is a long sequence of fp64
// operations, slow on this GPU, at the end of every sequence's decision.
struct RateTable {
    double v[SPECNG_MAX_K + 1][SPECNG_MAX_K + 1];  // [k_eff][a]
};
constexpr RateTable make_rate_table() {
    RateTable t{};
    for (int k = 1; k <= SPECNG_MAX_K; ++k)
        for (int a = 0; a <= k; ++a) t.v[k][a] = static_cast<double>(a) / static_cast<double>(k);
    return t;
}
__constant__ const RateTable c_rate = make_rate_table();
__device__ __forceinline__ double ema_rate(int a, int keff) { return c_rate.v[keff][a]; }

// EMA after a call with k_eff > 0 drafts and a accepted: (1 - tau) ema + tau a / k_eff,
// each operation rounded in fp64 (no contraction), then to fp32.
__device__ __forceinline__ float ema_update(float ema, float tau, int a, int keff) {
    const double t = static_cast<double>(tau);
    return static_cast<float>(__dadd_rn(__dmul_rn(1.0 - t, static_cast<double>(ema)), __dmul_rn(t, ema_rate(a, keff))));
}

// The call's decode step: the device counter when one is given (a call replayed
// from a CUDA graph keeps its host arguments), else the host argument.
__device__ __forceinline__ uint64_t call_step(const VerifyDev& P) {
    return P.step_dev != nullptr ? *P.step_dev : P.step64;
}
// The noise key of the call (the sequence field is set per use).
__device__ __forceinline__ NoiseKey noise_key(const VerifyDev& P) {
    NoiseKey nk = P.nk;
    nk.step = static_cast<uint32_t>(call_step(P));
    return nk;
}
// This call is a re-probe step of the gate (step a multiple of the interval).
__device__ __forceinline__ bool probe_now(const VerifyDev& P) {
    return P.probe > 0 && call_step(P) % static_cast<uint64_t>(P.probe) == 0;
}

// Drafts verified this call for a sequence with kb drafts, acceptance EMA ema
// and cooling count cool: the EMA gate (shut below the threshold, except on a
// re-probe step), then no drafts while cooling.
__device__ __forceinline__ int gate_rule(const VerifyDev& P, int kb, float ema, int cool) {
    int ke = kb;
    if (P.gate && kb > 0 && !(ema >= P.thresh) && !probe_now(P)) ke = 0;
    if (P.cool > 0 && cool > 0) ke = 0;
    return ke;
}

// Cooling count after the call: a cooling sequence counts down; a partial
// acceptance (0 < a < k_eff) starts P.cool calls without drafts.
__device__ __forceinline__ int cool_after(const VerifyDev& P, int cool, int a, int keff) {
    if (cool > 0) return cool - 1;
    return (a > 0 && a < keff) ? P.cool : 0;
}

__device__ __forceinline__ int gate_keff(const VerifyDev& P, int b, int* kb_out, bool flag) {
    int kb = P.k[b];
    if (kb < 0 || kb > P.K) {
        if (flag) raise_status(P.status, SPECNG_DEV_BAD_K);
        kb = kb < 0 ? 0 : P.K;
    }
    if (kb_out) *kb_out = kb;
    return gate_rule(P, kb, P.gate ? P.ema[b] : 1.0f, P.gate_state ? P.gate_state[b] : 0);
}

// Slack of the block bound: covers the fp32 rounding of z / T and ln M.
__device__ __forceinline__ float bound_slack(float z) { return 1e-5f * (1.0f + fabsf(z)); }

// A raw logit x_t such that every element whose block bound passes the best,
// z / T - ln M + bound_slack(.) >= thr with z the (unpenalised) transform of x,
// has x >= x_t.  The margins keep the screen a superset of the exact test in
// spite of fp32 rounding: 2e-5 (1 + |thr|) in score units, then 1e-5 relative
// in z, then (soft cap) 2e-5 c in z before the inverse map and 1e-4 relative
// after it, which covers the error of tanhf amplified by the steep atanh.
// Used only where the penalty cannot raise a value (r >= 1).
template <bool SOFTCAP>
__device__ __forceinline__ float raw_screen(float thr, float lnM, const VerifyDev& P) {
    if (!(thr > -INFINITY)) return -INFINITY;
    float zt = (thr + lnM - 2e-5f * (1.0f + fabsf(thr))) * P.T;
    zt -= 1e-5f * (1.0f + fabsf(zt));
    if constexpr (SOFTCAP) {
        zt -= 2e-5f * P.cap;
        if (zt <= -P.cap) return -INFINITY;
        if (zt >= P.cap) return INFINITY;  // the transform never exceeds c
        const float xr = P.cap * atanhf(zt * P.invcap);
        return xr - 1e-4f * (1.0f + fabsf(xr));
    }
    return zt;
}

// Elements n.. of a 16-byte vector set to -inf (n <= 0: all of them).
template <bool BF16>
__device__ __forceinline__ uint4 mask_tail(uint4 r, int n) {
    uint32_t w[4] = {r.x, r.y, r.z, r.w};
    if constexpr (BF16) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (e >= n) w[e >> 1] = (e & 1) ? ((w[e >> 1] & 0x0000FFFFu) | 0xFF800000u) : ((w[e >> 1] & 0xFFFF0000u) | 0xFF80u);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (e >= n) w[e] = 0xFF800000u;
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------- K1
// Streaming kernel: bandwidth only.  Persistent and warp-specialised, kK1PerSM
// CTAs per SM; the active row-chunks of the call (rows 0..k_eff of every
// sequence, chunks of 64 KB) are laid out row-major and split into equal
// contiguous ranges, one per CTA.
//   * A producer warp walks the CTA's range and keeps up to kStages chunks in
//     flight with cp.async.bulk into a shared-memory ring (full / empty
//     mbarriers, bounded waits), with each chunk's row metadata and penalty
//     bitmap.  The next sequence's drafts and history tail are fetched into
//     registers one sequence ahead, so no global round trip stalls the copies.
//   * Sixteen streaming warps each own a 4 KB slice of every chunk.  A warp's
//     vector row (32 lanes x one 16-byte vector) of a bf16 chunk is one noise
//     block (two rows for fp32): its largest raw logit goes to the workspace
//     (packed maxima reduced across the warp).  The rows that carry an accept
//     test (j < k_eff, T > 0) also add their exponentials to a sum kept against
//     a segment reference (so the sum does not wait for each chunk's maximum);
//     at the last chunk of a row segment the warps combine their sums into one
//     record.
//   * Rejection proofs (point-mass drafts): the producer gives every accept row
//     the threshold thr = z_d - T ln u + T mg (z_d: the draft's transformed
//     logit, read one sequence ahead, taken at its larger penalty value; u: the
//     test's draw; mg: a margin over fp32 error).  The log-normaliser is at
//     least z / T for every value z of the row, so a value z >= thr proves
//     ln p(d) < ln u: the test rejects and the row's sum is not needed.  A warp
//     that meets such a value (its lane maxima, taken at their smaller penalty
//     value) stops adding exponentials for the rest of the segment, and the
//     segment's record says so (s < 0).  Dense drafts keep every sum (the
//     residual needs the rejected row's normaliser).

constexpr int kCWarps = 16;                    // streaming warps
constexpr int kPWarp = kCWarps;                // producer warp index
constexpr int kPThreads = (kCWarps + 1) * 32;  // 544
constexpr int kK1PerSM = 1;                    // resident streaming CTAs per SM
constexpr int kStages = 3;                     // ring stages per CTA
constexpr int kVL = 8;                         // 16-byte vectors per lane per chunk
static_assert(kChunkBytes == kCWarps * 32 * kVL * 16, "stage layout");
static_assert(kVL <= 8, "the penalty mask holds 8 vectors of a lane");
static_assert((32 * 8) == (1 << kNoiseBlockShift), "a bf16 vector row of a warp is one noise block");

template <bool PENALTY>
__host__ __device__ constexpr size_t k1_dyn_smem() {
    return static_cast<size_t>(kStages) * kChunkBytes +
           (PENALTY ? static_cast<size_t>(kStages) * (kChunkBytes / 2 / 8) : 0);
}

struct StageMeta {
    int b, j, c;
    int seg_end;   // the last chunk of this row in the CTA's range
    int sum;       // the row's softmax sum is needed (accept test)
    float thr;     // rejection-proof threshold of the row's accept test (+inf: none)
    unsigned penw; // bit w: warp w's slice holds a penalised id
    int dnext;     // single-kernel schedule: d_{j+1} of the row (-1: none)
    int pend;      // single-kernel schedule: d_{j+1} is in the row's penalty window
};

// Running state of a lane's sum of exponentials: reference m (transformed
// units), the sum s of exp((z - m) / T), and m * log2(e) / T.
struct SumState {
    float m, s, msc;
};

// Element bit = 8 i + e of a lane's vectors rv[i] (register selects; taken
// only for the few penalised elements of a slice).
template <bool BF16>
__device__ __forceinline__ float elem_of_regs(const uint4 (&rv)[kVL], int bit) {
    const int i = bit >> 3, e = bit & 7;
    uint4 r = rv[0];
#pragma unroll
    for (int t = 1; t < kVL; ++t)
        if (i == t) r = rv[t];
    if constexpr (BF16) {
        const int q = e >> 1;
        const uint32_t w = q == 0 ? r.x : q == 1 ? r.y : q == 2 ? r.z : r.w;
        return (e & 1) ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16);
    } else {
        const uint32_t w = e == 0 ? r.x : e == 1 ? r.y : e == 2 ? r.z : r.w;
        return __uint_as_float(w);
    }
}

// Cold path of the streaming warps, kept out of line so the hot loop stays
// small in the instruction cache: a lane's vectors of a row's last chunk when
// they pass the row's end (read back from the stage, which the warp holds
// until it is done).  Two passes with the exact transform, a vector at a
// time (the elements of a vector in parallel): the largest valid value fixes
// the reference (raised as in the hot loop), then the terms of the valid
// elements; elements past the row's end are left out.
template <bool BF16, bool SOFTCAP, bool PENALTY>
__device__ __noinline__ SumState sum_partial(const uint4* stage, int off0, int v0, int v1, unsigned long long pmk,
                                             SumState st, const VerifyDev& P) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    const int nv0 = v1 - (v0 + off0);  // valid elements from my vector 0 on
    float zm = -INFINITY;
#pragma unroll 1
    for (int i = 0; i < kVL && nv0 - i * 32 * EPV > 0; ++i) {
        float x[EPV];
        unpack<BF16>(stage[off0 / EPV + i * 32], x);
        const int nv = nv0 - i * 32 * EPV;
        const unsigned pb = static_cast<unsigned>(pmk >> (8 * i));
#pragma unroll
        for (int e = 0; e < EPV; ++e)
            if (e < nv) zm = fmaxf(zm, transform_f32<SOFTCAP, PENALTY>(x[e], (pb >> e) & 1u, P));
    }
    if (zm > -INFINITY) {
        if (!(st.m > -INFINITY)) {
            st.s = 0.0f;
            st.m = zm;
            st.msc = zm * P.sc;
        } else if ((zm - st.m) * P.sc > 32.0f) {
            st.s *= ex2_approx((st.m - zm) * P.sc);
            st.m = zm;
            st.msc = zm * P.sc;
        }
    }
    if (!(st.m > -INFINITY)) return st;  // no valid finite value yet
#pragma unroll 1
    for (int i = 0; i < kVL && nv0 - i * 32 * EPV > 0; ++i) {
        float x[EPV];
        unpack<BF16>(stage[off0 / EPV + i * 32], x);
        const int nv = nv0 - i * 32 * EPV;
        const unsigned pb = static_cast<unsigned>(pmk >> (8 * i));
        float acc = 0.0f;
#pragma unroll
        for (int e = 0; e < EPV; ++e)
            if (e < nv) acc += ex2_approx(fmaf(transform_f32<SOFTCAP, PENALTY>(x[e], (pb >> e) & 1u, P), P.sc, -st.msc));
        st.s += acc;
    }
    return st;
}

template <bool BF16, bool GREEDY, bool SOFTCAP, bool PENALTY>
__global__ void __launch_bounds__(kPThreads, kK1PerSM) verify_stream_kernel(const __grid_constant__ VerifyDev P) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    constexpr int CHUNK = chunk_elems<BF16>();
    constexpr int SB = kChunkBytes;
    constexpr int SL = 32 * kVL * EPV;                          // ids per streaming slice
    constexpr int VPB = (1 << kNoiseBlockShift) / (32 * EPV);   // vector rows per noise block (bf16 1, fp32 2)
    extern __shared__ __align__(128) uint8_t s_dyn[];
    uint8_t* s_stage = s_dyn;
    uint32_t* s_bm = reinterpret_cast<uint32_t*>(s_dyn + kStages * SB);
    __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages];
    __shared__ StageMeta s_meta[kStages];
    // segment merge slots, two per stage (by ring-cycle parity): a warp releases
    // a stage as soon as its vectors are in registers, so the next cycle of the
    // same stage can reach its merge before this one's last warp has read it
    __shared__ SegSum s_slot[kStages][2][kCWarps];
    __shared__ int s_cnt[kStages][2];
    __shared__ long long s_wsum[kPThreads / 32];
    __shared__ int s_start[3];
    __shared__ int s_proved_row;  // the latest row a warp of this CTA proved to reject
    __shared__ int s_hwin[PENALTY ? SPECNG_MAX_REP_WINDOW : 1];
    __shared__ int s_pdrafts[SPECNG_MAX_K + 1];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K1 = P.K + 1;
    // k and ema come from the kernels before this one; once they are visible the
    // decision kernel may be launched (its own wait holds it until this one ends)
    pdl_wait();
    pdl_trigger();

    // ---- prologue: count the active row-chunks and find this CTA's range
    const int per = (P.B + kPThreads - 1) / kPThreads;
    const int bb0 = tid * per;
    long long mine = 0;
    for (int b = bb0; b < bb0 + per && b < P.B; ++b) mine += static_cast<long long>(gate_keff(P, b, nullptr, false) + 1) * P.nchunk;
    long long incl = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) s_wsum[warp] = incl;
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], kCWarps);
            s_cnt[i][0] = 0;
            s_cnt[i][1] = 0;
        }
        s_proved_row = -1;
        mbar_init_fence();
    }
    __syncthreads();
    long long base = 0, total = 0;
    for (int w = 0; w < kPThreads / 32; ++w) {
        if (w < warp) base += s_wsum[w];
        total += s_wsum[w];
    }
    const long long G = gridDim.x;
    const long long w0 = total * blockIdx.x / G, w1 = total * (blockIdx.x + 1) / G;
    const long long ex = base + incl - mine;  // first row-chunk index of my sequences
    if (w0 < w1 && w0 >= ex && w0 < ex + mine) {
        long long acc = ex;
        for (int b = bb0; b < bb0 + per && b < P.B; ++b) {
            const long long nb = static_cast<long long>(gate_keff(P, b, nullptr, false) + 1) * P.nchunk;
            if (w0 < acc + nb) {
                const long long r = w0 - acc;
                s_start[0] = b;
                s_start[1] = static_cast<int>(r / P.nchunk);
                s_start[2] = static_cast<int>(r % P.nchunk);
                break;
            }
            acc += nb;
        }
    }
    __syncthreads();
    const int nwork = static_cast<int>(w1 - w0);
    if (nwork <= 0) return;

    if (warp == kPWarp) {
        // ================= producer =================
        constexpr int kHW = PENALTY ? SPECNG_MAX_REP_WINDOW / 32 : 1;
        struct SeqData {
            int k, draft, L, cool;
            float ema, xd;  // xd: raw logit of the lane's draft in its row (loaded a step after draft)
            int hw[kHW];
        };
        auto clampL = [&](int L) {
            return L < 0 ? 0 : (static_cast<int64_t>(L) > P.hist_stride ? static_cast<int>(P.hist_stride) : L);
        };
        auto fetch = [&](int bq, int L, SeqData& d) {  // issues the loads; nothing waits here
            d.k = bq < P.B ? P.k[bq] : 0;
            d.ema = (P.gate && bq < P.B) ? P.ema[bq] : 1.0f;
            d.cool = (P.gate_state != nullptr && bq < P.B) ? P.gate_state[bq] : 0;
            d.draft = (bq < P.B && lane < P.K) ? draft_at(P, bq, lane) : -1;
            d.L = L;
            if constexpr (PENALTY) {
                const int nh = L < P.W ? L : P.W;
#pragma unroll
                for (int i = 0; i < kHW; ++i) {
                    const int t = lane + 32 * i;
                    d.hw[i] = (bq < P.B && t < nh) ? hist_at(P, bq, (L - nh) + t) : 0;
                }
            }
        };
        // proofs need a point-mass draft and T > 0
        const bool proofs = !GREEDY && P.q == nullptr;
        auto fetch_xd = [&](int bq, SeqData& d) {  // after d.draft has landed
            d.xd = (proofs && bq < P.B && lane < P.K && d.draft >= 0 && d.draft < P.V)
                       ? static_cast<float>(raw_logit_chk<BF16>(P, static_cast<size_t>(bq) * K1 + lane, d.draft))
                       : 0.0f;
        };
        int b = s_start[0], j = s_start[1], c = s_start[2];
        int keff = 0, nh = 0;
        float thr = INFINITY;  // lane j: row j's rejection-proof threshold
        auto install = [&](const SeqData& d, int bq) {
            int kb = d.k;
            if (kb < 0 || kb > P.K) kb = kb < 0 ? 0 : P.K;
            keff = gate_rule(P, kb, d.ema, d.cool);
            thr = INFINITY;
            if (proofs && lane < keff) {
                if (d.draft >= 0 && d.draft < P.V) {
                    float zd = transform_f32<SOFTCAP, false>(d.xd, false, P);
                    if constexpr (PENALTY) zd = fmaxf(zd, zd > 0.0f ? zd * P.invrep : zd * P.rep);
                    NoiseKey nk = noise_key(P);
                    nk.seq = static_cast<uint32_t>(bq);
                    const float lu = logf(static_cast<float>(accept_uniform_f64(nk, static_cast<uint32_t>(lane + 1))));
                    const float lp = zd * P.invT - lu;
                    thr = zd - P.T * lu + P.T * (1e-3f + 1e-4f * fabsf(lp));
                } else {
                    thr = -INFINITY;  // an id outside [0, V) is rejected without a test
                }
            }
            if (lane < keff) s_pdrafts[lane] = d.draft;
            if constexpr (PENALTY) {
                nh = d.L < P.W ? d.L : P.W;
#pragma unroll
                for (int i = 0; i < kHW; ++i)
                    if (lane + 32 * i < nh) s_hwin[lane + 32 * i] = d.hw[i];
            }
            __syncwarp();
        };
        SeqData cur, nxt;
        int Lnext2 = 0;
        {
            const int L0 = PENALTY ? clampL(P.lens[b]) : 0;
            const int L1 = (PENALTY && b + 1 < P.B) ? clampL(P.lens[b + 1]) : 0;
            fetch(b, L0, cur);
            fetch_xd(b, cur);
            install(cur, b);
            fetch(b + 1, L1, nxt);
            if (PENALTY && b + 2 < P.B) Lnext2 = P.lens[b + 2];
        }
        bool xd_due = true;  // nxt's draft logits are loaded one chunk after its drafts
        bool ok = true;
        int st = 0;
        int issued = 0;     // items whose copy was issued (copies complete in issue order per stage)
        unsigned eph = 0u;  // parity of the empty barrier phase to wait for
        for (int n = 0; n < nwork && ok; ++n) {
            const int v0 = c * CHUNK;
            const int v1 = min(P.V, v0 + CHUNK);
            const char* src = static_cast<const char*>(P.logits) +
                              ((static_cast<size_t>(b) * K1 + j) * P.V + v0) * ElemTraits<BF16>::SIZE;
            if (n >= kStages) ok = mbar_wait_bounded(&s_empty[st], eph);
            if (!ok) { if (lane == 0) raise_status(P.status, SPECNG_DEV_TIMEOUT); break; }
            // the copy goes first; the metadata is written while it is in flight, and the
            // phase completes once both the bytes and the arrive below are in
            if (P.aligned && lane == 0) {
                // the empty barrier already orders the consumers' reads of this stage
                // before the copy that overwrites it
                mbar_add_tx(&s_full[st], static_cast<unsigned>(v1 - v0) * ElemTraits<BF16>::SIZE);
                bulk_g2s(s_stage + st * SB, src, static_cast<unsigned>(v1 - v0) * ElemTraits<BF16>::SIZE, &s_full[st]);
            }
            issued = n + 1;
            if (xd_due) {
                fetch_xd(b + 1, nxt);
                xd_due = false;
            }
            StageMeta& mt = s_meta[st];
            const float rthr = __shfl_sync(0xffffffffu, thr, j & 31);
            if (lane == 0) {
                mt.b = b; mt.j = j; mt.c = c;
                mt.seg_end = (c == P.nchunk - 1 || n == nwork - 1) ? 1 : 0;
                mt.sum = (!GREEDY && j < keff) ? 1 : 0;
                mt.thr = j < keff ? rthr : INFINITY;
            }
            if constexpr (PENALTY) {
                // bitmap of the penalised ids of row j in [v0, v1), and which slices hold one
                uint32_t* bm = s_bm + st * (CHUNK / 32);
                for (int t = lane; t < CHUNK / 32; t += 32) bm[t] = 0u;
                __syncwarp();
                const WindowView wv{s_hwin, s_pdrafts, nh, P.W};
                const int nwin = wv.count(j);
                unsigned pw = 0u;
                for (int t = lane; t < nwin; t += 32) {
                    const int tok = wv.token(j, t);
                    if (tok >= v0 && tok < v1) {
                        atomicOr(&bm[(tok - v0) >> 5], 1u << ((tok - v0) & 31));
                        pw |= 1u << ((tok - v0) / SL);
                    }
                }
                pw = __reduce_or_sync(0xffffffffu, pw);
                if (lane == 0) mt.penw = pw;
            } else {
                if (lane == 0) mt.penw = 0u;
            }
            if (!P.aligned) {
                uint8_t* dst = s_stage + st * SB;
                for (int e = lane; e < v1 - v0; e += 32) {
                    if constexpr (BF16) reinterpret_cast<uint16_t*>(dst)[e] = reinterpret_cast<const uint16_t*>(src)[e];
                    else reinterpret_cast<uint32_t*>(dst)[e] = reinterpret_cast<const uint32_t*>(src)[e];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_full[st]);
            if (++st == kStages) {
                st = 0;
                if (n >= kStages) eph ^= 1u;  // the waits of ring cycle u (>= 1) are for phase u - 1
            }
            // advance to the next row-chunk
            if (++c == P.nchunk) {
                c = 0;
                if (++j > keff) {
                    j = 0;
                    ++b;
                    if (n + 1 < nwork) {
                        if (xd_due) fetch_xd(b, nxt);  // a sequence shorter than one chunk
                        install(nxt, b);
                        const int L2 = PENALTY ? clampL(Lnext2) : 0;
                        fetch(b + 1, L2, nxt);
                        xd_due = true;
                        if (PENALTY && b + 2 < P.B) Lnext2 = P.lens[b + 2];
                    }
                }
            }
        }
        // the CTA stays resident until every issued copy has landed: item n of a stage
        // completes that stage's phase n / kStages, so the last kStages issued items
        // (one per stage, each its stage's latest phase) are the ones to wait for; a
        // wait that runs out raises TIMEOUT
        if (P.aligned && lane == 0) {
            const int lo = issued > kStages ? issued - kStages : 0;
            for (int n = lo; n < issued; ++n)
                if (!mbar_wait_bounded(&s_full[n % kStages], static_cast<unsigned>((n / kStages) & 1)))
                    raise_status(P.status, SPECNG_DEV_TIMEOUT);
        }
        return;
    }

    // ================= streaming warps =================
    // The sum of exponentials of a segment is kept against a reference m, fixed
    // at the segment's first value and raised only when a value passes it by
    // more than 2^32 in the sum's units.
    const int ubase = warp * (32 * kVL);        // first 16-byte vector of my slice
    const int off0 = ubase * EPV + lane * EPV;  // chunk offset of vector 0's element 0
    float m = -INFINITY, s = 0.0f, msc = 0.0f;
    bool proved = false;  // this warp met a value proving the segment's row rejects
    int st = 0;
    unsigned fph = 0u;  // parity of the full barrier phase to wait for
    for (int n = 0; n < nwork; ++n) {
        if (!mbar_wait_bounded(&s_full[st], fph)) {
            if (lane == 0) raise_status(P.status, SPECNG_DEV_TIMEOUT);
            break;
        }
        const StageMeta mt = s_meta[st];
        const int c = mt.c;
        const int row = mt.b * K1 + mt.j;
        const bool dosum = !GREEDY && mt.sum != 0;
        const int v0 = c * CHUNK;
        const int v1 = min(P.V, v0 + CHUNK);
        const uint4* stage = reinterpret_cast<const uint4*>(s_stage + st * SB);
        const uint32_t* bm = s_bm + (PENALTY ? st * (CHUNK / 32) : 0);
        const bool full = v0 + off0 + (kVL - 1) * 32 * EPV + EPV <= v1;  // my vectors are whole
        uint4 rv[kVL];
#pragma unroll
        for (int i = 0; i < kVL; ++i) rv[i] = stage[ubase + i * 32 + lane];
        // penalised elements of my lane (bit 8 i + e of a 64-bit mask), only where the slice holds one
        unsigned long long pmk = 0ull;
        if constexpr (PENALTY) {
            if ((mt.penw >> warp) & 1u) {
#pragma unroll
                for (int i = 0; i < kVL; ++i) {
                    const int off = off0 + i * 32 * EPV;
                    pmk |= static_cast<unsigned long long>((bm[off >> 5] >> (off & 31)) & ((1u << EPV) - 1u)) << (8 * i);
                }
            }
        }
        // Everything below works on registers, except the element-by-element sum
        // of a slice that passes the row's end: release the stage now unless
        // that path will read it, so the producer can refill it while this
        // chunk's arithmetic runs.
        const bool hold = dosum && (v0 + ubase * EPV + 32 * kVL * EPV > v1);
        __syncwarp();
        if (!hold && lane == 0) mbar_arrive(&s_empty[st]);
        // packed maxima of my vectors (bf16: both halves of a word hold partial maxima;
        // fp32: the maximum), NaN propagated; elements past the row's end count as -inf
        uint32_t hv[kVL];
#pragma unroll
        for (int i = 0; i < kVL; ++i) {
            uint4 r = rv[i];
            if (!full) {
                const int nv = v1 - (v0 + off0 + i * 32 * EPV);
                r = mask_tail<BF16>(r, nv);
            }
            if constexpr (BF16) {
                hv[i] = as_u32(bf16x8_max2_nan(r));
            } else {
                hv[i] = __float_as_uint(fmax_nan(fmax_nan(__uint_as_float(r.x), __uint_as_float(r.y)),
                                                 fmax_nan(__uint_as_float(r.z), __uint_as_float(r.w))));
            }
        }
        if (dosum) {
            // the lane's largest raw logit of the chunk (NaN if it holds one)
            float lraw;
            if constexpr (BF16) {
                uint32_t h = hv[0];
#pragma unroll
                for (int i = 1; i < kVL; ++i) h = as_u32(__hmax2_nan(as_bf162(h), as_bf162(hv[i])));
                lraw = fmax_nan(bf16lo(h), bf16hi(h));
            } else {
                lraw = __uint_as_float(hv[0]);
#pragma unroll
                for (int i = 1; i < kVL; ++i) lraw = fmax_nan(lraw, __uint_as_float(hv[i]));
            }
            const bool bad = !(lraw < INFINITY);  // NaN or +inf
            if (__any_sync(0xffffffffu, bad) && lane == 0) raise_status(P.status, SPECNG_DEV_NONFINITE);
            const float zl = SOFTCAP ? transform_f32<true, false>(lraw, false, P) : lraw;
            if (!proved) {
                // a proof found by any warp of the CTA holds for the whole row
                float zlo = zl;
                if constexpr (PENALTY) zlo = fminf(zl, zl > 0.0f ? zl * P.invrep : zl * P.rep);
                const bool mine = __any_sync(0xffffffffu, !bad && zlo >= mt.thr);
                if (mine && lane == 0) *reinterpret_cast<volatile int*>(&s_proved_row) = row;
                proved = __any_sync(0xffffffffu, mine || *reinterpret_cast<volatile int*>(&s_proved_row) == row);
            }
            if (proved) {
                // the test rejects: no sum for the rest of the segment
            } else if (full) {
                if (!(m > -INFINITY)) {
                    m = zl;
                    msc = m * P.sc;
                } else if ((zl - m) * P.sc > 32.0f) {
                    // far above the reference: raise it before this chunk's terms
                    s *= ex2_approx((m - zl) * P.sc);
                    m = zl;
                    msc = m * P.sc;
                }
                if (m > -INFINITY) {
                    float2 acc2[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                                      make_float2(0.0f, 0.0f)};
                    const float2 sc2 = make_float2(P.sc, P.sc), nm2 = make_float2(-msc, -msc);
#pragma unroll
                    for (int i = 0; i < kVL; ++i) {
                        float x[EPV];
                        unpack<BF16>(rv[i], x);
#pragma unroll
                        for (int e = 0; e < EPV; e += 2) {
                            const float2 t = __ffma2_rn(make_float2(sum_transform<SOFTCAP>(x[e], P),
                                                                    sum_transform<SOFTCAP>(x[e + 1], P)),
                                                        sc2, nm2);
                            acc2[i & 3] = __fadd2_rn(acc2[i & 3], make_float2(ex2_approx(t.x), ex2_approx(t.y)));
                        }
                    }
                    s += ((acc2[0].x + acc2[0].y) + (acc2[1].x + acc2[1].y)) +
                         ((acc2[2].x + acc2[2].y) + (acc2[3].x + acc2[3].y));
                }
                if constexpr (PENALTY) {
                    // the few penalised elements: their terms are replaced by the penalised ones
                    unsigned long long pw = pmk;
                    while (pw != 0ull) {
                        const int bit = __ffsll(static_cast<long long>(pw)) - 1;
                        pw &= pw - 1ull;
                        const float xe = elem_of_regs<BF16>(rv, bit);
                        const float zu = sum_transform<SOFTCAP>(xe, P);
                        const float zp = sum_transform_pen<SOFTCAP>(xe, P);
                        if ((zp - m) * P.sc > 32.0f) {
                            s = m > -INFINITY ? s * ex2_approx((m - zp) * P.sc) : 0.0f;
                            m = zp;
                            msc = m * P.sc;
                        }
                        s += ex2_approx(fmaf(zp, P.sc, -msc)) - ex2_approx(fmaf(zu, P.sc, -msc));
                    }
                }
            } else {
                // partial vectors (a row's last chunk): exact transform element by element
                const SumState st = sum_partial<BF16, SOFTCAP, PENALTY>(stage, off0, v0, v1, pmk, SumState{m, s, msc}, P);
                m = st.m;
                s = st.s;
                msc = st.msc;
            }
        }
        // ---- block maxima (raw logits): vector row i of the warp (rows i, i + 1 for
        //      fp32) is one noise block; the warp's four (two) blocks are contiguous
        {
            const int blk0 = (v0 >> kNoiseBlockShift) + warp * (kVL / VPB);
            float* dst = P.bmax + static_cast<size_t>(row) * P.nblk + blk0;
            const int nb = min(kVL / VPB, P.nblk - blk0);
            if constexpr (BF16) {
                // the maximum of each vector in one half, two vectors per word
                uint32_t bw[kVL / 2];
#pragma unroll
                for (int p = 0; p < kVL / 2; ++p)
                    bw[p] = as_u32(__hmax2(as_bf162(__byte_perm(hv[2 * p], hv[2 * p + 1], 0x5410)),
                                           as_bf162(__byte_perm(hv[2 * p], hv[2 * p + 1], 0x7632))));
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                    for (int p = 0; p < kVL / 2; ++p)
                        bw[p] = as_u32(__hmax2(as_bf162(bw[p]), as_bf162(__shfl_xor_sync(0xffffffffu, bw[p], off))));
                // lane i < nb stores block i (every lane holds the warp-reduced maxima)
                float raw = -INFINITY;
#pragma unroll
                for (int i = 0; i < kVL; ++i)
                    if (lane == i) raw = (i & 1) ? bf16hi(bw[i >> 1]) : bf16lo(bw[i >> 1]);
                if (lane < nb) dst[lane] = raw;
            } else {
                float bm[kVL / VPB];
#pragma unroll
                for (int p = 0; p < kVL / VPB; ++p) {
                    bm[p] = __uint_as_float(hv[VPB * p]);
#pragma unroll
                    for (int u = 1; u < VPB; ++u) bm[p] = fmaxf(bm[p], __uint_as_float(hv[VPB * p + u]));
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                    for (int p = 0; p < kVL / VPB; ++p) bm[p] = fmaxf(bm[p], __shfl_xor_sync(0xffffffffu, bm[p], off));
                float raw = -INFINITY;
#pragma unroll
                for (int p = 0; p < kVL / VPB; ++p)
                    if (lane == p) raw = bm[p];
                if (lane < nb) dst[lane] = raw;
            }
        }

        if (mt.seg_end && dosum) {
            // ---- end of this row's segment: one record for the segment (s < 0: proved)
            float pm = 0.0f, ps = -1.0f;  // proved: nothing to merge
            if (!proved) {
                pm = m;
                ps = pm > -INFINITY ? s : 0.0f;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float mo = __shfl_xor_sync(0xffffffffu, pm, off);
                    const float so = __shfl_xor_sync(0xffffffffu, ps, off);
                    ms_merge(pm, ps, mo, so, P.sc);
                }
            }
            int last = 0;
            if (lane == 0) {
                s_slot[st][fph][warp] = SegSum{pm, ps};
                __threadfence_block();
                last = atomicAdd(&s_cnt[st][fph], 1) == kCWarps - 1;
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence_block();
                const SegSum wp = lane < kCWarps ? s_slot[st][fph][lane] : SegSum{-INFINITY, 0.0f};
                const bool anyp = __any_sync(0xffffffffu, wp.s < 0.0f);
                float cm = 0.0f, cs = -1.0f;  // a proof from any warp stands for the segment
                if (!anyp) {
                    cm = wp.m;
                    cs = wp.s;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        const float mo = __shfl_xor_sync(0xffffffffu, cm, off);
                        const float so = __shfl_xor_sync(0xffffffffu, cs, off);
                        ms_merge(cm, cs, mo, so, P.sc);
                    }
                }
                if (lane == 0) {
                    // keyed by the segment's last chunk; a written record is never all-zero
                    P.part[static_cast<size_t>(row) * P.nchunk + c] = SegSum{cm, cs};
                    s_cnt[st][fph] = 0;
                }
            }
        }
        if (mt.seg_end) {
            m = -INFINITY;
            s = 0.0f;
            msc = 0.0f;
            proved = false;
        }
        __syncwarp();
        if (hold && lane == 0) mbar_arrive(&s_empty[st]);
        if (++st == kStages) {
            st = 0;
            fph ^= 1u;
        }
    }
}

// ---------------------------------------------------------------- K2
// Decision kernel: one CTA of kSW warps per sequence, launched chained to the
// streaming kernel (its prologue -- drafts, gate, the penalty window's table --
// runs before the streaming kernel has finished).
//   1. The accept tests (T > 0): warp w takes rows w, w + kSW, ... < k_eff;
//      the log-sum-exp of a row comes from its segment sums, and the test of
//      d_{j+1} is taken in fp32 unless it is within 1e-4 of the boundary,
//      then in fp64.  At T = 0 every row 0..k_eff gets its argmax instead:
//      the blocks whose largest value is within the tie margin of the best
//      value found are read again.
//   2. a = the first rejection (k_eff when none).
//   3. The token at row a (T > 0): Gumbel-max over the row, draft d_{a+1}
//      left out for a point-mass draft.  Each warp's block with the largest
//      value is loaded first (the seed); meanwhile each block's draw gives M
//      and its slot, and the bound z_max / T - ln M of every block goes to
//      shared memory.  Each lane scores its largest element of the seed block,
//      which starts the best; then only the blocks whose bound reaches the
//      best are read again (kBatch per warp at once, screened against one
//      raw-logit threshold per block), and each lane scores its own elements
//      whose bound z / T - ln M reaches it (per-id draw, E_v = M + F_v).  The
//      two best fp32 scores are re-scored in fp64 when they are within the
//      fp32 error of each other.  With dense q a rejection's token is left to
//      the residual pass.
//   4. Epilogue: tokens, accept length, kv_len, EMA.

constexpr int kSW = 16;                         // warps per sequence
constexpr int kST = kSW * 32;
// blocks a warp reads again at once (bf16 8, fp32 4: 8 KB per warp either way)
template <bool BF16> __host__ __device__ constexpr int k2_batch() { return BF16 ? 8 : 4; }
constexpr int kPenSlots = 2 * SPECNG_MAX_REP_WINDOW;
constexpr int kPenBits = 9;
static_assert((1 << kPenBits) == kPenSlots, "penalty table size");
static_assert(SPECNG_MAX_K + 1 <= kST, "one thread per output token");

// Dynamic shared memory of the decision kernel at T > 0: the block scratch
// (when it fits) and each warp's staging of a batch of blocks.
__host__ __device__ constexpr size_t k2_stage_bytes(bool bf16) {
    return static_cast<size_t>(kSW) * (bf16 ? k2_batch<true>() : k2_batch<false>()) * 32 * (bf16 ? 1 : 2) * 16;
}
__host__ __device__ inline size_t k2_blk_bytes(int nblk) {
    return nblk <= kSmemBlkCap ? (static_cast<size_t>(nblk) * kBlkScratchBytes + 15) / 16 * 16 : 0;
}
__host__ __device__ inline size_t k2_dyn_smem(int nblk, bool bf16) {
    return k2_blk_bytes(nblk) + k2_stage_bytes(bf16);
}

// Open-addressed table of the history tail of the penalty window: the token
// and its latest position in the tail (-1 = empty slot).
__device__ __forceinline__ uint32_t pen_hash(int v) { return (static_cast<uint32_t>(v) * 2654435761u) >> (32 - kPenBits); }

// Bound of the transformed logits of a block from its largest raw logit: the
// soft cap is increasing, and a penalty r >= 1 only lowers a value (r < 1 may
// raise it: then the larger of the two).
template <bool SOFTCAP, bool PENALTY>
__device__ __forceinline__ float block_zmax(float xmax, const VerifyDev& P) {
    float z = transform_f32<SOFTCAP, false>(xmax, false, P);
    if (PENALTY && P.rep < 1.0f) z = fmaxf(z, transform_f32<SOFTCAP, true>(xmax, true, P));
    return z;
}

// Is id v in the penalty window of row j (the last W tokens of the history
// tail ++ d_1..d_j)?  key / pos: the table above; d: the drafts; nh: the
// tail's length.  Out of line: it is called from several places.
static __device__ __noinline__ bool pen_lookup(const int* key, const int* pos, const int* d, int nh, int W, int v, int j) {
    const int total = nh + j;
    const int start = total - (total < W ? total : W);
    uint32_t h = pen_hash(v);
    for (int probe = 0; probe < kPenSlots; ++probe) {
        const int k = key[h];
        if (k == v) {
            if (pos[h] >= start) return true;
            break;
        }
        if (k == -1) break;
        h = (h + 1u) & (kPenSlots - 1u);
    }
    for (int i = start > nh ? start - nh : 0; i < j; ++i)
        if (d[i] == v) return true;
    return false;
}

// The two best fp32 sampling scores of row `row` (position a) re-scored in
// fp64, the oracle's arithmetic: returns the winner (lower id on a tie).  Out
// of line: it runs only for near ties, and keeps the fp64 code out of the
// kernel's hot path.
template <bool BF16, bool SOFTCAP, bool PENALTY>
__device__ __noinline__ int rescore_top2_f64(const VerifyDev& P, const NoiseKey& nk, int row, int a, int i1, int i2,
                                             bool pen1, bool pen2) {
    double sc[2];
    for (int h = 0; h < 2; ++h) {
        const int id = h == 0 ? i1 : i2;
        const double z = transform_f64<SOFTCAP, PENALTY>(raw_logit_chk<BF16>(P, row, id), h == 0 ? pen1 : pen2, P);
        sc[h] = z / P.Td - log(noise_exp_f64(nk, static_cast<uint32_t>(id), static_cast<uint32_t>(a)));
    }
    return better64(sc[1], i2, sc[0], i1) ? i2 : i1;
}

// The accept test u q(d) <= p(d) in fp64, the oracle's arithmetic, for a test
// within the fp32 screen's margin of its boundary; x: the draft's raw logit,
// (mf, Sf): the row's normaliser.  Out of line: it is rarely taken.
template <bool SOFTCAP, bool PENALTY>
__device__ __noinline__ int accept_f64(const VerifyDev& P, float x, bool pen, double u, double q, float mf, float Sf) {
    const double lse = static_cast<double>(mf) / P.Td + log(static_cast<double>(Sf));
    const double zd = transform_f64<SOFTCAP, PENALTY>(static_cast<double>(x), pen, P);
    return u * q <= exp(zd / P.Td - lse) ? 1 : 0;
}

// Preparation of the sampling at row ra of sequence b (T > 0): every noise
// block's draw and bound z_max / T - ln M into s_bnd / s_M / s_I, and each
// participating warp's seed score (its largest element in its block with the
// largest value, with the element's own draw) into *thr_slot.  Threads t of
// nt take part, whole warps; ex is the id left out (-1: none).  Out of line:
// the decision kernel calls it from two places and its code would otherwise
// be there twice.
// Block draws of row ra (M, slot, and -ln M in s_bnd), threads t of nt: they
// depend on the row's key only, so the decision kernel takes row 0's before
// the stream kernel has finished.
static __device__ __noinline__ void draw_row_blocks(const VerifyDev& P, const NoiseKey& nk, int ra, int t, int nt, float* s_bnd,
                                             float* s_M, int* s_I) {
    for (int q = t; q < P.nblk; q += nt) {
        const BlockNoise bn = block_noise(nk, static_cast<uint32_t>(q), static_cast<uint32_t>(ra));
        s_bnd[q] = -bn.lnM;
        s_M[q] = bn.M;
        s_I[q] = bn.I;
    }
}

template <bool BF16, bool SOFTCAP, bool PENALTY>
__device__ __noinline__ void prepare_row(const VerifyDev& P, const NoiseKey& nk, int b, int ra, int ex, int t, int nt,
                                         unsigned* thr_slot, float* s_bnd, float* s_M, int* s_I, const int* pen_key,
                                         const int* pen_pos, const int* drafts, int nh, bool drawn) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    constexpr int BLK = 1 << kNoiseBlockShift;
    constexpr int VPL = BLK / (32 * EPV);
    const int lane = threadIdx.x & 31;
    const int K1 = P.K + 1;
    const int nblk = P.nblk;
    const float* bmx = P.bmax + static_cast<size_t>(b * K1 + ra) * nblk;
    const char* rowp = static_cast<const char*>(P.logits) + static_cast<size_t>(b * K1 + ra) * P.V * ElemTraits<BF16>::SIZE;
    const RowPhilox rpr = row_philox(nk, static_cast<uint32_t>(ra));
    // each warp's seed: its block with the largest value (the blocks' maxima are
    // loaded first); the seed block's load is issued before the block draws, so
    // its latency overlaps them
    float lb = -INFINITY;
    int lq = -1;
    for (int q = t; q < nblk; q += nt) {
        const float zq = bmx[q];
        if (zq > lb) { lb = zq; lq = q; }
    }
    const unsigned kq = warp_best_key(lb);
    const unsigned own = __ballot_sync(0xffffffffu, kq != 0u && lb > -INFINITY && score_key(lb) == kq);
    const int qs = own ? __shfl_sync(0xffffffffu, lq, __ffs(own) - 1) : -1;
    uint4 rs[VPL];
    if (qs >= 0) {
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
            const int e0 = qs * BLK + (u * 32 + lane) * EPV;
            rs[u] = e0 < P.V ? load_vec_chk<BF16>(P, rowp, e0, P.V) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    // block draws (unless drawn already) and bounds
    for (int q0 = t; q0 < nblk; q0 += 4 * nt) {
        float zq[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) zq[i] = q0 + i * nt < nblk ? bmx[q0 + i * nt] : -INFINITY;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int q = q0 + i * nt;
            if (q >= nblk) break;
            if (drawn) {
                s_bnd[q] += block_zmax<SOFTCAP, PENALTY>(zq[i], P) * P.invT;
            } else {
                const BlockNoise bn = block_noise(nk, static_cast<uint32_t>(q), static_cast<uint32_t>(ra));
                s_bnd[q] = block_zmax<SOFTCAP, PENALTY>(zq[i], P) * P.invT - bn.lnM;
                s_M[q] = bn.M;
                s_I[q] = bn.I;
            }
        }
    }
    // seed: each lane scores its largest element of the warp's seed block (the
    // seed block's draw is the same function of (row, block) as above)
    {
        float sc = -INFINITY;
        if (qs >= 0) {
            float xb = -INFINITY;
            int vb = -1;
#pragma unroll
            for (int u = 0; u < VPL; ++u) {
                float x[EPV];
                unpack<BF16>(rs[u], x);
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    const int v = qs * BLK + (u * 32 + lane) * EPV + e;
                    if (v < P.V && v != ex && (vb < 0 || x[e] > xb)) { xb = x[e]; vb = v; }
                }
            }
            if (vb >= 0) {
                // drawn: the block's draw is in shared memory already (taken before this
                // kernel waited); otherwise it is taken again here (another warp wrote it)
                float Mq;
                int Iq;
                if (drawn) {
                    Mq = s_M[qs];
                    Iq = s_I[qs];
                } else {
                    const BlockNoise bn = block_noise(nk, static_cast<uint32_t>(qs), static_cast<uint32_t>(ra));
                    Mq = bn.M;
                    Iq = bn.I;
                }
                const bool pen = PENALTY && pen_lookup(pen_key, pen_pos, drafts, nh, P.W, vb, ra);
                const float zb = transform_f32<SOFTCAP, PENALTY>(xb, pen, P) * P.invT;
                sc = zb - ln_fast(noise_exp_f32(rpr, Mq, Iq, static_cast<uint32_t>(vb)));
            }
        }
        const unsigned kw = warp_best_key(sc);
        if (kw != 0u && lane == 0) atomicMax(thr_slot, kw);
    }
}

template <bool BF16, bool GREEDY, bool SOFTCAP, bool PENALTY>
__global__ void __launch_bounds__(kST, 2) verify_seq_kernel(const __grid_constant__ VerifyDev P) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    constexpr int BLK = 1 << kNoiseBlockShift;
    constexpr int VPL = BLK / (32 * EPV);  // 16-byte vectors per lane per block (bf16 1, fp32 2)
    constexpr int NE = VPL * EPV;          // elements per lane per block
    constexpr int kBatch = k2_batch<BF16>();
    static_assert(kBatch * NE <= 64, "one 64-bit candidate mask per batch");
    extern __shared__ __align__(128) uint8_t s_dyn[];
    __shared__ int s_pkey[PENALTY ? kPenSlots : 1];
    __shared__ int s_ppos[PENALTY ? kPenSlots : 1];
    __shared__ int s_d[SPECNG_MAX_K + 1];
    __shared__ float2 s_ms[SPECNG_MAX_K + 1];
    __shared__ int s_acc[SPECNG_MAX_K + 1];
    __shared__ int s_arg[SPECNG_MAX_K + 1];
    __shared__ Top2 s_top[kSW];
    __shared__ unsigned s_thr, s_thr0;
    __shared__ int s_nl;
    __shared__ int s_y;
    __shared__ int s_bq[kSW][8];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x;
    const int K1 = P.K + 1;
    pdl_trigger();  // the next kernel may launch; it waits for this one's end itself
    int kb;
    const int keff = gate_keff(P, b, &kb, tid == 0);
    const bool dense = P.q != nullptr;
    NoiseKey nk = noise_key(P);
    nk.seq = static_cast<uint32_t>(b);
    int nh = 0;
    if (tid < keff) {
        const int d = draft_at(P, b, tid);
        s_d[tid] = d;
        if (!(d >= 0 && d < P.V)) raise_status(P.status, SPECNG_DEV_TOKEN_OOR);
    }
    if (tid == 0) {
        s_thr = 0u;
        s_thr0 = 0u;
        s_nl = 0;
    }
    if constexpr (PENALTY) {
        int L = P.lens[b];
        L = L < 0 ? 0 : (static_cast<int64_t>(L) > P.hist_stride ? static_cast<int>(P.hist_stride) : L);
        nh = L < P.W ? L : P.W;
        for (int t = tid; t < kPenSlots; t += kST) {
            s_pkey[t] = -1;
            s_ppos[t] = -1;
        }
        __syncthreads();
        const int* tail = P.hist + static_cast<size_t>(b) * P.hist_stride + (L - nh);
        for (int t = tid; t < nh; t += kST) {
            const int v = tail[t];
            if (v < 0) continue;  // matches no id
            uint32_t h = pen_hash(v);
            for (int probe = 0; probe < kPenSlots; ++probe) {
                const int old = atomicCAS(&s_pkey[h], -1, v);
                if (old == -1 || old == v) {
                    atomicMax(&s_ppos[h], t);
                    break;
                }
                h = (h + 1u) & (kPenSlots - 1u);
            }
        }
    }
    // the sampling scratch of row a (block draws and bounds, the list of blocks)
    const int nblk = P.nblk;
    uint8_t* scr = nblk <= kSmemBlkCap ? s_dyn : P.blkws + static_cast<size_t>(b) * nblk * kBlkScratchBytes;
    float* s_bnd = reinterpret_cast<float*>(scr);
    float* s_M = s_bnd + nblk;
    int* s_I = reinterpret_cast<int*>(s_M + nblk);
    int* s_list = s_I + nblk;
    // Row 0 is sampled by this kernel whenever a = 0 and no residual pass takes it
    // (point-mass drafts, or no draft at all): its block draws are taken here, and
    // the warps without an accept test prepare the rest of it meanwhile, which
    // takes its preparation off the critical path when the first draft is rejected.
    const bool spec0 = !GREEDY && (!dense || keff == 0) && keff < kSW;  // (needs a warp without a test)
    if (spec0) draw_row_blocks(P, nk, 0, tid, kST, s_bnd, s_M, s_I);
    // the epilogue's inputs (written by no kernel of this call before this one)
    int kv_in = 0, gs_in = 0;
    float ema_in = 0.0f;
    if (tid == 0) {
        kv_in = P.kv_len[b];
        ema_in = P.ema[b];
        gs_in = P.gate_state != nullptr ? P.gate_state[b] : 0;
    }
    __syncthreads();
    // everything above reads the call's inputs only; the stream kernel's records from here on
    pdl_wait();

    auto pen_of = [&](int v, int j) -> bool {
        if constexpr (!PENALTY) return false;
        return pen_lookup(s_pkey, s_ppos, s_d, nh, P.W, v, j);
    };
    auto rowp_of = [&](int row) {
        return static_cast<const char*>(P.logits) + static_cast<size_t>(row) * P.V * ElemTraits<BF16>::SIZE;
    };
    // lane's vectors of block q of a row
    auto load_block = [&](const char* rowp, int q, uint4* r) {
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
            const int e0 = q * BLK + (u * 32 + lane) * EPV;
            r[u] = e0 < P.V ? load_vec_chk<BF16>(P, rowp, e0, P.V) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    auto elem_id = [&](int q, int k) { return q * BLK + ((k / EPV) * 32 + lane) * EPV + (k % EPV); };

    uint4* stg = reinterpret_cast<uint4*>(s_dyn + k2_blk_bytes(nblk)) + warp * (kBatch * 32 * VPL);
    // ---- 1. accept tests (T > 0) / argmax of every row (T = 0)
    for (int j = warp; j <= keff; j += kSW) {
        const int row = b * K1 + j;
        if constexpr (GREEDY) {
            // the block with the largest value first, then every block within the tie margin
            const float* bmx = P.bmax + static_cast<size_t>(row) * P.nblk;
            const char* rowp = rowp_of(row);
            float lb = -INFINITY;
            int lq = -1;
            for (int q = lane; q < P.nblk; q += 32) {
                const float x = bmx[q];
                if (x > lb || lq < 0) { lb = x; lq = q; }
            }
            const unsigned kq = __reduce_max_sync(0xffffffffu, score_key(lb));
            const unsigned own = __ballot_sync(0xffffffffu, score_key(lb) == kq);
            const int q0 = __shfl_sync(0xffffffffu, lq, __ffs(own) - 1);
            Top2 t = top2_empty();
            auto scan = [&](int q, float gth) {
                uint4 r[VPL];
                load_block(rowp, q, r);
#pragma unroll
                for (int u = 0; u < VPL; ++u) {
                    float x[EPV];
                    unpack<BF16>(r[u], x);
#pragma unroll
                    for (int e = 0; e < EPV; ++e) {
                        const int v = elem_id(q, u * EPV + e);
                        if (v >= P.V) continue;
                        const float z = transform_f32<SOFTCAP, PENALTY>(x[e], PENALTY && pen_of(v, j), P);
                        if (z >= gth) top2_push(t, z, v);
                    }
                }
            };
            scan(q0, -INFINITY);
            const unsigned kw = warp_best_key(t.s1);
            const float gth = kw ? key_score(kw) - cand_delta(key_score(kw)) : -INFINITY;
            for (int qb = 0; qb < P.nblk; qb += 32) {
                const int q = qb + lane;
                unsigned pass = __ballot_sync(0xffffffffu, q < P.nblk && q != q0 && block_zmax<SOFTCAP, PENALTY>(bmx[q], P) >= gth);
                while (pass != 0u) {
                    const int qq = qb + __ffs(pass) - 1;
                    pass &= pass - 1u;
                    scan(qq, gth);
                }
            }
            t = top2_warp_reduce(t);
            int y = t.i1;
            if (t.i2 >= 0 && t.s2 >= t.s1 - cand_delta(t.s1)) {
                if (lane == 0) {
                    count_diag(P, SPECNG_DIAG_GREEDY_F64);
                    const double z1 = transform_f64<SOFTCAP, PENALTY>(raw_logit_chk<BF16>(P, row, t.i1),
                                                                      PENALTY && pen_of(t.i1, j), P);
                    const double z2 = transform_f64<SOFTCAP, PENALTY>(raw_logit_chk<BF16>(P, row, t.i2),
                                                                      PENALTY && pen_of(t.i2, j), P);
                    if (better64(z2, t.i2, z1, t.i1)) y = t.i2;
                }
                y = __shfl_sync(0xffffffffu, y, 0);
            }
            if (lane == 0) {
                s_arg[j] = y;
                s_acc[j] = j < keff && s_d[j] >= 0 && s_d[j] < P.V && s_d[j] == y;
            }
        } else {
            if (j == keff) break;
            // the draft's logit and q first: their latency overlaps the sums'
            const int d = s_d[j];
            const bool dv = d >= 0 && d < P.V;
            float xd = 0.0f, qdf = 1.0f;
            double u = 0.0;
            bool pend = false;
            if (lane == 0 && dv) {
                xd = static_cast<float>(raw_logit_chk<BF16>(P, row, d));
                if (dense) qdf = P.q[(static_cast<size_t>(b) * P.K + j) * P.V + chk_id(P, d)];
                // the draw and the window test need no load: they run while the loads are in flight
                u = accept_uniform_f64(nk, static_cast<uint32_t>(j + 1));
                pend = pen_of(d, j);
            }
            // one pass over the segment sums: a lane keeps its first kPr records in registers
            constexpr int kPr = 4;
            SegSum* pr = P.part + static_cast<size_t>(row) * P.nchunk;
            float2 pv[kPr];
            float mf = -INFINITY;
            bool proof = false;  // a segment proved the test rejects (s < 0)
#pragma unroll
            for (int i = 0; i < kPr; ++i) {
                const int cc = lane + 32 * i;
                pv[i] = cc < P.nchunk ? __ldcg(reinterpret_cast<const float2*>(pr + cc)) : make_float2(0.0f, 0.0f);
            }
            // the rest (rows of many records, e.g. one per noise block): four loads in flight
            for (int c0 = lane + 32 * kPr; c0 < P.nchunk; c0 += 32 * kPr) {
                float2 pb[kPr];
#pragma unroll
                for (int u = 0; u < kPr; ++u) {
                    const int cc = c0 + 32 * u;
                    pb[u] = cc < P.nchunk ? __ldcg(reinterpret_cast<const float2*>(pr + cc)) : make_float2(0.0f, 0.0f);
                }
#pragma unroll
                for (int u = 0; u < kPr; ++u) {
                    if (pb[u].y != 0.0f || __float_as_uint(pb[u].x) != 0u) mf = fmaxf(mf, pb[u].x);
                    proof |= pb[u].y < 0.0f;
                }
            }
#pragma unroll
            for (int i = 0; i < kPr; ++i) {
                if (pv[i].y != 0.0f || __float_as_uint(pv[i].x) != 0u) mf = fmaxf(mf, pv[i].x);
                proof |= pv[i].y < 0.0f;
            }
            proof = __any_sync(0xffffffffu, proof);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mf = fmaxf(mf, __shfl_xor_sync(0xffffffffu, mf, off));
            // the records' sums relative to mf (each term <= its record's sum; fp32 keeps 2^-24
            // relative per term, far inside the accept test's margin)
            float Sf = 0.0f;
            auto term = [&](float2 p) {
                return ((p.y != 0.0f || __float_as_uint(p.x) != 0u) && p.x > -INFINITY)
                           ? p.y * ex2_approx((p.x - mf) * P.sc) : 0.0f;
            };
#pragma unroll
            for (int i = 0; i < kPr; ++i) Sf += term(pv[i]);
            for (int c0 = lane + 32 * kPr; c0 < P.nchunk; c0 += 32 * kPr) {
                float2 pb[kPr];
#pragma unroll
                for (int u = 0; u < kPr; ++u) {
                    const int cc = c0 + 32 * u;
                    pb[u] = cc < P.nchunk ? __ldcg(reinterpret_cast<const float2*>(pr + cc)) : make_float2(0.0f, 0.0f);
                }
#pragma unroll
                for (int u = 0; u < kPr; ++u) Sf += term(pb[u]);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) Sf += __shfl_xor_sync(0xffffffffu, Sf, off);
            for (int cc = lane; cc < P.nchunk; cc += 32) pr[cc] = SegSum{0.0f, 0.0f};  // leave the workspace zeroed
            if (lane == 0 && proof) {
                s_acc[j] = 0;
                s_ms[j] = make_float2(0.0f, 0.0f);
            } else if (lane == 0) {
                if (!(Sf > 0.0f && Sf < INFINITY && mf < INFINITY)) raise_status(P.status, SPECNG_DEV_NONFINITE);
                const float lsef = mf * P.invT + logf(Sf);
                int accepted = 0;
                if (dv) {
                    const double qd = static_cast<double>(qdf);
                    const float lp = transform_f32<SOFTCAP, PENALTY>(xd, pend, P) * P.invT - lsef;
                    const float lr = logf(static_cast<float>(u)) + logf(static_cast<float>(qd));
                    if (lr < lp - 1e-4f * (1.0f + fabsf(lp))) {
                        accepted = 1;
                    } else if (lr > lp + 1e-4f * (1.0f + fabsf(lp))) {
                        accepted = 0;
                    } else {
                        count_diag(P, SPECNG_DIAG_ACCEPT_F64);
                        accepted = accept_f64<SOFTCAP, PENALTY>(P, xd, pend, u, qd, mf, Sf);
                    }
                }
                s_acc[j] = accepted;
                s_ms[j] = make_float2(mf, Sf);
            }
        }
    }
    if constexpr (!GREEDY) {
        if (spec0 && warp >= keff)
            prepare_row<BF16, SOFTCAP, PENALTY>(P, nk, b, 0, keff > 0 && s_d[0] >= 0 && s_d[0] < P.V ? s_d[0] : -1,
                                                tid - 32 * keff, kST - 32 * keff, &s_thr0, s_bnd, s_M, s_I, s_pkey, s_ppos,
                                                s_d, nh, true);
    }
    __syncthreads();

    // ---- 2. acceptance length
    int a = keff;
    for (int i = 0; i < keff; ++i)
        if (!s_acc[i]) { a = i; break; }
    const int da = a < keff ? s_d[a] : -1;
    const bool dvalid = da >= 0 && da < P.V;
    const bool need = dense && !GREEDY && a < keff && dvalid;

    // ---- 3. the token at row a
    int y;
    if constexpr (GREEDY) {
        y = s_arg[a];
    } else if (need) {
        y = -1;  // the residual pass samples row a (CTA-uniform branch)
    } else {
        const int row = b * K1 + a;
        const int excl = (a < keff && dvalid) ? da : -1;  // point mass here: dense rejections took the branch above
        const char* rowp = rowp_of(row);
        const RowPhilox rp = row_philox(nk, static_cast<uint32_t>(a));
        if (a == 0 && spec0) {
            if (tid == 0) s_thr = s_thr0;  // row 0 was prepared during the accept tests
        } else {
            prepare_row<BF16, SOFTCAP, PENALTY>(P, nk, b, a, excl, tid, kST, &s_thr, s_bnd, s_M, s_I, s_pkey, s_ppos, s_d,
                                                nh, false);
        }
        __syncthreads();
        float thr = -INFINITY;
        if (s_thr != 0u) thr = key_score(s_thr) - cand_delta(key_score(s_thr));
        // the blocks whose bound reaches the best
        for (int qb = warp * 32; qb < nblk; qb += kST) {
            const int q = qb + lane;
            const bool pass = q < nblk && s_bnd[q] + bound_slack(s_bnd[q]) >= thr;
            const unsigned bal = __ballot_sync(0xffffffffu, pass);
            int at = 0;
            if (lane == 0 && bal) at = atomicAdd(&s_nl, __popc(bal));
            at = __shfl_sync(0xffffffffu, at, 0);
            if (pass) s_list[at + __popc(bal & ((1u << lane) - 1u))] = q;
        }
        __syncthreads();
        const int nl = s_nl;
        Top2 t = top2_empty();
        // the listed blocks, kBatch per warp at a time: their loads all in flight
        // together, one raw-logit screening threshold per block, then each lane
        // scores its own candidates (usually none or one per batch): the exact
        // transform (penalty) and the element's own draw
        for (int l0 = warp * kBatch; l0 < nl; l0 += kSW * kBatch) {
            // blocks whose bound no longer reaches the best found so far are skipped;
            // lane h < kBatch holds block h of the batch
            const unsigned kc0 = __shfl_sync(0xffffffffu, max(*reinterpret_cast<volatile unsigned*>(&s_thr), warp_best_key(t.s1)), 0);
            const float thw = kc0 != 0u ? key_score(kc0) - cand_delta(key_score(kc0)) : -INFINITY;
            thr = fmaxf(thr, thw);
            int myq = -1;
            if (lane < kBatch && l0 + lane < nl) {
                const int q = s_list[l0 + lane];
                if (s_bnd[q] + bound_slack(s_bnd[q]) >= thw) myq = q;
            }
            if (lane < kBatch) s_bq[warp][lane] = myq;
            int qh[kBatch];
#pragma unroll
            for (int h = 0; h < kBatch; ++h) qh[h] = __shfl_sync(0xffffffffu, myq, h);
            uint4 r[kBatch * VPL];
#pragma unroll
            for (int h = 0; h < kBatch; ++h)
#pragma unroll
                for (int u = 0; u < VPL; ++u) {
                    const int e0 = qh[h] * BLK + (u * 32 + lane) * EPV;
                    r[h * VPL + u] = (qh[h] >= 0 && e0 < P.V) ? load_vec_chk<BF16>(P, rowp, e0, P.V)
                                                               : make_uint4(0u, 0u, 0u, 0u);
                }
            // screening thresholds (a penalty below 1 may raise a value: then every
            // element goes to the exact test)
            float xt[kBatch];
#pragma unroll
            for (int h = 0; h < kBatch; ++h)
                xt[h] = qh[h] < 0 ? INFINITY
                                  : ((PENALTY && P.rep < 1.0f) ? -INFINITY : raw_screen<SOFTCAP>(thr, ln_fast(s_M[qh[h]]), P));
#pragma unroll
            for (int i = 0; i < kBatch * VPL; ++i) stg[i * 32 + lane] = r[i];
            unsigned long long cm = 0ull;  // bit 8 h + k: element k of my share of block h
#pragma unroll
            for (int h = 0; h < kBatch; ++h)
#pragma unroll
                for (int u = 0; u < VPL; ++u) {
                    const uint4 rv = r[h * VPL + u];
                    unsigned bits;
                    if constexpr (BF16) {
                        bits = bf16x8_ge_bits(rv, bf16x2_floor(xt[h]));
                    } else {
                        bits = (__uint_as_float(rv.x) >= xt[h] ? 1u : 0u) | (__uint_as_float(rv.y) >= xt[h] ? 2u : 0u) |
                               (__uint_as_float(rv.z) >= xt[h] ? 4u : 0u) | (__uint_as_float(rv.w) >= xt[h] ? 8u : 0u);
                    }
                    cm |= static_cast<unsigned long long>(bits) << (h * NE + u * EPV);
                }
            __syncwarp();  // the staging and the batch's block ids are visible
            while (cm != 0ull) {
                const int bit = __ffsll(static_cast<long long>(cm)) - 1;
                cm &= cm - 1ull;
                const int h = bit / NE, k = bit % NE;
                const int q = s_bq[warp][h];
                const int v = elem_id(q, k);
                if (v >= P.V || v == excl) continue;
                const float xv = elem_of_stage<BF16>(stg, ((h * VPL + k / EPV) * 32 + lane) * EPV + k % EPV);
                const float zb = transform_f32<SOFTCAP, PENALTY>(xv, PENALTY && pen_of(v, a), P) * P.invT;
                const float Mq = s_M[q];
                const float lnMq = ln_fast(Mq);
                if (zb - lnMq + bound_slack(zb - lnMq) < thr) continue;
                const float score = zb - ln_fast(noise_exp_f32(rp, Mq, s_I[q], static_cast<uint32_t>(v)));
                if (score >= thr) {
                    top2_push(t, score, v);
                    thr = fmaxf(thr, t.s1 - cand_delta(t.s1));
                }
            }
            __syncwarp();  // the staging is read before the next batch overwrites it
            // share the best with the other warps
            const unsigned kw = warp_best_key(t.s1);
            if (kw != 0u && lane == 0) atomicMax(&s_thr, kw);
            const unsigned kc = max(*reinterpret_cast<volatile unsigned*>(&s_thr), kw);
            if (kc != 0u) thr = fmaxf(thr, key_score(kc) - cand_delta(key_score(kc)));
        }
        t = top2_warp_reduce(t);
        if (lane == 0) s_top[warp] = t;
        __syncthreads();
        if (warp == 0) {
            Top2 tw = lane < kSW ? s_top[lane] : top2_empty();
#pragma unroll
            for (int off = kSW / 2; off > 0; off >>= 1) tw = top2_merge(tw, top2_shfl_xor(tw, off));
            int w = tw.i1;
            if (lane == 0 && tw.i2 >= 0 && tw.s2 >= tw.s1 - cand_delta(tw.s1)) {
                count_diag(P, SPECNG_DIAG_SAMPLE_F64);
                w = rescore_top2_f64<BF16, SOFTCAP, PENALTY>(P, nk, row, a, tw.i1, tw.i2, PENALTY && pen_of(tw.i1, a),
                                                            PENALTY && pen_of(tw.i2, a));
            }
            if (lane == 0) s_y = w;
        }
        __syncthreads();
        y = s_y;
    }

    // ---- 4. epilogue (with dense q the residual pass writes the token at row a)
    if (tid < K1)
        P.out_tokens[static_cast<size_t>(b) * K1 + tid] = tid < a ? s_d[tid] : (tid == a && !need ? y : -1);
    if (tid == 0) {
        P.out_accept[b] = a;
        P.kv_len[b] = kv_in - kb + a;
        if (P.gate_state != nullptr) P.gate_state[b] = cool_after(P, gs_in, a, keff);
        if (keff > 0) P.ema[b] = ema_update(ema_in, P.tau, a, keff);
        if (need) {
            RowRes rr;
            rr.m = s_ms[a].x;
            rr.S = s_ms[a].y;
            rr.winner = -1;
            rr.pad = 0;
            P.rowres[b * K1 + a] = rr;
            SeqRes sr;
            sr.a = a;
            sr.keff = keff;
            sr.need_residual = 1;
            sr.pad = 0;
            P.seqres[b] = sr;
        }
    }
}

// ---------------------------------------------------------------- K2
// Dense draft distributions: after a rejection at row a, sample from the
// residual max(0, p_a - q_a) by Gumbel-max over row a (the logits of row a
// read once more and q_a read at the candidates only, for the rejected
// sequences).  log r_v <= log p_v = z_v / T - lse and E_v >= M of its block,
// so an element can beat the best score only if z_v / T - lse - ln M reaches
// it.  The best starts from the exact residual score of each lane's largest p
// and is shared by the CTA's warps and, through the workspace, by the CTAs of
// the row.

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kNV = 8;  // 16-byte vectors per thread per chunk
static_assert(kResChunkBytes == kThreads * kNV * 16, "residual chunk layout");

// log max(0, p - q) for log p = lp, in fp32 without cancellation: for q > 0,
// p - q = q (e^(lp - ln q) - 1), and expm1 keeps the relative accuracy when
// p and q are close.  -inf when the residual is zero.
__device__ __forceinline__ float log_residual(float lp, float q) {
    if (!(q > 0.0f)) return lp;
    const float d = lp - logf(q);
    if (!(d > 0.0f)) return -INFINITY;
    return logf(q) + logf(expm1f(d));
}

// Penalty window of row j of sequence b: the last W tokens of
// history[:lens] ++ d_1..d_j.  Fills s_win / s_nwin and, for the chunk
// [v0, v1), the bitmap s_bm.  Whole CTA calls it.
template <int CHUNK>
__device__ __forceinline__ void build_window(const VerifyDev& P, int b, int j, int v0, int v1,
                                             uint32_t* s_bm, int* s_win, int* s_nwin) {
    const int tid = threadIdx.x;
    int L = P.lens[b];
    L = L < 0 ? 0 : (static_cast<int64_t>(L) > P.hist_stride ? static_cast<int>(P.hist_stride) : L);
    const int total = L + j;
    const int start = total - P.W > 0 ? total - P.W : 0;
    const int nw = total - start;
    for (int t = tid; t < CHUNK / 32; t += kThreads) s_bm[t] = 0u;
    int tok = -1;
    if (tid < nw) {
        const int idx = start + tid;
        tok = idx < L ? hist_at(P, b, idx) : draft_at(P, b, idx - L);
        s_win[tid] = tok;
    }
    if (tid == 0) *s_nwin = nw;
    __syncthreads();
    if (tok >= v0 && tok < v1) atomicOr(&s_bm[(tok - v0) >> 5], 1u << ((tok - v0) & 31));
    __syncthreads();
}

// Gumbel-max over p of row `row` (sampling position a), every id competing:
// argmax_v (z_v / T - ln E_v), the rule an all-zero residual falls back to.
// Whole CTA calls it; it reads the row once and draws per-id noise only
// where a warp's running best can still be reached (E_v >= M of its block).
// Slow by design (the case needs p <= q everywhere in floating point) but
// exact: the top two are re-scored in fp64.  s_top: kWarps Top2 slots.
template <bool BF16, bool SOFTCAP, bool PENALTY>
__device__ __noinline__ int sample_p_row(const VerifyDev& P, const NoiseKey& nk, int row, int a, const int* s_win, int nw,
                                         Top2* s_top) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    constexpr int BLK = 1 << kNoiseBlockShift;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const char* rowp = static_cast<const char*>(P.logits) + static_cast<size_t>(row) * P.V * ElemTraits<BF16>::SIZE;
    const RowPhilox rp = row_philox(nk, static_cast<uint32_t>(a));
    auto pen = [&](int v) {
        if constexpr (!PENALTY) return false;
        for (int t = 0; t < nw; ++t)
            if (s_win[t] == v) return true;
        return false;
    };
    Top2 t = top2_empty();
    float thr = -INFINITY;
    __syncthreads();  // s_top may still be read by the caller's earlier merge
    for (int q = warp; q < P.nblk; q += kWarps) {
        const BlockNoise bn = block_noise(nk, static_cast<uint32_t>(q), static_cast<uint32_t>(a));
        for (int e0 = q * BLK + lane * EPV; e0 < min(P.V, (q + 1) * BLK); e0 += 32 * EPV) {
            float x[EPV];
            unpack<BF16>(load_vec_chk<BF16>(P, rowp, e0, P.V), x);
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                const int v = e0 + e;
                if (v >= P.V) break;
                float zb = transform_f32<SOFTCAP, false>(x[e], false, P);
                if (PENALTY && P.rep < 1.0f) zb = fmaxf(zb, transform_f32<SOFTCAP, true>(x[e], true, P));
                zb *= P.invT;
                if (zb - bn.lnM + bound_slack(zb - bn.lnM) < thr) continue;
                const float z = transform_f32<SOFTCAP, PENALTY>(x[e], PENALTY && pen(v), P) * P.invT;
                const float score = z - ln_fast(noise_exp_f32(rp, bn.M, bn.I, static_cast<uint32_t>(v)));
                top2_push(t, score, v);
                thr = fmaxf(thr, t.s2 > -INFINITY ? t.s2 - cand_delta(t.s2) : -INFINITY);
            }
        }
        const unsigned kw = warp_best_key(t.s1);
        if (kw != 0u) thr = fmaxf(thr, key_score(kw) - cand_delta(key_score(kw)));
    }
    t = top2_warp_reduce(t);
    if (lane == 0) s_top[warp] = t;
    __syncthreads();
    Top2 tw = lane < kWarps ? s_top[lane] : top2_empty();
#pragma unroll
    for (int off = kWarps / 2; off > 0; off >>= 1) tw = top2_merge(tw, top2_shfl_xor(tw, off));
    int w = tw.i1;
    if (tw.i2 >= 0 && tw.s2 >= tw.s1 - cand_delta(tw.s1)) {
        if (threadIdx.x == 0) count_diag(P, SPECNG_DIAG_SAMPLE_F64);
        double sc[2];
        for (int h = 0; h < 2; ++h) {
            const int id = h == 0 ? tw.i1 : tw.i2;
            const double z = transform_f64<SOFTCAP, PENALTY>(raw_logit_chk<BF16>(P, row, id),
                                                             PENALTY && pen(id), P);
            sc[h] = z / P.Td - log(noise_exp_f64(nk, static_cast<uint32_t>(id), static_cast<uint32_t>(a)));
        }
        if (better64(sc[1], tw.i2, sc[0], tw.i1)) w = tw.i2;
    }
    return w;  // the same value in every thread
}

template <bool BF16, bool SOFTCAP, bool PENALTY>
__global__ void __launch_bounds__(kThreads, 2) verify_residual_kernel(const __grid_constant__ VerifyDev P) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    constexpr int CHUNK = res_chunk_elems<BF16>();
    constexpr int NB = CHUNK >> kNoiseBlockShift;
    __shared__ uint32_t s_bm[PENALTY ? CHUNK / 32 : 1];
    __shared__ int s_win[PENALTY ? SPECNG_MAX_REP_WINDOW : 1];
    __shared__ int s_nwin;
    __shared__ Top2 s_t[kWarps];
    __shared__ int s_last;
    __shared__ int s_dec;
    __shared__ unsigned s_thr;
    __shared__ BlockNoise s_bn[NB];
    __shared__ uint16_t s_q2[kWarps * 32 * kNV * EPV];  // per-warp candidate queues (chunk offsets)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K1 = P.K + 1;
    const int b = blockIdx.x / P.nchunk2;
    const int c = blockIdx.x - b * P.nchunk2;
    pdl_wait();  // the decision kernel's records
    const int need = __ldcg(&P.seqres[b].need_residual);
    if (!need) return;
    const int a = __ldcg(&P.seqres[b].a);
    const int row = b * K1 + a;
    const float2 rms = __ldcg(reinterpret_cast<const float2*>(&P.rowres[row]));
    const float lse_f = rms.x * P.invT + logf(rms.y);
    const int v0 = c * CHUNK;
    const int v1 = min(P.V, v0 + CHUNK);
    const char* rowp = static_cast<const char*>(P.logits) +
                       static_cast<size_t>(row) * P.V * ElemTraits<BF16>::SIZE;
    const float* qrow = P.q + (static_cast<size_t>(b) * P.K + a) * P.V;
    NoiseKey nk = noise_key(P);
    nk.seq = static_cast<uint32_t>(b);
    const RowPhilox rp = row_philox(nk, static_cast<uint32_t>(a));

    if (tid == 0) s_thr = 0u;
    if (tid < NB) s_bn[tid] = block_noise(nk, static_cast<uint32_t>((v0 >> kNoiseBlockShift) + tid), static_cast<uint32_t>(a));
    if constexpr (PENALTY) build_window<CHUNK>(P, b, a, v0, v1, s_bm, s_win, &s_nwin);
    __syncthreads();
    // the chunk in registers: every thread's eight 16-byte vectors, loaded together
    uint4 rv[kNV];
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
        const int e0 = v0 + (i * kThreads + tid) * EPV;
        rv[i] = e0 < v1 ? load_vec_chk<BF16>(P, rowp, e0, v1) : make_uint4(0u, 0u, 0u, 0u);
    }
    auto lp_of = [&](float x, bool pen) { return transform_f32<SOFTCAP, PENALTY>(x, pen, P) * P.invT - lse_f; };
    auto pen_at = [&](int off) -> unsigned {
        if constexpr (PENALTY) return (s_bm[off >> 5] >> (off & 31)) & ((1u << EPV) - 1u);
        return 0u;
    };
    // ---- seed: each lane scores the residual of its largest p; the CTA and the row
    //      share the best (any element's exact score bounds the best from below)
    Top2 tt = top2_empty();
    int seeded = -1;
    {
        float lm = -INFINITY;
        int im = -1;
#pragma unroll
        for (int i = 0; i < kNV; ++i) {
            const int off = (i * kThreads + tid) * EPV;
            const int nv = min(EPV, v1 - (v0 + off));
            if (nv <= 0) continue;
            float x[EPV];
            unpack<BF16>(rv[i], x);
            const unsigned pb = pen_at(off);
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                if (e >= nv) break;
                const float lp = lp_of(x[e], (pb >> e) & 1u);
                if (lp > lm) { lm = lp; im = v0 + off + e; }
            }
        }
        float t0 = -INFINITY;
        if (im >= 0) {
            const float lr = log_residual(lm, __ldcs(qrow + im));
            if (lr > -INFINITY) {
                const BlockNoise bn = s_bn[(im - v0) >> kNoiseBlockShift];
                t0 = lr - ln_fast(noise_exp_f32(rp, bn.M, bn.I, static_cast<uint32_t>(im)));
                top2_push(tt, t0, im);
                seeded = im;
            }
        }
        const unsigned kw = warp_best_key(t0);
        if (kw != 0u && lane == 0) atomicMax(&s_thr, kw);
    }
    __syncthreads();
    if (tid == 0 && s_thr != 0u) atomicMax(&P.row_thr[row], s_thr);
    float thr = -INFINITY;
    {
        const unsigned kb = max(s_thr, __ldcg(&P.row_thr[row]));
        if (kb != 0u) {
            const float bw = key_score(kb);
            thr = bw - cand_delta(bw);
        }
    }
    // ---- candidates: log r_v - ln E_v <= lp_v - ln M, so that bound must reach the best.
    //      They are compacted per warp (chunk offsets), then scored 32 at a time, so the
    //      loads of a batch (the logit, from L2, and q) are issued together
    uint16_t* qw = s_q2 + warp * (32 * kNV * EPV);
    int nq = 0;
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
        const int off = (i * kThreads + tid) * EPV;
        const int nv = min(EPV, v1 - (v0 + off));
        unsigned mi = 0u;
        if (nv > 0) {
            float x[EPV];
            unpack<BF16>(rv[i], x);
            const unsigned pb = pen_at(off);
            const float lnM = s_bn[off >> kNoiseBlockShift].lnM;
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                if (e >= nv) break;
                const float bnd = lp_of(x[e], (pb >> e) & 1u) - lnM;
                if (bnd + bound_slack(bnd) >= thr && v0 + off + e != seeded) mi |= 1u << e;
            }
        }
        const unsigned cnt = __popc(mi);
        unsigned incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        int slot = nq + static_cast<int>(incl - cnt);
        while (mi != 0u) {
            const int e = __ffs(mi) - 1;
            mi &= mi - 1u;
            qw[slot++] = static_cast<uint16_t>(off + e);
        }
        nq += static_cast<int>(__shfl_sync(0xffffffffu, incl, 31));
    }
    __syncwarp();
    for (int base = 0; base < nq; base += 32) {
        const int idx = base + lane;
        const bool in = idx < nq;
        const int loc = in ? static_cast<int>(qw[idx]) : 0;
        const int v = v0 + loc;
        const float x = in ? static_cast<float>(raw_logit_chk<BF16>(P, row, v)) : 0.0f;
        const float qv = in ? __ldcs(qrow + v) : 0.0f;
        const bool pen = PENALTY && ((s_bm[loc >> 5] >> (loc & 31)) & 1u);
        const BlockNoise bn = s_bn[loc >> kNoiseBlockShift];
        const float lp = lp_of(x, pen);
        const float lr = in && lp - bn.lnM + bound_slack(lp) >= thr ? log_residual(lp, qv) : -INFINITY;
        const bool live = lr > -INFINITY && lr - bn.lnM + bound_slack(lr) >= thr;
        if (__any_sync(0xffffffffu, live)) {
            const float E = noise_exp_f32(rp, bn.M, bn.I, static_cast<uint32_t>(v));
            if (live) {
                const float score = lr - ln_fast(E);
                if (score >= thr) {
                    top2_push(tt, score, v);
                    thr = fmaxf(thr, tt.s1 - cand_delta(tt.s1));
                }
            }
        }
        // share the warp's best with the CTA, adopt the CTA's
        const unsigned kw = warp_best_key(tt.s1);
        if (kw != 0u && lane == 0) atomicMax(&s_thr, kw);
        const unsigned kb = max(*reinterpret_cast<volatile unsigned*>(&s_thr), kw);
        if (kb != 0u) {
            const float bw = key_score(kb);
            thr = fmaxf(thr, bw - cand_delta(bw));
        }
    }
    tt = top2_warp_reduce(tt);
    if (lane == 0) s_t[warp] = tt;
    __syncthreads();
    if (warp == 0) {
        Top2 t = lane < kWarps ? s_t[lane] : top2_empty();
#pragma unroll
        for (int off = 4; off > 0; off >>= 1) t = top2_merge(t, top2_shfl_xor(t, off));
        if (lane == 0) {
            st_partial(P.part2 + blockIdx.x, 0.0f, 0.0f, t);
            __threadfence();
            const unsigned prev = atomicAdd(&P.seq_ticket2[b], 1u);
            s_last = prev == static_cast<unsigned>(P.nchunk2 - 1);
        }
    }
    __syncthreads();
    if (!s_last) return;  // CTA-uniform: the row's last CTA decides
    __threadfence();
    if (warp == 0) {
        if (lane == 0) {
            P.seq_ticket2[b] = 0u;
            P.row_thr[row] = 0u;  // leave the workspace zeroed
        }
        const Partial* pr = P.part2 + static_cast<size_t>(b) * P.nchunk2;
        Top2 t = top2_empty();
        for (int cc = lane; cc < P.nchunk2; cc += 32) t = top2_merge(t, ldcg_partial(pr + cc).t);
        t = top2_warp_reduce(t);
        __syncwarp();
        for (int cc = lane; cc < P.nchunk2; cc += 32) st_zero(const_cast<Partial*>(pr) + cc);
        const int nw = PENALTY ? s_nwin : 0;
        const bool pen1 = PENALTY && t.i1 >= 0 ? warp_in_window(t.i1, s_win, nw) : false;
        const bool pen2 = PENALTY && t.i2 >= 0 ? warp_in_window(t.i2, s_win, nw) : false;
        // fp32 decision when it is safe: the best is clear of the second by more than
        // the fp32 error and its residual clearly positive (ln p - ln q > 1e-4, far
        // above the fp32 error of either); otherwise both are re-scored in fp64
        float dres = 0.0f;
        if (lane == 0 && t.i1 >= 0) {
            const float x1 = static_cast<float>(raw_logit_chk<BF16>(P, row, t.i1));
            dres = lp_of(x1, pen1) - logf(__ldcg(qrow + t.i1));
        }
        if (lane == 0) {
            st_zero(P.rowres + row);
            st_zero(P.seqres + b);
            double best = -INFINITY;
            int winner = -1;
            const bool clear2 = t.i2 < 0 || !(t.s2 >= t.s1 - cand_delta(t.s1));
            if (t.i1 >= 0 && clear2 && dres > 1e-4f) winner = t.i1;
            if (winner < 0) {
            count_diag(P, SPECNG_DIAG_RESIDUAL_F64);
            const double lse = static_cast<double>(rms.x) / P.Td + log(static_cast<double>(rms.y));
            for (int h = 0; h < 2; ++h) {
                const int id = h == 0 ? t.i1 : t.i2;
                if (id < 0) continue;
                if (h == 1 && !(t.s2 >= t.s1 - cand_delta(t.s1))) continue;
                const double z = transform_f64<SOFTCAP, PENALTY>(raw_logit_chk<BF16>(P, row, id),
                                                                 h == 0 ? pen1 : pen2, P);
                const double rsd = exp(z / P.Td - lse) - static_cast<double>(qrow[id]);
                if (!(rsd > 0.0)) continue;
                const double score = log(rsd) - log(noise_exp_f64(nk, static_cast<uint32_t>(id), static_cast<uint32_t>(a)));
                if (winner < 0 || better64(score, id, best, winner)) { best = score; winner = id; }
            }
            }
            s_dec = winner;  // -1 for an all-zero residual
        }
    }
    __syncthreads();
    int winner = s_dec;
    // all-zero residual (p <= q everywhere): sample from p at row a with the same noise
    if (winner < 0) {
        if (tid == 0) count_diag(P, SPECNG_DIAG_RESIDUAL_ZERO);
        winner = sample_p_row<BF16, SOFTCAP, PENALTY>(P, nk, row, a, s_win, PENALTY ? s_nwin : 0, s_t);
    }
    if (tid == 0) P.out_tokens[static_cast<size_t>(b) * K1 + a] = winner;
}

}  // namespace specng

#include "verify_fused.cuh"

namespace specng {

// ---------------------------------------------------------------- launch

// Event recorded on the stream between the streaming kernel and the decision
// kernel of every spec_verify call while it is set (a measurement hook: it
// lets a caller time the streaming kernel alone; the decision kernel then
// starts after the streaming kernel has finished instead of overlapping its
// tail).  One process-wide slot.
__host__ inline cudaEvent_t& verify_marker() {
    static cudaEvent_t marker = nullptr;
    return marker;
}

// Per-device flag for a one-time function attribute (the attribute belongs to
// the device's context, so each device needs its own call).
__host__ inline bool* attr_flag(bool* flags) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) dev = 0;
    return &flags[dev];
}

__host__ inline int sm_count_cached() {
    static int cached[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 1;
    if (cached[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 1;
    }
    return cached[dev];
}

template <bool BF16, bool G, bool C, bool R>
cudaError_t launch_stream(const VerifyDev& P, cudaStream_t s) {
    // one persistent CTA per SM; the staging ring lives in dynamic shared memory
    constexpr size_t smem = k1_dyn_smem<R>();
    static bool configured[128] = {};
    bool* done = attr_flag(configured);
    if (!*done) {
        const cudaError_t e = cudaFuncSetAttribute(verify_stream_kernel<BF16, G, C, R>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        *done = true;
    }
    return launch_chained(verify_stream_kernel<BF16, G, C, R>, dim3(kK1PerSM * sm_count_cached()), dim3(kPThreads), smem, s,
                          P);
}

template <bool BF16, bool G, bool C, bool R>
cudaError_t launch_seq(const VerifyDev& P, cudaStream_t s) {
    // block scratch of the sampled row (when it fits) and the warps' staging
    const size_t smem = G ? 0 : k2_dyn_smem(P.nblk, BF16);
    static bool configured[128] = {};
    bool* done = attr_flag(configured);
    if (!G && !*done) {
        const cudaError_t e = cudaFuncSetAttribute(verify_seq_kernel<BF16, G, C, R>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(k2_dyn_smem(kSmemBlkCap, BF16)));
        if (e != cudaSuccess) return e;
        *done = true;
    }
    return launch_chained(verify_seq_kernel<BF16, G, C, R>, dim3(static_cast<unsigned>(P.B)), dim3(kST), smem, s, P);
}

template <bool BF16, bool C, bool R>
cudaError_t launch_residual(const VerifyDev& P, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>(P.B) * static_cast<unsigned>(P.nchunk2);
    return launch_chained(verify_residual_kernel<BF16, C, R>, dim3(grid), dim3(kThreads), 0, s, P);
}

template <bool BF16, bool G, bool C, bool R>
cudaError_t launch_fused(const VerifyDev& P, cudaStream_t s) {
    constexpr size_t smem = fused_dyn_smem<BF16, R>();
    static bool configured[128] = {};
    bool* done = attr_flag(configured);
    if (!*done) {
        const cudaError_t e = cudaFuncSetAttribute(verify_fused_kernel<BF16, G, C, R>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        *done = true;
    }
    return launch_chained(verify_fused_kernel<BF16, G, C, R>, dim3(sm_count_cached()), dim3(kFThreads), smem, s, P);
}

template <bool BF16, bool G, bool C, bool R>
cudaError_t launch_all(const VerifyDev& P, bool dense, cudaStream_t s) {
    if (P.fused) {
        cudaError_t e = launch_fused<BF16, G, C, R>(P, s);
        if (e != cudaSuccess) return e;
        if (cudaEvent_t m = verify_marker()) e = cudaEventRecord(m, s);  // measurement only: after the one kernel
        return e;
    }
    cudaError_t e = cudaSuccess;
    if (!P.records_given) {
        e = launch_stream<BF16, G, C, R>(P, s);
        if (e != cudaSuccess) return e;
    }
    if (cudaEvent_t m = verify_marker()) {
        e = cudaEventRecord(m, s);  // measurement only: ends the streaming (or LM-head) kernel's span
        if (e != cudaSuccess) return e;
    }
    e = launch_seq<BF16, G, C, R>(P, s);
    if (e != cudaSuccess || !dense || G) return e;
    return launch_residual<BF16, C, R>(P, s);
}

template <bool BF16, bool G>
cudaError_t launch_all_cr(const VerifyDev& P, bool c, bool r, bool dense, cudaStream_t s) {
    if (c) return r ? launch_all<BF16, G, true, true>(P, dense, s) : launch_all<BF16, G, true, false>(P, dense, s);
    return r ? launch_all<BF16, G, false, true>(P, dense, s) : launch_all<BF16, G, false, false>(P, dense, s);
}

// The kernels of one spec_verify call for one logits dtype: the streaming
// kernel, the decision kernel and, for dense q at T > 0, the residual pass.
template <bool BF16>
cudaError_t launch_verify_dtype(const VerifyDev& P, bool greedy, bool softcap, bool penalty, bool dense,
                                cudaStream_t s);

// The fused LM-head kernel (logits = h W^T on the tensor cores, with the
// per-block records in its epilogue), then the decision kernel and, for dense
// q at T > 0, the residual pass.  cudaErrorInvalidValue: the tensor maps of
// hidden / weight could not be encoded.
cudaError_t launch_lmhead_verify(const void* hidden, const void* weight, int d, void* logits, VerifyDev P, bool greedy,
                                 bool softcap, bool dense, cudaStream_t s);

template <bool BF16>
cudaError_t launch_verify_impl(const VerifyDev& P, bool greedy, bool softcap, bool penalty, bool dense,
                               cudaStream_t s) {
    return greedy ? launch_all_cr<BF16, true>(P, softcap, penalty, dense, s)
                  : launch_all_cr<BF16, false>(P, softcap, penalty, dense, s);
}

}  // namespace specng
