// spec_verify kernels (sm_103a): the streaming pass over the logit rows with
// the row merges and sequence epilogues folded in, and the dense-q residual
// pass.
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
// at most log w_v - ln M.  The streaming pass keeps, per row, the running
// best score; a block whose largest logit cannot reach it under that bound
// is skipped without a single per-id draw.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace specng {

template <bool BF16> struct ElemTraits;
template <> struct ElemTraits<true> { static constexpr int EPV = 8; static constexpr int SIZE = 2; };
template <> struct ElemTraits<false> { static constexpr int EPV = 4; static constexpr int SIZE = 4; };

// One chunk of a row = one 64 KB stage of the streaming ring; the residual
// pass takes 32 KB chunks, one per CTA.
constexpr int kChunkBytes = 32768;
constexpr int kResChunkBytes = 32768;
template <bool BF16>
__host__ __device__ constexpr int chunk_elems() { return kChunkBytes / ElemTraits<BF16>::SIZE; }
template <bool BF16>
__host__ __device__ constexpr int res_chunk_elems() { return kResChunkBytes / ElemTraits<BF16>::SIZE; }

// Workspace records.
struct __align__(32) Partial {
    float m, s;  // maximum (transformed units) and sum of exp((z - m) / T) of a row segment
    Top2 t;      // top-two candidates (fp32 scores)
    int pad[2];
};
struct __align__(16) RowRes {
    double lse;    // log-sum-exp of row / T (T > 0)
    int winner;    // sampled id of this row (residual or bonus candidate); argmax at T = 0
    int accepted;  // accept decision for the draft this row verifies
};
struct __align__(16) SeqRes {
    int a, keff, need_residual, pad;
};

struct VerifyDev {
    const void* logits;
    int B, K, V, nchunk;      // nchunk: streaming chunks per row
    int nchunk2;              // residual-pass chunks per row
    const int32_t* drafts;
    const float* q;
    const int32_t* k;
    const int32_t* hist;
    int64_t hist_stride;
    const int32_t* lens;
    float T, invT, sc;        // temperature, 1/T, log2(e)/T
    double Td;                // (double)T
    float cap, invcap;        // soft cap c and 1/c
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
    Partial* part;
    RowRes* rowres;
    SeqRes* seqres;
    unsigned* row_ticket;
    unsigned* row_thr;        // best residual score published per row (score_key)
    unsigned* seq_ticket;
    Partial* part2;
    unsigned* seq_ticket2;
    unsigned* status;
};

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

__device__ __forceinline__ int gate_keff(const VerifyDev& P, int b, int* kb_out, bool flag) {
    int kb = P.k[b];
    if (kb < 0 || kb > P.K) {
        if (flag) raise_status(P.status, SPECNG_DEV_BAD_K);
        kb = kb < 0 ? 0 : P.K;
    }
    if (kb_out) *kb_out = kb;
    if (P.gate && kb > 0 && !(P.ema[b] >= P.thresh)) return 0;
    return kb;
}

// Slack of the block bound: covers the fp32 rounding of z / T and ln M.
__device__ __forceinline__ float bound_slack(float z) { return 1e-5f * (1.0f + fabsf(z)); }

// ---------------------------------------------------------------- row merge
// One warp: combine the row's segment partials (log-sum-exp, sampled
// candidate), run the accept test of the draft the row verifies; the last
// row of a sequence to finish runs the epilogue (tokens, kv_len, EMA).

template <bool BF16, bool GREEDY, bool SOFTCAP, bool PENALTY>
__device__ __noinline__ void merge_row(const VerifyDev& P, int row) {
    const int lane = threadIdx.x & 31;
    const int K1 = P.K + 1;
    const int b = row / K1, j = row - b * K1;
    int kb;
    const int keff = gate_keff(P, b, &kb, false);
    const bool dense = P.q != nullptr;
    NoiseKey nk = P.nk;
    nk.seq = static_cast<uint32_t>(b);
    int nh = 0, L = 0;
    if constexpr (PENALTY) {
        L = P.lens[b];
        L = L < 0 ? 0 : (static_cast<int64_t>(L) > P.hist_stride ? static_cast<int>(P.hist_stride) : L);
        nh = L < P.W ? L : P.W;
    }
    const WindowView wv{PENALTY ? P.hist + static_cast<size_t>(b) * P.hist_stride + (L - nh) : nullptr,
                        P.drafts + static_cast<size_t>(b) * P.K, nh, PENALTY ? P.W : 0};

    // the draft's logit (and q) are loaded first: their latency overlaps the partials'
    const int dnext = j < keff ? wv.drafts[j] : -1;
    const bool dvalid = dnext >= 0 && dnext < P.V;
    float xd = 0.0f, qd = 1.0f;
    if (!GREEDY && lane == 0 && dvalid) {
        xd = static_cast<float>(raw_logit_f64<BF16>(P.logits, row, P.V, dnext));
        if (dense) qd = P.q[(static_cast<size_t>(b) * P.K + j) * P.V + dnext];
    }

    // one partial per row segment, stored at the segment's last chunk; the
    // other slots are all-zero (a written partial never is)
    Partial* pr = P.part + static_cast<size_t>(row) * P.nchunk;
    constexpr int kHeld = 2;
    Partial held[kHeld];
    float mf = -INFINITY;
#pragma unroll
    for (int h = 0; h < kHeld; ++h) {
        const int cc = lane + 32 * h;
        held[h] = cc < P.nchunk ? ldcg_partial(pr + cc) : Partial{0.0f, 0.0f, top2_empty(), {0, 0}};
        if (cc < P.nchunk && (held[h].s != 0.0f || __float_as_uint(held[h].m) != 0u)) mf = fmaxf(mf, held[h].m);
    }
    for (int cc = lane + 32 * kHeld; cc < P.nchunk; cc += 32) {
        const Partial p = ldcg_partial(pr + cc);
        if (p.s != 0.0f || __float_as_uint(p.m) != 0u) mf = fmaxf(mf, p.m);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mf = fmaxf(mf, __shfl_xor_sync(0xffffffffu, mf, off));
    double S = 0.0;
    Top2 t = top2_empty();
#pragma unroll
    for (int h = 0; h < kHeld; ++h) {
        const Partial& p = held[h];
        if (lane + 32 * h >= P.nchunk || (p.s == 0.0f && __float_as_uint(p.m) == 0u)) continue;
        if (!GREEDY && p.m > -INFINITY) S += static_cast<double>(p.s) * static_cast<double>(expf((p.m - mf) * P.invT));
        t = top2_merge(t, p.t);
    }
    for (int cc = lane + 32 * kHeld; cc < P.nchunk; cc += 32) {
        const Partial p = ldcg_partial(pr + cc);
        if (p.s == 0.0f && __float_as_uint(p.m) == 0u) continue;
        if (!GREEDY && p.m > -INFINITY) S += static_cast<double>(p.s) * static_cast<double>(expf((p.m - mf) * P.invT));
        t = top2_merge(t, p.t);
    }
    S = warp_sum_f64(S);
    t = top2_warp_reduce(t);
    __syncwarp();
    for (int cc = lane; cc < P.nchunk; cc += 32) st_zero(pr + cc);  // leave the workspace zeroed
    if (lane == 0) P.row_ticket[row] = 0u;
    const double lse = GREEDY ? 0.0 : static_cast<double>(mf) / P.Td + log(S);
    if (!GREEDY && !(S > 0.0 && S < INFINITY && mf < INFINITY) && lane == 0)
        raise_status(P.status, SPECNG_DEV_NONFINITE);

    // winner: fp32 order unless the two best are within the fp32 error, then fp64
    int winner = t.i1;
    const bool close = t.i2 >= 0 && t.s2 >= t.s1 - cand_delta(t.s1);
    if (close) {
        const bool pen1 = PENALTY ? wv.warp_has(j, t.i1) : false;
        const bool pen2 = PENALTY ? wv.warp_has(j, t.i2) : false;
        if (lane == 0) {
            double sc[2];
            for (int h = 0; h < 2; ++h) {
                const int id = h == 0 ? t.i1 : t.i2;
                const double z = transform_f64<SOFTCAP, PENALTY>(raw_logit_f64<BF16>(P.logits, row, P.V, id),
                                                                 h == 0 ? pen1 : pen2, P);
                if constexpr (GREEDY) {
                    sc[h] = z;
                } else {
                    sc[h] = z / P.Td - log(noise_exp_f64(nk, static_cast<uint32_t>(id), static_cast<uint32_t>(j)));
                }
            }
            if (better64(sc[1], t.i2, sc[0], t.i1)) winner = t.i2;
        }
        winner = __shfl_sync(0xffffffffu, winner, 0);
    }

    // accept test of d_{j+1}: fp32 unless within 1e-4 of the boundary, then fp64
    int accepted = 0;
    if (j < keff && dvalid) {
        if constexpr (GREEDY) {
            accepted = dnext == winner;
        } else {
            const bool pend = PENALTY ? wv.warp_has(j, dnext) : false;
            if (lane == 0) {
                const double u = accept_uniform_f64(nk, static_cast<uint32_t>(j + 1));
                const double q = dense ? static_cast<double>(qd) : 1.0;
                const float lp = transform_f32<SOFTCAP, PENALTY>(xd, pend, P) * P.invT - static_cast<float>(lse);
                const float lr = logf(static_cast<float>(u)) + logf(static_cast<float>(q));
                if (lr < lp - 1e-4f * (1.0f + fabsf(lp))) {
                    accepted = 1;
                } else if (lr > lp + 1e-4f * (1.0f + fabsf(lp))) {
                    accepted = 0;
                } else {
                    const double zd = transform_f64<SOFTCAP, PENALTY>(static_cast<double>(xd), pend, P);
                    accepted = u * q <= exp(zd / P.Td - lse);
                }
            }
            accepted = __shfl_sync(0xffffffffu, accepted, 0);
        }
    }

    int last_row = 0;
    if (lane == 0) {
        RowRes rr;
        rr.lse = lse;
        rr.winner = winner;
        rr.accepted = accepted;
        P.rowres[row] = rr;
        __threadfence();
        const unsigned prev = atomicAdd(&P.seq_ticket[b], 1u);
        last_row = prev == static_cast<unsigned>(keff);
    }
    last_row = __shfl_sync(0xffffffffu, last_row, 0);
    if (!last_row) return;
    __threadfence();

    // ---- last row of the sequence: epilogue
    if (lane == 0) P.seq_ticket[b] = 0u;
    RowRes* rs = P.rowres + static_cast<size_t>(b) * K1;
    int acc = 1;
    if (lane < keff) acc = __ldcg(&rs[lane].accepted);
    const unsigned rej = __ballot_sync(0xffffffffu, lane < keff && !acc);
    const int a = rej ? __ffs(rej) - 1 : keff;
    // a rejected draft outside [0, V) leaves the residual equal to p: the
    // row's own candidate (over all ids) is then the sample
    const int da = a < keff ? wv.drafts[a] : -1;
    const bool need = dense && !GREEDY && a < keff && da >= 0 && da < P.V;
    const int y = need ? -1 : __ldcg(&rs[a].winner);
    __syncwarp();
    if (lane <= keff && !(need && lane == a)) st_zero(rs + lane);
    if (lane < K1) P.out_tokens[static_cast<size_t>(b) * K1 + lane] = lane < a ? wv.drafts[lane] : (lane == a ? y : -1);
    if (lane == 0) {
        P.out_accept[b] = a;
        P.kv_len[b] = P.kv_len[b] - kb + a;
        if (keff > 0) {
            // (1 - tau) * ema + tau * a / k_eff, rounded step by step (no contraction)
            const double tau = static_cast<double>(P.tau);
            const double rate = static_cast<double>(a) / static_cast<double>(keff);
            P.ema[b] = static_cast<float>(
                __dadd_rn(__dmul_rn(1.0 - tau, static_cast<double>(P.ema[b])), __dmul_rn(tau, rate)));
        }
        if (need) {
            SeqRes sr;
            sr.a = a;
            sr.keff = keff;
            sr.need_residual = 1;
            sr.pad = 0;
            P.seqres[b] = sr;
        }
    }
}

// ---------------------------------------------------------------- K1
// Persistent, warp-specialised streaming kernel.  One CTA per SM; the active
// row-chunks of the call (rows 0..k_eff of every sequence, chunks of 64 KB)
// are laid out row-major and split into equal contiguous ranges, one per CTA.
//   * A producer warp walks the CTA's range and keeps up to kStages chunks in
//     flight with cp.async.bulk into a shared-memory ring (full / empty
//     mbarriers, bounded waits).  It draws the noise of a chunk's 256-id
//     blocks before the chunk's ring slot is free, and writes the row's
//     metadata, the penalty bitmap and the noise while the copy is in flight.
//   * Sixteen streaming warps each own a 4 KB slice of every chunk.  A lane's
//     16-byte vector i of a bf16 chunk covers 8 ids of noise block 8 w + i, so
//     its packed maximum gives the block test z / T - ln M >= best for its
//     eight ids at once; a single test of the lane's maximum against the
//     smallest ln M of the slice gates them.  Per slice: packed maxima, the
//     exponentials of the sum, the block tests; only the vectors that pass
//     compare their elements, and each lane scores its few survivors
//     (per-id Philox draw, E_v, score) in step with the warp.  At the first
//     chunk of a row segment each lane scores its largest element, which
//     starts the segment's best; the warps of the CTA share the best through
//     shared memory.
//   * A merge warp runs the row merges: the CTA that completes a row (atomic
//     ticket over the row's chunks) queues it, and the merge warp combines the
//     row's partials, takes the accept test and, for the last row of a
//     sequence (second ticket), runs the epilogue.  Nothing waits on another
//     CTA.

constexpr int kCWarps = 16;                    // streaming warps
constexpr int kPWarp = kCWarps;                // producer warp index
constexpr int kMWarp = kCWarps + 1;            // merge warp index
constexpr int kPThreads = (kCWarps + 2) * 32;  // 576
constexpr int kStages = 6;
constexpr int kVL = 4;                         // 16-byte vectors per lane per chunk
constexpr int kMaxBlk = kChunkBytes / 2 >> kNoiseBlockShift;  // noise blocks per chunk (bf16: 128)
constexpr int kMQ = 16;                        // merge-queue entries per streaming warp
static_assert(kChunkBytes == kCWarps * 32 * kVL * 16, "stage layout");
static_assert((32 * 8) == (1 << kNoiseBlockShift), "a bf16 vector row of a warp is one noise block");

template <bool PENALTY>
__host__ __device__ constexpr size_t k1_dyn_smem() {
    return static_cast<size_t>(kStages) * kChunkBytes +
           (PENALTY ? static_cast<size_t>(kStages) * (kChunkBytes / 2 / 8) : 0);
}

struct StageMeta {
    int b, j, c, excl, seg_end;  // seg_end: the last chunk of this row in the CTA's range
    int cand;                    // the row's Gumbel candidates can be the emitted token
    unsigned penw;               // bit w: warp w's slice holds a penalised id
    int pad;
    float wmin[kCWarps];         // smallest ln M of each warp's slice
    BlockNoise bn[kMaxBlk];      // noise of the chunk's 256-id blocks
};

struct WarpPart {
    float m, s;
    Top2 t;
};

template <bool BF16, bool GREEDY, bool SOFTCAP, bool PENALTY>
__global__ void __launch_bounds__(kPThreads, 1) verify_stream_kernel(const VerifyDev P) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    constexpr int CHUNK = chunk_elems<BF16>();
    constexpr int SB = kChunkBytes;
    constexpr int SL = 32 * kVL * EPV;  // ids per streaming slice
    constexpr int NB = CHUNK >> kNoiseBlockShift;
    constexpr int BPW = NB / kCWarps;   // noise blocks per slice
    extern __shared__ __align__(128) uint8_t s_dyn[];
    uint8_t* s_stage = s_dyn;
    uint32_t* s_bm = reinterpret_cast<uint32_t*>(s_dyn + kStages * SB);
    __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages];
    __shared__ StageMeta s_meta[kStages];
    __shared__ WarpPart s_slot[kStages][kCWarps];
    __shared__ int s_cnt[kStages];
    __shared__ unsigned s_rthr[kStages + 1];  // per-segment best score (score_key; 0 = none)
    __shared__ long long s_wsum[kPThreads / 32];
    __shared__ int s_start[3];
    __shared__ int s_hwin[PENALTY ? SPECNG_MAX_REP_WINDOW : 1];
    __shared__ int s_pdrafts[SPECNG_MAX_K + 1];
    __shared__ volatile int s_mq[kCWarps][kMQ];  // rows to merge, per streaming warp (single producer / consumer)
    __shared__ volatile int s_mq_tail[kCWarps];
    __shared__ volatile int s_mq_head[kCWarps];
    __shared__ int s_done;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K1 = P.K + 1;
    const bool dense = P.q != nullptr;

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
            s_cnt[i] = 0;
        }
        for (int i = 0; i <= kStages; ++i) s_rthr[i] = 0u;
        s_done = 0;
        mbar_init_fence();
    }
    if (tid < kCWarps) {
        s_mq_tail[tid] = 0;
        s_mq_head[tid] = 0;
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
        // The data of the next sequence (k, EMA, drafts, the tail of its history
        // for the penalty window) is fetched into registers one sequence ahead,
        // and its history length two ahead, so no global round trip stalls the
        // copies at a sequence change.
        constexpr int kHW = PENALTY ? SPECNG_MAX_REP_WINDOW / 32 : 1;
        struct SeqData {
            int k, draft, L;
            float ema;
            int hw[kHW];
        };
        auto clampL = [&](int L) {
            return L < 0 ? 0 : (static_cast<int64_t>(L) > P.hist_stride ? static_cast<int>(P.hist_stride) : L);
        };
        auto fetch = [&](int bq, int L, SeqData& d) {  // issues the loads; nothing waits here
            d.k = bq < P.B ? P.k[bq] : 0;
            d.ema = (P.gate && bq < P.B) ? P.ema[bq] : 1.0f;
            d.draft = (bq < P.B && lane < P.K) ? P.drafts[bq * P.K + lane] : -1;
            d.L = L;
            if constexpr (PENALTY) {
                const int nh = L < P.W ? L : P.W;
#pragma unroll
                for (int i = 0; i < kHW; ++i) {
                    const int t = lane + 32 * i;
                    d.hw[i] = (bq < P.B && t < nh) ? P.hist[static_cast<size_t>(bq) * P.hist_stride + (L - nh) + t] : 0;
                }
            }
        };
        int b = s_start[0], j = s_start[1], c = s_start[2];
        int kb = 0, keff = 0, nh = 0;
        auto install = [&](const SeqData& d) {
            kb = d.k;
            if (kb < 0 || kb > P.K) {
                if (lane == 0) raise_status(P.status, SPECNG_DEV_BAD_K);
                kb = kb < 0 ? 0 : P.K;
            }
            keff = (P.gate && kb > 0 && !(d.ema >= P.thresh)) ? 0 : kb;
            if (lane < keff) {
                s_pdrafts[lane] = d.draft;
                if (!(d.draft >= 0 && d.draft < P.V)) raise_status(P.status, SPECNG_DEV_TOKEN_OOR);
            }
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
            install(cur);
            fetch(b + 1, L1, nxt);
            if (PENALTY && b + 2 < P.B) Lnext2 = P.lens[b + 2];
        }
        NoiseKey nk = P.nk;
        bool ok = true;
        int st = 0;
        unsigned eph = 0u;  // parity of the empty barrier phase to wait for
        for (int n = 0; n < nwork && ok; ++n) {
            const int v0 = c * CHUNK;
            const int v1 = min(P.V, v0 + CHUNK);
            const char* src = static_cast<const char*>(P.logits) +
                              ((static_cast<size_t>(b) * K1 + j) * P.V + v0) * ElemTraits<BF16>::SIZE;
            // with dense q, row j < k_eff is sampled by the residual pass unless
            // its draft is invalid (the residual is then p itself)
            int excl = -1, cand = 1;
            if (!GREEDY && j < keff) {
                const int d = s_pdrafts[j];
                const bool valid = d >= 0 && d < P.V;
                if (!dense && valid) excl = d;
                if (dense && valid) cand = 0;
            }
            // the noise of the chunk's blocks (lane q: blocks q, q + 32, ...), before the
            // ring slot is free
            constexpr int NBL = (NB + 31) / 32;
            BlockNoise bnl[NBL];
            if (!GREEDY && cand) {
                nk.seq = static_cast<uint32_t>(b);
                const uint32_t blk0 = static_cast<uint32_t>(v0 >> kNoiseBlockShift);
#pragma unroll
                for (int r = 0; r < NBL; ++r)
                    if (lane + 32 * r < NB) bnl[r] = block_noise(nk, blk0 + lane + 32 * r, static_cast<uint32_t>(j));
            }
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
            StageMeta& mt = s_meta[st];
            if (lane == 0) {
                mt.b = b; mt.j = j; mt.c = c; mt.excl = excl;
                mt.seg_end = (c == P.nchunk - 1 || n == nwork - 1) ? 1 : 0;
                mt.cand = cand;
            }
            if (!GREEDY && cand) {
#pragma unroll
                for (int r = 0; r < NBL; ++r)
                    if (lane + 32 * r < NB) mt.bn[lane + 32 * r] = bnl[r];
                __syncwarp();
                if (lane < kCWarps) {
                    float mn = INFINITY;
#pragma unroll
                    for (int q = 0; q < BPW; ++q) mn = fminf(mn, mt.bn[lane * BPW + q].lnM);
                    mt.wmin[lane] = mn;
                }
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
                        install(nxt);
                        const int L2 = PENALTY ? clampL(Lnext2) : 0;
                        fetch(b + 1, L2, nxt);
                        if (PENALTY && b + 2 < P.B) Lnext2 = P.lens[b + 2];
                    }
                }
            }
        }
        // the CTA stays resident until every issued copy has landed
        if (P.aligned && lane == 0) {
            const int lo = nwork > kStages ? nwork - kStages : 0;
            for (int n = lo; n < nwork; ++n) mbar_wait_bounded(&s_full[n % kStages], static_cast<unsigned>((n / kStages) & 1));
        }
        return;
    }

    if (warp == kMWarp) {
        // ================= merge warp =================
        // Polls the streaming warps' queues (lane q watches queue q) until every
        // streaming warp has finished and every queue is drained.  The wait is bounded.
        unsigned idle = 0;
        while (true) {
            const bool has = lane < kCWarps && s_mq_head[lane] != s_mq_tail[lane];
            const unsigned qs = __ballot_sync(0xffffffffu, has);
            if (qs != 0u) {
                idle = 0;
                const int q = __ffs(qs) - 1;
                const int h = s_mq_head[q];
                const int row = s_mq[q][h % kMQ];
                __syncwarp();
                merge_row<BF16, GREEDY, SOFTCAP, PENALTY>(P, row);
                __syncwarp();
                if (lane == 0) s_mq_head[q] = h + 1;
                __syncwarp();
                continue;
            }
            if (*reinterpret_cast<volatile int*>(&s_done) == kCWarps) {
                // every push happened before its warp's increment of s_done
                __threadfence_block();
                const bool again = lane < kCWarps && s_mq_head[lane] != s_mq_tail[lane];
                if (!__any_sync(0xffffffffu, again)) break;
                continue;
            }
            if (++idle > (1u << 22)) {
                if (lane == 0) raise_status(P.status, SPECNG_DEV_TIMEOUT);
                break;
            }
            __nanosleep(idle < 64 ? 32 : 256);
        }
        return;
    }

    // ================= streaming warps =================
    // Per-lane accumulators live across the chunks of one row (a segment of
    // the CTA's range); warps combine them once, at the segment's last chunk.
    const int ubase = warp * (32 * kVL);        // first 16-byte vector of my slice
    const int off0 = ubase * EPV + lane * EPV;  // chunk offset of vector 0's element 0
    float thr = -INFINITY;
    float m = -INFINITY, s = 0.0f, msc = 0.0f;
    Top2 tt = top2_empty();
    int seg = 0, cfirst = 0;
    int row = 0, excl = -1;
    bool cand = false;
    RowPhilox rp{};
    bool fresh = true;
    int st = 0;
    unsigned fph = 0u;  // parity of the full barrier phase to wait for
    for (int n = 0; n < nwork; ++n) {
        if (!mbar_wait_bounded(&s_full[st], fph)) {
            if (lane == 0) raise_status(P.status, SPECNG_DEV_TIMEOUT);
            break;
        }
        const StageMeta& mt = s_meta[st];
        const int c = mt.c;
        unsigned* rth = &s_rthr[seg % (kStages + 1)];
        const bool seg_start = fresh;
        if (seg_start) {
            const int b = mt.b, j = mt.j;
            row = b * K1 + j;
            excl = mt.excl;
            cand = !GREEDY && mt.cand != 0;
            cfirst = c;
            if (cand) {
                NoiseKey nk = P.nk;
                nk.seq = static_cast<uint32_t>(b);
                rp = row_philox(nk, static_cast<uint32_t>(j));
            }
        }
        const int v0 = c * CHUNK;
        const int v1 = min(P.V, v0 + CHUNK);
        const uint4* stage = reinterpret_cast<const uint4*>(s_stage + st * SB);
        const uint32_t* bm = s_bm + (PENALTY ? st * (CHUNK / 32) : 0);
        const bool full = v0 + off0 + (kVL - 1) * 32 * EPV + EPV <= v1;  // my vectors are whole
        uint4 rv[kVL];
#pragma unroll
        for (int i = 0; i < kVL; ++i) rv[i] = stage[ubase + i * 32 + lane];
        // penalised elements of my lane (bit 8 i + e), only where the slice holds one
        uint64_t pmk = 0u;
        if constexpr (PENALTY) {
            if ((mt.penw >> warp) & 1u) {
#pragma unroll
                for (int i = 0; i < kVL; ++i) {
                    const int off = off0 + i * 32 * EPV;
                    pmk |= static_cast<uint64_t>((bm[off >> 5] >> (off & 31)) & ((1u << EPV) - 1u)) << (8 * i);
                }
            }
        }

        // ---- streaming: lane maximum zl (bounds my transformed values, penalised ones
        //      included), sum of exponentials
        float zl = -INFINITY;
        float lraw = -INFINITY;
        uint32_t hv[kVL];  // packed vector maxima (bf16), or the fp32 maxima
        if (full) {
            if constexpr (BF16) {
#pragma unroll
                for (int i = 0; i < kVL; ++i) hv[i] = as_u32(bf16x8_max2(rv[i]));
                uint32_t hr[kVL];
#pragma unroll
                for (int i = 0; i < kVL; ++i) hr[i] = hv[i];
#pragma unroll
                for (int w2 = kVL / 2; w2 > 0; w2 >>= 1)
#pragma unroll
                    for (int i = 0; i < w2; ++i) hr[i] = as_u32(__hmax2(as_bf162(hr[i]), as_bf162(hr[i + w2])));
                lraw = fmaxf(bf16lo(hr[0]), bf16hi(hr[0]));
            } else {
#pragma unroll
                for (int i = 0; i < kVL; ++i) {
                    const float f = fmaxf(fmaxf(__uint_as_float(rv[i].x), __uint_as_float(rv[i].y)),
                                          fmaxf(__uint_as_float(rv[i].z), __uint_as_float(rv[i].w)));
                    hv[i] = __float_as_uint(f);
                    lraw = fmaxf(lraw, f);
                }
            }
            zl = SOFTCAP ? transform_f32<true, false>(lraw, false, P) : lraw;
            if constexpr (GREEDY) {
                if (zl > m) m = zl;
            } else {
                // m is the segment's reference: fixed at its first value and raised only when a
                // value passes it by more than 2^32 in the sum's units, so the exponentials of a
                // chunk do not wait for the chunk's maximum
                if (!(m > -INFINITY)) {
                    m = zl;
                    msc = m * P.sc;
                }
                float2 acc2[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                                  make_float2(0.0f, 0.0f)};
                const float2 sc2 = make_float2(P.sc, P.sc), nm2 = make_float2(-msc, -msc);
#pragma unroll
                for (int i = 0; i < kVL; ++i) {
                    float x[EPV];
                    unpack<BF16>(rv[i], x);
#pragma unroll
                    for (int e = 0; e < EPV; e += 2) {
                        const float2 t = __ffma2_rn(make_float2(transform_f32<SOFTCAP, false>(x[e], false, P),
                                                                transform_f32<SOFTCAP, false>(x[e + 1], false, P)),
                                                    sc2, nm2);
                        acc2[i & 3] = __fadd2_rn(acc2[i & 3], make_float2(ex2_approx(t.x), ex2_approx(t.y)));
                    }
                }
                float add = ((acc2[0].x + acc2[0].y) + (acc2[1].x + acc2[1].y)) + ((acc2[2].x + acc2[2].y) + (acc2[3].x + acc2[3].y));
                if ((zl - m) * P.sc > 32.0f) {
                    // far above the reference: raise it and take the chunk again
                    s *= ex2_approx((m - zl) * P.sc);
                    m = zl;
                    msc = m * P.sc;
                    add = 0.0f;
#pragma unroll
                    for (int i = 0; i < kVL; ++i) {
                        float x[EPV];
                        unpack<BF16>(rv[i], x);
#pragma unroll
                        for (int e = 0; e < EPV; ++e)
                            add += ex2_approx(fmaf(transform_f32<SOFTCAP, false>(x[e], false, P), P.sc, -msc));
                    }
                }
                s += add;
            }
            if constexpr (PENALTY) {
                // the few penalised elements: replace their terms by the penalised ones (and
                // raise the maximum if a penalty below 1 lifted one above it)
                uint64_t pw = pmk;
                while (pw != 0u) {
                    const int bit = __ffsll(static_cast<long long>(pw)) - 1;
                    pw &= pw - 1u;
                    const float xe = elem_of_stage<BF16>(stage, off0 + (bit >> 3) * 32 * EPV + (bit & 7));
                    const float zu = transform_f32<SOFTCAP, false>(xe, false, P);
                    const float zp = transform_f32<SOFTCAP, true>(xe, true, P);
                    zl = fmaxf(zl, zp);
                    if constexpr (GREEDY) {
                        m = fmaxf(m, zp);
                    } else {
                        if ((zp - m) * P.sc > 32.0f) {
                            s *= ex2_approx((m - zp) * P.sc);
                            m = zp;
                            msc = m * P.sc;
                        }
                        s += ex2_approx(fmaf(zp, P.sc, -msc)) - ex2_approx(fmaf(zu, P.sc, -msc));
                    }
                }
            }
        } else {
            // partial vectors (a row's last chunk): exact transform element by element
#pragma unroll
            for (int i = 0; i < kVL; ++i) {
                hv[i] = BF16 ? 0xFF80FF80u : __float_as_uint(-INFINITY);
                const int off = off0 + i * 32 * EPV;
                const int nv = min(EPV, v1 - (v0 + off));
                if (nv <= 0) continue;
                float x[EPV];
                unpack<BF16>(rv[i], x);
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    if (e >= nv) break;
                    const float z = transform_f32<SOFTCAP, PENALTY>(x[e], (pmk >> (8 * i + e)) & 1u, P);
                    lraw = fmaxf(lraw, x[e]);
                    zl = fmaxf(zl, z);
                    if constexpr (GREEDY) {
                        m = fmaxf(m, z);
                    } else {
                        if (!(m > -INFINITY) || (z - m) * P.sc > 32.0f) {
                            s = m > -INFINITY ? s * ex2_approx((m - z) * P.sc) : 0.0f;
                            m = z;
                            msc = m * P.sc;
                        }
                        s += ex2_approx(fmaf(z, P.sc, -msc));
                    }
                }
            }
        }

        // ---- candidates
        if constexpr (GREEDY) {
            // top two transformed values (lower id on ties) within cand_delta of the best
            // value any warp of the CTA has reached in this segment.  Without a penalty the
            // lane maximum is itself a value of the row (the transform is monotone)
            float gth = fmaxf(tt.s1, key_score(*reinterpret_cast<volatile unsigned*>(rth)));
            if constexpr (!PENALTY) gth = fmaxf(gth, key_score(warp_best_key(zl)));
            gth = gth > -INFINITY ? gth - cand_delta(gth) : -INFINITY;
            if (zl >= gth) {
#pragma unroll
                for (int i = 0; i < kVL; ++i) {
                    const int off = off0 + i * 32 * EPV;
                    const int nv = min(EPV, v1 - (v0 + off));
                    if (nv <= 0) continue;
                    float x[EPV];
                    unpack<BF16>(rv[i], x);
#pragma unroll
                    for (int e = 0; e < EPV; ++e) {
                        if (e >= nv) break;
                        const float z = transform_f32<SOFTCAP, PENALTY>(x[e], (pmk >> (8 * i + e)) & 1u, P);
                        if (z >= gth) {
                            top2_push(tt, z, v0 + off + e);
                            gth = fmaxf(gth, tt.s1 - cand_delta(tt.s1));
                        }
                    }
                }
            }
            const unsigned kw = warp_best_key(tt.s1);
            if (lane == 0 && kw != 0u) atomicMax(rth, kw);
        } else if (cand) {
            int seeded = -1;
            if (seg_start) {
                // seed: every lane scores its largest raw element (any exact score bounds the
                // best from below); the CTA's warps share the best seed
                int am = -1;
#pragma unroll
                for (int i = kVL - 1; i >= 0; --i) {
                    const int off = off0 + i * 32 * EPV;
                    const int nv = min(EPV, v1 - (v0 + off));
                    float x[EPV];
                    unpack<BF16>(rv[i], x);
#pragma unroll
                    for (int e = EPV - 1; e >= 0; --e)
                        if (e < nv && x[e] == lraw) am = off + e;
                }
                float t0 = -INFINITY;
                if (am >= 0 && v0 + am != excl) {
                    const float z = transform_f32<SOFTCAP, PENALTY>(elem_of_stage<BF16>(stage, am),
                                                                    PENALTY && ((bm[am >> 5] >> (am & 31)) & 1u), P);
                    const uint32_t v = static_cast<uint32_t>(v0 + am);
                    const BlockNoise bk = mt.bn[am >> kNoiseBlockShift];
                    t0 = z * P.invT - ln_fast(noise_exp_f32(rp, bk.M, bk.I, v));
                    top2_push(tt, t0, static_cast<int>(v));
                    seeded = static_cast<int>(v);
                }
                const unsigned k0 = warp_best_key(t0);
                if (k0 != 0u) {
                    const float b0 = key_score(k0);
                    thr = fmaxf(thr, b0 - cand_delta(b0));
                    if (lane == 0) atomicMax(rth, k0);
                }
            }
            {
                // adopt the best score another warp published for this segment
                const float best = key_score(*reinterpret_cast<volatile unsigned*>(rth));
                if (best > -INFINITY) thr = fmaxf(thr, best - cand_delta(best));
            }
            // gate: no score of my lane exceeds zl / T - (smallest ln M of the slice)
            const float zlb = zl * P.invT;
            const bool lpass = zlb - mt.wmin[warp] + bound_slack(zlb) >= thr;
            if (__any_sync(0xffffffffu, lpass)) {
                // block tests: every score of vector i is at most z / T - ln M_i; then the
                // elements of the passing vectors that can reach the best
                uint64_t msk = 0u;
                if (lpass) {
#pragma unroll
                    for (int i = 0; i < kVL; ++i) {
                        const int off = off0 + i * 32 * EPV;
                        const float lnM = mt.bn[off >> kNoiseBlockShift].lnM;
                        float zv;
                        if constexpr (BF16) zv = fmaxf(bf16lo(hv[i]), bf16hi(hv[i]));
                        else zv = __uint_as_float(hv[i]);
                        if (SOFTCAP && full) zv = transform_f32<true, false>(zv, false, P);
                        const unsigned pb = static_cast<unsigned>(pmk >> (8 * i)) & 0xFFu;
                        const float zvb = zv * P.invT;
                        if (!(pb != 0u || !full || zvb - lnM + bound_slack(zvb) >= thr)) continue;
                        unsigned mi;
                        if (full) {
                            // z >= T (thr + ln M), in raw units
                            const float zt = (thr + lnM) * P.T;
                            float xt = zt;
                            if constexpr (SOFTCAP) {
                                // shrink by more than the fp32 error of c tanh(x / c) before
                                // inverting: atanh is steep near |u| = 1
                                float u = zt * P.invcap;
                                u -= 1e-6f * fabsf(u) + 1e-7f;
                                xt = u > 1.0f ? INFINITY : (u <= -1.0f ? -INFINITY : P.cap * atanhf(fminf(u, 1.0f - 1e-7f)));
                            }
                            xt -= 1e-5f * (1.0f + fabsf(xt));  // slack for the rounding of the transform
                            if constexpr (BF16) {
                                mi = bf16x8_ge_bits(rv[i], bf16x2_floor(xt));
                            } else {
                                mi = static_cast<unsigned>(__uint_as_float(rv[i].x) >= xt);
                                mi |= static_cast<unsigned>(__uint_as_float(rv[i].y) >= xt) << 1;
                                mi |= static_cast<unsigned>(__uint_as_float(rv[i].z) >= xt) << 2;
                                mi |= static_cast<unsigned>(__uint_as_float(rv[i].w) >= xt) << 3;
                            }
                            mi |= pb;  // penalised: decided exactly below
                        } else {
                            const int nv = min(EPV, v1 - (v0 + off));
                            mi = nv > 0 ? (1u << nv) - 1u : 0u;
                        }
                        msk |= static_cast<uint64_t>(mi) << (8 * i);
                    }
                    if (seeded >= 0) {
                        const int so = seeded - v0 - off0;
                        const int si = so / (32 * EPV), se = so - si * 32 * EPV;
                        if (se >= 0 && se < EPV) msk &= ~(static_cast<uint64_t>(1) << (8 * si + se));
                    }
                }
                // score the lane's candidates one per iteration, the warp in step
                while (__any_sync(0xffffffffu, msk != 0u)) {
                    int v = -1, loc = 0;
                    float zb = -INFINITY;
                    if (msk != 0u) {
                        const int bit = __ffsll(static_cast<long long>(msk)) - 1;
                        msk &= msk - 1u;
                        loc = off0 + (bit >> 3) * 32 * EPV + (bit & 7);
                        const bool pen = PENALTY && ((pmk >> bit) & 1u);
                        zb = transform_f32<SOFTCAP, PENALTY>(elem_of_stage<BF16>(stage, loc), pen, P) * P.invT;
                        v = v0 + loc;
                    }
                    const BlockNoise bk = mt.bn[loc >> kNoiseBlockShift];
                    const bool live = v >= 0 && v != excl && zb - bk.lnM + bound_slack(zb) >= thr;
                    if (__any_sync(0xffffffffu, live)) {
                        const float E = noise_exp_f32(rp, bk.M, bk.I, static_cast<uint32_t>(v < 0 ? 0 : v));
                        if (live) {
                            const float score = zb - ln_fast(E);
                            if (score >= thr) {
                                top2_push(tt, score, v);
                                thr = fmaxf(thr, tt.s1 - cand_delta(tt.s1));
                            }
                        }
                    }
                }
                // share the warp's best score with the CTA
                const unsigned kw = warp_best_key(tt.s1);
                if (kw != 0u) {
                    const float bw = key_score(kw);
                    thr = fmaxf(thr, bw - cand_delta(bw));
                    if (lane == 0) atomicMax(rth, kw);
                }
            }
        }

        fresh = mt.seg_end != 0;
        if (fresh) {
            // ---- end of this row's segment: one partial for the segment
            float pm = m, ps = s;
            Top2 pt = tt;
            if constexpr (!GREEDY) {
                if (!(pm > -INFINITY)) ps = 0.0f;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float mo = __shfl_xor_sync(0xffffffffu, pm, off);
                    const float so = __shfl_xor_sync(0xffffffffu, ps, off);
                    ms_merge(pm, ps, mo, so, P.sc);
                }
            }
            pt = top2_warp_reduce(pt);
            int last = 0;
            if (lane == 0) {
                s_slot[st][warp] = WarpPart{pm, ps, pt};
                __threadfence_block();
                last = atomicAdd(&s_cnt[st], 1) == kCWarps - 1;
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence_block();
                WarpPart wp = lane < kCWarps ? s_slot[st][lane] : WarpPart{-INFINITY, 0.0f, top2_empty()};
                float cm = wp.m, cs = wp.s;
                Top2 ct = wp.t;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float mo = __shfl_xor_sync(0xffffffffu, cm, off);
                    const float so = __shfl_xor_sync(0xffffffffu, cs, off);
                    ms_merge(cm, cs, mo, so, P.sc);
                    ct = top2_merge(ct, top2_shfl_xor(ct, off));
                }
                int merge_now = 0;
                if (lane == 0) {
                    // keyed by the segment's last chunk; a written partial is never all-zero
                    st_partial(P.part + static_cast<size_t>(row) * P.nchunk + c, GREEDY ? 0.0f : cm,
                               GREEDY ? 1.0f : cs, ct);
                    s_cnt[st] = 0;
                    *rth = 0u;  // every warp is past this segment: the slot is free
                    // the CTA that completes the row's chunks merges it
                    __threadfence();
                    const unsigned nseg = static_cast<unsigned>(c - cfirst + 1);
                    const unsigned prev = atomicAdd(&P.row_ticket[row], nseg);
                    if (prev + nseg == static_cast<unsigned>(P.nchunk)) {
                        __threadfence();
                        const int tl = s_mq_tail[warp];
                        if (tl - s_mq_head[warp] < kMQ) {
                            s_mq[warp][tl % kMQ] = row;
                            __threadfence_block();
                            s_mq_tail[warp] = tl + 1;
                        } else {
                            merge_now = 1;  // queue full: merge here
                        }
                    }
                }
                merge_now = __shfl_sync(0xffffffffu, merge_now, 0);
                if (merge_now) merge_row<BF16, GREEDY, SOFTCAP, PENALTY>(P, row);
            }
            m = -INFINITY;
            s = 0.0f;
            msc = 0.0f;
            tt = top2_empty();
            thr = -INFINITY;
            ++seg;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[st]);
        if (++st == kStages) {
            st = 0;
            fph ^= 1u;
        }
    }
    __syncwarp();
    if (lane == 0) {
        __threadfence_block();
        atomicAdd(&s_done, 1);
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
        tok = idx < L ? P.hist[static_cast<size_t>(b) * P.hist_stride + idx] : P.drafts[b * P.K + (idx - L)];
        s_win[tid] = tok;
    }
    if (tid == 0) *s_nwin = nw;
    __syncthreads();
    if (tok >= v0 && tok < v1) atomicOr(&s_bm[(tok - v0) >> 5], 1u << ((tok - v0) & 31));
    __syncthreads();
}

template <bool BF16, bool SOFTCAP, bool PENALTY>
__global__ void __launch_bounds__(kThreads, 2) verify_residual_kernel(const VerifyDev P) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    constexpr int CHUNK = res_chunk_elems<BF16>();
    constexpr int NB = CHUNK >> kNoiseBlockShift;
    __shared__ uint32_t s_bm[PENALTY ? CHUNK / 32 : 1];
    __shared__ int s_win[PENALTY ? SPECNG_MAX_REP_WINDOW : 1];
    __shared__ int s_nwin;
    __shared__ Top2 s_t[kWarps];
    __shared__ int s_last;
    __shared__ unsigned s_thr;
    __shared__ BlockNoise s_bn[NB];
    __shared__ uint16_t s_q2[kWarps * 32 * kNV * EPV];  // per-warp candidate queues (chunk offsets)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K1 = P.K + 1;
    const int b = blockIdx.x / P.nchunk2;
    const int c = blockIdx.x - b * P.nchunk2;
    const int need = __ldcg(&P.seqres[b].need_residual);
    if (!need) return;
    const int a = __ldcg(&P.seqres[b].a);
    const int row = b * K1 + a;
    const double lse = __ldcg(&P.rowres[row].lse);
    const float lse_f = static_cast<float>(lse);
    const int v0 = c * CHUNK;
    const int v1 = min(P.V, v0 + CHUNK);
    const char* rowp = static_cast<const char*>(P.logits) +
                       static_cast<size_t>(row) * P.V * ElemTraits<BF16>::SIZE;
    const float* qrow = P.q + (static_cast<size_t>(b) * P.K + a) * P.V;
    NoiseKey nk = P.nk;
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
        rv[i] = e0 < v1 ? load_vec<BF16>(rowp, e0, v1, P.aligned) : make_uint4(0u, 0u, 0u, 0u);
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
        const float x = in ? static_cast<float>(raw_logit_f64<BF16>(P.logits, row, P.V, v)) : 0.0f;
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
    if (!s_last || warp != 0) return;
    __threadfence();
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
    if (lane != 0) return;
    const int bonus = __ldcg(&P.rowres[row].winner);
    st_zero(P.rowres + row);
    st_zero(P.seqres + b);
    double best = -INFINITY;
    int winner = -1;
    for (int h = 0; h < 2; ++h) {
        const int id = h == 0 ? t.i1 : t.i2;
        if (id < 0) continue;
        if (h == 1 && !(t.s2 >= t.s1 - cand_delta(t.s1))) continue;
        const double z = transform_f64<SOFTCAP, PENALTY>(raw_logit_f64<BF16>(P.logits, row, P.V, id), h == 0 ? pen1 : pen2, P);
        const double rsd = exp(z / P.Td - lse) - static_cast<double>(qrow[id]);
        if (!(rsd > 0.0)) continue;
        const double score = log(rsd) - log(noise_exp_f64(nk, static_cast<uint32_t>(id), static_cast<uint32_t>(a)));
        if (winner < 0 || better64(score, id, best, winner)) { best = score; winner = id; }
    }
    // all-zero residual (p <= q everywhere): sample from p, the row's bonus candidate
    if (winner < 0) winner = bonus;
    P.out_tokens[static_cast<size_t>(b) * K1 + a] = winner;
}

// ---------------------------------------------------------------- launch

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
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(verify_stream_kernel<BF16, G, C, R>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    verify_stream_kernel<BF16, G, C, R><<<sm_count_cached(), kPThreads, smem, s>>>(P);
    return cudaGetLastError();
}

template <bool BF16, bool C, bool R>
cudaError_t launch_residual(const VerifyDev& P, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>(P.B) * static_cast<unsigned>(P.nchunk2);
    verify_residual_kernel<BF16, C, R><<<grid, kThreads, 0, s>>>(P);
    return cudaGetLastError();
}

template <bool BF16, bool G>
cudaError_t launch_stream_cr(const VerifyDev& P, bool c, bool r, cudaStream_t s) {
    if (c) return r ? launch_stream<BF16, G, true, true>(P, s) : launch_stream<BF16, G, true, false>(P, s);
    return r ? launch_stream<BF16, G, false, true>(P, s) : launch_stream<BF16, G, false, false>(P, s);
}

// The kernels of one spec_verify call for one logits dtype: the streaming
// kernel (with the merges), then, for dense q at T > 0, the residual pass.
template <bool BF16>
cudaError_t launch_verify_dtype(const VerifyDev& P, bool greedy, bool softcap, bool penalty, bool dense,
                                cudaStream_t s);

template <bool BF16>
cudaError_t launch_verify_impl(const VerifyDev& P, bool greedy, bool softcap, bool penalty, bool dense,
                               cudaStream_t s) {
    cudaError_t e = greedy ? launch_stream_cr<BF16, true>(P, softcap, penalty, s)
                           : launch_stream_cr<BF16, false>(P, softcap, penalty, s);
    if (e != cudaSuccess || !dense || greedy) return e;
    if (softcap) return penalty ? launch_residual<BF16, true, true>(P, s) : launch_residual<BF16, true, false>(P, s);
    return penalty ? launch_residual<BF16, false, true>(P, s) : launch_residual<BF16, false, false>(P, s);
}

}  // namespace specng
