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
constexpr int kChunkBytes = 65536;
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
// One warp per piece of a row.  The active rows of the call (rows 0..k_eff of
// every sequence) are cut into pieces of 16 KB; each warp reads its piece from
// HBM once and leaves one partial (maximum, sum of exponentials, top-two
// sampling candidates).  The warp that finishes a row's last piece (atomic
// ticket) merges the row at once; the last row of a sequence (second ticket)
// runs the epilogue.  Warps never wait on each other.
//
// Sampling in two phases per warp.  A piece holds 32 noise blocks of 256 ids
// (bf16; 16 for fp32); lane q draws block q's minimum M_q and its slot I_q.
//   A  streams the piece with 16-byte loads (the next iteration's in flight):
//      sum of exponentials, and the maximum of every 16-byte vector, kept in
//      registers as bf16 (rounded up for fp32 data).  Meanwhile each block's
//      argmin element is loaded: its score z / T - ln M_q is exact without a
//      per-id draw.  After the stream the lanes holding the warp's four largest
//      values score them.  The best of these exact scores is published to the
//      row's shared best (global atomic maximum) and read back.
//   B  every score of a vector is at most (its maximum) / T - ln M of its block,
//      so the vector maxima in registers are tested against the best without
//      touching the data; the few vectors that pass are reloaded (from L2) and
//      their surviving elements scored (per-id Philox draw, E_v = M + F_v).

constexpr int kPieceBytes = 16384;
constexpr int kPW = 8;           // warps per CTA
constexpr int kPT = kPW * 32;    // threads per CTA
constexpr int kIV = 4;           // 16-byte vectors per lane per iteration
constexpr int kTop = 4;          // largest values scored after phase A

template <bool BF16>
__host__ __device__ constexpr int piece_elems() { return kPieceBytes / ElemTraits<BF16>::SIZE; }

// Smallest bf16 value >= f (an upper bound in bf16), as the low 16 bits.
__device__ __forceinline__ uint32_t bf16_ceil_bits(float f) {
    const uint32_t u = __float_as_uint(f);
    uint32_t h = u >> 16;
    if ((u & 0xFFFFu) != 0u && !(u & 0x80000000u) && (u & 0x7FFFFFFFu) < 0x7F800000u) h += 1u;  // positive: up
    return h;
}

template <bool BF16, bool GREEDY, bool SOFTCAP, bool PENALTY>
__global__ void __launch_bounds__(kPT, 2) verify_piece_kernel(const VerifyDev P) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    constexpr int PIECE = piece_elems<BF16>();
    constexpr int RV = 32 * EPV;                  // ids per vector row of the warp
    constexpr int NIT = PIECE / (kIV * RV);       // iterations per piece (8)
    constexpr int NV = NIT * kIV;                 // vectors per lane per piece (32)
    constexpr int NBP = PIECE >> kNoiseBlockShift;  // noise blocks per piece (bf16 32, fp32 16)
    static_assert(NIT * kIV * RV == PIECE && NBP <= 32 && NV == 32, "piece layout");
    __shared__ uint32_t s_pbm[PENALTY ? kPW * (PIECE / 32) : 1];  // per-warp penalty bitmap of the piece

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int K1 = P.K + 1;
    const long long item = static_cast<long long>(blockIdx.x) * kPW + warp;
    const int row = static_cast<int>(item / P.nchunk);
    const int p = static_cast<int>(item - static_cast<long long>(row) * P.nchunk);
    if (row >= P.B * K1) return;
    const int b = row / K1, j = row - b * K1;
    int kb;
    const int keff = gate_keff(P, b, &kb, j == 0 && p == 0);
    if (j > keff) return;
    const bool dense = P.q != nullptr;
    const int v0 = p * PIECE;
    const int v1 = min(P.V, v0 + PIECE);
    const char* rowp = static_cast<const char*>(P.logits) + static_cast<size_t>(row) * P.V * ElemTraits<BF16>::SIZE;

    // the draft this row verifies: excluded from the point-mass residual; with dense q
    // the residual pass samples the row (unless the draft is invalid: the residual is p)
    int excl = -1;
    bool cand = !GREEDY;
    if (!GREEDY && j < keff) {
        const int d = P.drafts[b * P.K + j];
        const bool valid = d >= 0 && d < P.V;
        if (!valid && p == 0 && lane == 0) raise_status(P.status, SPECNG_DEV_TOKEN_OOR);
        if (!dense && valid) excl = d;
        if (dense && valid) cand = false;
    }
    NoiseKey nk = P.nk;
    nk.seq = static_cast<uint32_t>(b);

    // the first iteration's loads go out before anything else
    const int ebase = v0 + lane * EPV;  // id of element 0 of my vector 0
    auto load_it = [&](int it, uint4* dst) {
#pragma unroll
        for (int i = 0; i < kIV; ++i) {
            const int e0 = ebase + (it * kIV + i) * RV;
            dst[i] = e0 < v1 ? load_vec<BF16>(rowp, e0, v1, P.aligned) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    uint4 rv[kIV], rn[kIV];
    load_it(0, rn);

    // noise of block q (lane q) and its argmin element, loaded now and scored after phase A
    BlockNoise bn{};
    RowPhilox rp{};
    float xI = 0.0f;
    int vI = -1;
    if (cand) {
        if (lane < NBP) {
            bn = block_noise(nk, static_cast<uint32_t>((v0 >> kNoiseBlockShift) + lane), static_cast<uint32_t>(j));
            vI = v0 + (lane << kNoiseBlockShift) + bn.I;
            if (vI < v1) xI = static_cast<float>(raw_logit_f64<BF16>(P.logits, row, P.V, vI));
            else vI = -1;
        }
        rp = row_philox(nk, static_cast<uint32_t>(j));
    }
    // penalty window of row j: the last W tokens of history ++ d_1..d_j, as a bitmap of the piece
    uint32_t* pbm = s_pbm + (PENALTY ? warp * (PIECE / 32) : 0);
    bool anypen = false;
    if constexpr (PENALTY) {
        for (int t = lane; t < PIECE / 32; t += 32) pbm[t] = 0u;
        int L = P.lens[b];
        L = L < 0 ? 0 : (static_cast<int64_t>(L) > P.hist_stride ? static_cast<int>(P.hist_stride) : L);
        const int total = L + j;
        const int nw = total < P.W ? total : P.W;
        __syncwarp();
        bool mine = false;
        for (int t = lane; t < nw; t += 32) {
            const int idx = total - nw + t;
            const int tok = idx < L ? P.hist[static_cast<size_t>(b) * P.hist_stride + idx] : P.drafts[b * P.K + (idx - L)];
            if (tok >= v0 && tok < v1) {
                atomicOr(&pbm[(tok - v0) >> 5], 1u << ((tok - v0) & 31));
                mine = true;
            }
        }
        anypen = __any_sync(0xffffffffu, mine);
        __syncwarp();
    }
    auto pen_at = [&](int v) -> bool {  // is id v (inside the piece) penalised?
        if constexpr (PENALTY) {
            const int o = v - v0;
            return anypen && ((pbm[o >> 5] >> (o & 31)) & 1u);
        }
        return false;
    };

    float mref = -INFINITY, s = 0.0f, m = -INFINITY;
    Top2 tt = top2_empty();
    float gth = -INFINITY;         // greedy: the best value so far, less the tie margin
    uint32_t vmx[NV / 2];          // phase A: bf16 maxima of my vectors, two per register
    unsigned penv = 0u;            // my vectors that hold a penalised element
    float lbest = -INFINITY;       // my largest raw value and the vector holding it
    int lbk = -1;

    // ================= phase A =================
#pragma unroll 1
    for (int it = 0; it < NIT; ++it) {
#pragma unroll
        for (int i = 0; i < kIV; ++i) rv[i] = rn[i];
        if (it + 1 < NIT) load_it(it + 1, rn);
        const int ib = ebase + it * kIV * RV;
        const bool full = ib + (kIV - 1) * RV + EPV <= v1;
        unsigned pmk = 0u;  // penalised elements of this iteration (bit 8 i + e)
        if constexpr (PENALTY) {
            if (anypen) {
#pragma unroll
                for (int i = 0; i < kIV; ++i) {
                    const int off = ib + i * RV - v0;
                    if (off < PIECE) pmk |= ((pbm[off >> 5] >> (off & 31)) & ((1u << EPV) - 1u)) << (8 * i);
                }
            }
        }
        float vm[kIV];
        float zl = -INFINITY;
        if (full) {
#pragma unroll
            for (int i = 0; i < kIV; ++i) {
                if constexpr (BF16) {
                    const uint32_t h = as_u32(bf16x8_max2(rv[i]));
                    vm[i] = fmaxf(bf16lo(h), bf16hi(h));
                } else {
                    vm[i] = fmaxf(fmaxf(__uint_as_float(rv[i].x), __uint_as_float(rv[i].y)),
                                  fmaxf(__uint_as_float(rv[i].z), __uint_as_float(rv[i].w)));
                }
            }
            const float lraw = fmaxf(fmaxf(vm[0], vm[1]), fmaxf(vm[2], vm[3]));
            zl = SOFTCAP ? transform_f32<true, false>(lraw, false, P) : lraw;
            if constexpr (!GREEDY) {
                if (!(mref > -INFINITY)) mref = zl;
                const float msc = mref * P.sc;
                float2 acc2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
                const float2 sc2 = make_float2(P.sc, P.sc), nm2 = make_float2(-msc, -msc);
#pragma unroll
                for (int i = 0; i < kIV; ++i) {
                    float x[EPV];
                    unpack<BF16>(rv[i], x);
#pragma unroll
                    for (int e = 0; e < EPV; e += 2) {
                        const float2 t = __ffma2_rn(make_float2(transform_f32<SOFTCAP, false>(x[e], false, P),
                                                                transform_f32<SOFTCAP, false>(x[e + 1], false, P)),
                                                    sc2, nm2);
                        acc2[i & 1] = __fadd2_rn(acc2[i & 1], make_float2(ex2_approx(t.x), ex2_approx(t.y)));
                    }
                }
                float add = (acc2[0].x + acc2[0].y) + (acc2[1].x + acc2[1].y);
                if ((zl - mref) * P.sc > 32.0f) {
                    // a value far above the reference: raise it and take the iteration again
                    s *= ex2_approx((mref - zl) * P.sc);
                    mref = zl;
                    const float msc2 = mref * P.sc;
                    add = 0.0f;
#pragma unroll
                    for (int i = 0; i < kIV; ++i) {
                        float x[EPV];
                        unpack<BF16>(rv[i], x);
#pragma unroll
                        for (int e = 0; e < EPV; ++e)
                            add += ex2_approx(fmaf(transform_f32<SOFTCAP, false>(x[e], false, P), P.sc, -msc2));
                    }
                }
                s += add;
            }
            if constexpr (PENALTY) {
                // the few penalised elements: replace their terms by the penalised ones
                unsigned pw = pmk;
                while (pw != 0u) {
                    const int bit = __ffs(pw) - 1;
                    pw &= pw - 1u;
                    const float xe = static_cast<float>(raw_logit_f64<BF16>(P.logits, row, P.V, ib + (bit >> 3) * RV + (bit & 7)));
                    const float zu = transform_f32<SOFTCAP, false>(xe, false, P);
                    const float zp = transform_f32<SOFTCAP, true>(xe, true, P);
                    zl = fmaxf(zl, zp);
                    if constexpr (!GREEDY) {
                        if ((zp - mref) * P.sc > 32.0f) {
                            s *= ex2_approx((mref - zp) * P.sc);
                            mref = zp;
                        }
                        const float msc = mref * P.sc;
                        s += ex2_approx(fmaf(zp, P.sc, -msc)) - ex2_approx(fmaf(zu, P.sc, -msc));
                    }
                }
            }
        } else {
            // partial vectors (a row's last piece): exact transform element by element
#pragma unroll
            for (int i = 0; i < kIV; ++i) {
                vm[i] = -INFINITY;
                const int e0 = ib + i * RV;
                const int nv = min(EPV, v1 - e0);
                if (nv <= 0) continue;
                float x[EPV];
                unpack<BF16>(rv[i], x);
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    if (e >= nv) break;
                    const float z = transform_f32<SOFTCAP, PENALTY>(x[e], (pmk >> (8 * i + e)) & 1u, P);
                    vm[i] = fmaxf(vm[i], x[e]);
                    zl = fmaxf(zl, z);
                    if constexpr (!GREEDY) {
                        if (!(mref > -INFINITY) || (z - mref) * P.sc > 32.0f) {
                            s = mref > -INFINITY ? s * ex2_approx((mref - z) * P.sc) : 0.0f;
                            mref = z;
                        }
                        s += ex2_approx(fmaf(z, P.sc, -mref * P.sc));
                    }
                }
            }
        }
        m = fmaxf(m, zl);
        // bookkeeping of the vectors for phase B: bf16 upper bounds of the raw maxima,
        // the vectors with a penalised element, my largest value and its vector
#pragma unroll
        for (int i = 0; i < kIV; i += 2) {
            const uint32_t lo = BF16 ? (__float_as_uint(vm[i]) >> 16) : bf16_ceil_bits(vm[i]);
            const uint32_t hi = BF16 ? (__float_as_uint(vm[i + 1]) >> 16) : bf16_ceil_bits(vm[i + 1]);
            vmx[(it * kIV + i) >> 1] = lo | (hi << 16);
        }
#pragma unroll
        for (int i = 0; i < kIV; ++i) {
            if ((pmk >> (8 * i)) & 0xFFu) penv |= 1u << (it * kIV + i);
            if (vm[i] > lbest) {
                lbest = vm[i];
                lbk = it * kIV + i;
            }
        }
        if constexpr (GREEDY) {
            // top two transformed values (lower id on ties) within cand_delta of the best
            // value seen; without a penalty the lane maximum is itself a value of the row
            float g = fmaxf(gth, tt.s1 > -INFINITY ? tt.s1 - cand_delta(tt.s1) : -INFINITY);
            if constexpr (!PENALTY) {
                const float wb = key_score(warp_best_key(zl));
                if (wb > -INFINITY) g = fmaxf(g, wb - cand_delta(wb));
            }
            gth = g;
            if (zl >= gth) {
#pragma unroll
                for (int i = 0; i < kIV; ++i) {
                    const int e0 = ib + i * RV;
                    const int nv = min(EPV, v1 - e0);
                    if (nv <= 0) continue;
                    float x[EPV];
                    unpack<BF16>(rv[i], x);
#pragma unroll
                    for (int e = 0; e < EPV; ++e) {
                        if (e >= nv) break;
                        const float z = transform_f32<SOFTCAP, PENALTY>(x[e], (pmk >> (8 * i + e)) & 1u, P);
                        if (z >= gth) {
                            top2_push(tt, z, e0 + e);
                            gth = fmaxf(gth, tt.s1 - cand_delta(tt.s1));
                        }
                    }
                }
            }
        }
    }

    if (!GREEDY && cand) {
        // ---- exact scores that need no per-id draw: each block's argmin element
        if (vI >= 0 && vI != excl) {
            const float zb = transform_f32<SOFTCAP, PENALTY>(xI, pen_at(vI), P) * P.invT;
            top2_push(tt, zb - bn.lnM, vI);
        }
        // ---- the warp's four largest values (their lanes score them)
        int sv = -1;  // the id this lane scored
        {
            unsigned ku = lbest > -INFINITY ? score_key(lbest) : 0u;
            bool pick = false;
#pragma unroll
            for (int r = 0; r < kTop; ++r) {
                const unsigned kmax = __reduce_max_sync(0xffffffffu, ku);
                if (kmax == 0u) break;
                const unsigned own = __ballot_sync(0xffffffffu, ku == kmax);
                if (lane == __ffs(own) - 1) {
                    pick = true;
                    ku = 0u;
                }
            }
            int q = 0;
            float M = 0.0f;
            int I = 0;
            if (pick) {
                // locate the value in its vector (lowest id among equal values), then score it
                const int e0 = ebase + lbk * RV;
                const uint4 r = load_vec<BF16>(rowp, e0, v1, P.aligned);
                float x[EPV];
                unpack<BF16>(r, x);
                int e = -1;
#pragma unroll
                for (int k = EPV - 1; k >= 0; --k)
                    if (e0 + k < v1 && x[k] == lbest) e = k;
                sv = e >= 0 ? e0 + e : -1;
                if (sv == excl) sv = -1;
                q = sv >= 0 ? (sv - v0) >> kNoiseBlockShift : 0;
            }
            M = __shfl_sync(0xffffffffu, bn.M, q);
            I = __shfl_sync(0xffffffffu, bn.I, q);
            if (__any_sync(0xffffffffu, sv >= 0)) {
                const float E = noise_exp_f32(rp, M, I, static_cast<uint32_t>(sv < 0 ? 0 : sv));
                if (sv >= 0) {
                    const float zb = transform_f32<SOFTCAP, PENALTY>(lbest, pen_at(sv), P) * P.invT;
                    // the argmin element is already in; its score here is the same
                    if (static_cast<int>(static_cast<uint32_t>(sv) & kNoiseBlockMask) != I)
                        top2_push(tt, zb - ln_fast(E), sv);
                    else
                        sv = -1;
                }
            }
        }
        // ---- publish the warp's best to the row, read back the row's best
        unsigned* gthr = P.row_thr + row;
        const unsigned kw = warp_best_key(tt.s1);
        unsigned kg = 0u;
        if (lane == 0) {
            if (kw != 0u) atomicMax(gthr, kw);
            kg = __ldcg(gthr);
        }
        kg = __shfl_sync(0xffffffffu, max(kg, kw), 0);
        const float best = key_score(kg);
        float thr = best > -INFINITY ? best - cand_delta(best) : -INFINITY;

        // ================= phase B =================
        // lane q (block q) turns the best into a raw-value bound for its block, packed
        // twice: element x of block q can reach the best only if x >= xt_q
        uint32_t xt2 = 0u;
        {
            const float zt = (thr + bn.lnM) * P.T;
            float xt = zt;
            if constexpr (SOFTCAP) {
                // shrink by more than the fp32 error of c tanh(x / c) before inverting:
                // atanh is steep near |u| = 1
                float u = zt * P.invcap;
                u -= 1e-6f * fabsf(u) + 1e-7f;
                xt = u > 1.0f ? INFINITY : (u <= -1.0f ? -INFINITY : P.cap * atanhf(fminf(u, 1.0f - 1e-7f)));
            }
            xt -= 1e-5f * (1.0f + fabsf(xt));  // slack for the rounding of the transform
            if (!(thr > -INFINITY)) xt = -INFINITY;
            xt2 = bf16x2_floor(xt);
        }
        // vector k of a lane lies in block k * EPV / 8; two vectors per test
        unsigned pv = penv;
#pragma unroll
        for (int k2 = 0; k2 < NV / 2; ++k2) {
            const int q0 = (2 * k2) * EPV / 8, q1 = (2 * k2 + 1) * EPV / 8;
            const uint32_t t0 = __shfl_sync(0xffffffffu, xt2, q0), t1 = __shfl_sync(0xffffffffu, xt2, q1);
            const uint32_t th = (t0 & 0xFFFFu) | (t1 & 0xFFFF0000u);
            const unsigned mk = __hge2_mask(as_bf162(vmx[k2]), as_bf162(th));
            pv |= ((mk & 1u) | ((mk >> 15) & 2u)) << (2 * k2);
        }
        pv &= (ebase < v1 ? 0xFFFFFFFFu : 0u);  // (a lane wholly past the end has nothing)
        // the passing vectors: reload, bound each element exactly, score the survivors
        while (__any_sync(0xffffffffu, pv != 0u)) {
            int k = -1;
            uint4 r = make_uint4(0u, 0u, 0u, 0u);
            if (pv != 0u) {
                k = __ffs(pv) - 1;
                pv &= pv - 1u;
                const int e0 = ebase + k * RV;
                if (e0 < v1) r = load_vec<BF16>(rowp, e0, v1, P.aligned);
                else k = -1;
            }
            float x[EPV];
            unpack<BF16>(r, x);
            const int q = k >= 0 ? (k * EPV) >> 3 : 0;
            const float Mq = __shfl_sync(0xffffffffu, bn.M, q);
            const float lnq = __shfl_sync(0xffffffffu, bn.lnM, q);
            const int Iq = __shfl_sync(0xffffffffu, bn.I, q);
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                const int v = k >= 0 ? ebase + k * RV + e : -1;
                bool live = false;
                float zb = -INFINITY;
                if (v >= 0 && v < v1 && v != excl && v != sv && static_cast<int>(static_cast<uint32_t>(v) & kNoiseBlockMask) != Iq) {
                    zb = transform_f32<SOFTCAP, PENALTY>(x[e], pen_at(v), P) * P.invT;
                    live = zb - lnq + bound_slack(zb) >= thr;
                }
                if (__any_sync(0xffffffffu, live)) {
                    const float E = noise_exp_f32(rp, Mq, Iq, static_cast<uint32_t>(v < 0 ? 0 : v));
                    if (live) {
                        const float score = zb - ln_fast(E);
                        if (score >= thr) {
                            top2_push(tt, score, v);
                            thr = fmaxf(thr, tt.s1 - cand_delta(tt.s1));
                        }
                    }
                }
            }
        }
        const unsigned kw2 = warp_best_key(tt.s1);
        if (lane == 0 && kw2 > kw) atomicMax(gthr, kw2);
    }

    // ---- the piece's partial, then the row merge if this warp completes the row
    float pm = GREEDY ? m : mref, ps = s;
    if constexpr (!GREEDY) {
        if (!(pm > -INFINITY)) ps = 0.0f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, pm, off);
            const float so = __shfl_xor_sync(0xffffffffu, ps, off);
            ms_merge(pm, ps, mo, so, P.sc);
        }
    }
    const Top2 pt = top2_warp_reduce(tt);
    int last = 0;
    if (lane == 0) {
        // a written partial is never all-zero
        st_partial(P.part + static_cast<size_t>(row) * P.nchunk + p, GREEDY ? 0.0f : pm, GREEDY ? 1.0f : ps, pt);
        __threadfence();
        last = atomicAdd(&P.row_ticket[row], 1u) == static_cast<unsigned>(P.nchunk - 1);
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
    if (lane == 0) P.row_thr[row] = 0u;  // every piece of the row is done
    merge_row<BF16, GREEDY, SOFTCAP, PENALTY>(P, row);
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
    // one warp per piece of every row that may be active; warps of inactive rows exit at once
    const long long warps = static_cast<long long>(P.B) * (P.K + 1) * P.nchunk;
    const unsigned grid = static_cast<unsigned>((warps + kPW - 1) / kPW);
    verify_piece_kernel<BF16, G, C, R><<<grid, kPT, 0, s>>>(P);
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

// The kernels of one spec_verify call for one logits dtype: the piece kernel
// (with the merges), then, for dense q at T > 0, the residual pass.
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
