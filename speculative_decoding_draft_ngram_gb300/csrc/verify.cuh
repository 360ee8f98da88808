// spec_verify kernels (sm_103a): the streaming pass over the logit rows, the
// dense-q residual pass, and the per-row / per-sequence epilogues.
//
// Method (SwiftLM page, paragraph on algorithmic equivalence after Leviathan
// et al.; AX Engine page, "Core Technical Architecture & Methods"):
//   row transform  soft cap -> repetition penalty -> temperature
//   p_j = softmax(x_j / T); accept draft i iff u_i q(d_i) <= p(d_i)
//   a = number accepted before the first rejection (<= k_eff, EMA gate)
//   sample at row a: residual max(0, p_a - q_a) on a rejection, p_a (bonus)
//   otherwise, by Gumbel-max with Philox noise; T = 0: argmax matching
//   epilogue: tokens, kv_len <- kv_len - k + a, EMA update.
//
// Design (one GPU, HBM-bound):
//   * grid = (sequence, row, V-chunk); a CTA of 256 threads owns one chunk
//     of one row; each thread keeps its 8 x 16-byte vectors in registers, so
//     the chunk is read from HBM exactly once with coalesced 16-byte loads;
//   * pass A over the registers: per-vector maximum (the soft cap is
//     monotone, so it is applied to the vector maximum only);
//   * pass B: sum of exponentials against the thread's own maximum (no
//     rescaling in the loop) and Gumbel candidates.  A vector is skipped
//     unless max(x)/T + g_max can still reach the current threshold, and
//     Philox runs only for the few elements that pass; the threshold is seeded
//     per warp by the exact score of the warp's largest element;
//   * candidates are kept as the top two by fp32 score; the last CTA of a
//     row merges the chunk partials (max / sum in fp64, candidates), re-scores
//     the two candidates in fp64 from the raw logits and takes the accept
//     test in fp64, so the integer decisions are taken in the oracle's
//     precision;
//   * cross-CTA merges use the fence + atomic ticket pattern: the last CTA of
//     a row merges the row; the last row of a sequence runs the epilogue.
//     Nothing waits on another CTA.
#pragma once

#include "common.cuh"

namespace specng {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kNV = 8;  // 16-byte vectors per thread per chunk

template <bool BF16> struct ElemTraits;
template <> struct ElemTraits<true> { static constexpr int EPV = 8; static constexpr int SIZE = 2; };
template <> struct ElemTraits<false> { static constexpr int EPV = 4; static constexpr int SIZE = 4; };

template <bool BF16>
__host__ __device__ constexpr int chunk_elems() { return kThreads * kNV * ElemTraits<BF16>::EPV; }

// Workspace records.
struct __align__(32) Partial {
    float m, s;  // chunk maximum (transformed units) and sum of exp((z - m) / T)
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
    int B, K, V, nchunk;
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
    NoiseKey nk;              // seq filled per CTA
    int aligned;              // logits (and q) allow 16-byte vector loads
    int32_t* kv_len;
    float* ema;
    int32_t* out_tokens;
    int32_t* out_accept;
    Partial* part;
    RowRes* rowres;
    SeqRes* seqres;
    unsigned* row_ticket;
    unsigned* row_thr;        // best candidate score published per row (score_key)
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

__device__ __forceinline__ double warp_max_f64(double v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
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

// Gumbel variate from a Philox word with hardware log2 (error ~1e-5): a
// pre-filter only; candidates that pass it are re-scored with gumbel_f32.
__device__ __forceinline__ float gumbel_fast(uint32_t w) {
    const float u = static_cast<float>(uniform_numerator(w)) * 0x1p-24f;
    const float y = 1.0f - u;  // exact
    float e;
    if (y < 0.0625f) {
        e = y * fmaf(y, fmaf(y, fmaf(y, 0.25f, 0.33333334f), 0.5f), 1.0f);  // -log1p(-y) series
    } else {
        e = -0.6931472f * __log2f(u);
    }
    return -0.6931472f * __log2f(e);
}

constexpr int kQCap = 32 + 32 * 8;  // per-warp candidate queue: a drained remainder + one push

// Merge (m, s) pairs whose sums are relative to their own maxima.
__device__ __forceinline__ void ms_merge(float& m, float& s, float mo, float so, float sc) {
    const float M = fmaxf(m, mo);
    float r = 0.0f;
    if (m > -INFINITY) r += s * ex2_approx((m - M) * sc);
    if (mo > -INFINITY) r += so * ex2_approx((mo - M) * sc);
    m = M;
    s = r;
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

template <bool PENALTY, int EPV>
__device__ __forceinline__ unsigned pen_bits(const uint32_t* s_bm, int off) {
    if constexpr (!PENALTY) {
        return 0u;
    } else {
        return (s_bm[off >> 5] >> (off & 31)) & ((1u << EPV) - 1u);
    }
}

// ---------------------------------------------------------------- K1

template <bool BF16, bool GREEDY, bool SOFTCAP, bool PENALTY>
__global__ void __launch_bounds__(kThreads, 2) verify_stream_kernel(const VerifyDev P) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    constexpr int CHUNK = chunk_elems<BF16>();
    __shared__ uint32_t s_bm[PENALTY ? CHUNK / 32 : 1];
    __shared__ int s_win[PENALTY ? SPECNG_MAX_REP_WINDOW : 1];
    __shared__ int s_nwin;
    __shared__ float s_m[kWarps], s_s[kWarps], s_seed[kWarps];
    __shared__ Top2 s_t[kWarps];
    __shared__ int s_last;
    __shared__ int s_qn[kWarps];
    __shared__ int2 s_q[GREEDY ? 1 : kWarps * kQCap];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K1 = P.K + 1;
    const int rows = P.B * K1;
    // chunk-major order: chunk c of every row is scheduled before chunk c + 1,
    // so later chunks start from the best score the earlier ones published
    const int c = blockIdx.x / rows;
    const int row = blockIdx.x - c * rows;
    const int b = row / K1, j = row - b * K1;

    int kb = P.k[b];
    if (kb < 0 || kb > P.K) {
        if (j == 0 && c == 0 && tid == 0) raise_status(P.status, SPECNG_DEV_BAD_K);
        kb = kb < 0 ? 0 : P.K;
    }
    if (j > kb) return;
    int keff = kb;
    if (P.gate && kb > 0 && !(P.ema[b] >= P.thresh)) keff = 0;
    if (j > keff) return;

    const bool dense = P.q != nullptr;
    const int dnext = j < keff ? P.drafts[b * P.K + j] : -1;  // d_{j+1}
    const bool dvalid = dnext >= 0 && dnext < P.V;
    if (j < keff && !dvalid && c == 0 && tid == 0) raise_status(P.status, SPECNG_DEV_TOKEN_OOR);
    const int excl = (!GREEDY && !dense && j < keff && dvalid) ? dnext : -1;
    const int v0 = c * CHUNK;
    const int v1 = min(P.V, v0 + CHUNK);
    const char* rowp = static_cast<const char*>(P.logits) +
                       static_cast<size_t>(row) * P.V * ElemTraits<BF16>::SIZE;
    NoiseKey nk = P.nk;
    nk.seq = static_cast<uint32_t>(b);

    if constexpr (PENALTY) build_window<CHUNK>(P, b, j, v0, v1, s_bm, s_win, &s_nwin);

    // ---- load the chunk into registers (one HBM read of every byte)
    uint4 raw[kNV];
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
        const int e0 = v0 + (i * kThreads + tid) * EPV;
        raw[i] = e0 < v1 ? load_vec<BF16>(rowp, e0, v1, P.aligned) : make_uint4(0u, 0u, 0u, 0u);
    }

    // ---- pass A: per-vector maximum of the transformed values
    float vmax[kNV];
    float m_t = -INFINITY;
    int arg_t = -1;
    Top2 gt = top2_empty();
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
        const int off = (i * kThreads + tid) * EPV;
        const int e0 = v0 + off;
        const int nv = min(EPV, v1 - e0);
        vmax[i] = -INFINITY;
        if (nv <= 0) continue;
        float x[EPV];
        unpack<BF16>(raw[i], x);
        const unsigned pb = pen_bits<PENALTY, EPV>(s_bm, off);
        float zm = -INFINITY;
        int am = -1;
        if (nv == EPV && pb == 0u) {
            float mx = x[0];
            int ax = 0;
#pragma unroll
            for (int e = 1; e < EPV; ++e) if (x[e] > mx) { mx = x[e]; ax = e; }
            zm = SOFTCAP ? transform_f32<true, false>(mx, false, P) : mx;
            am = ax;
        } else {
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                if (e >= nv) break;
                const float z = transform_f32<SOFTCAP, PENALTY>(x[e], (pb >> e) & 1u, P);
                if (z > zm || am < 0) { zm = z; am = e; }
            }
        }
        vmax[i] = zm;
        if (zm > m_t) { m_t = zm; arg_t = e0 + am; }
        if constexpr (GREEDY) {
            if (zm >= gt.s2) {
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    if (e >= nv) break;
                    top2_push(gt, transform_f32<SOFTCAP, PENALTY>(x[e], (pb >> e) & 1u, P), e0 + e);
                }
            }
        }
    }

    float m_c = -INFINITY, s_c = 0.0f;
    Top2 tt = top2_empty();
    if constexpr (!GREEDY) {
        // ---- threshold seed: exact score of each warp's largest element; the
        //      best of them over the CTA and of what earlier chunks published
        {
            float t0 = -INFINITY;
            float wm = m_t;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, off));
            const unsigned own = __ballot_sync(0xffffffffu, wm > -INFINITY && m_t == wm && arg_t >= 0 && arg_t != excl);
            if (own != 0u) {
                const int src = __ffs(own) - 1;
                if (lane == src) {
                    const uint4 w = gumbel_block(nk, static_cast<uint32_t>(arg_t) >> 2, static_cast<uint32_t>(j));
                    t0 = m_t * P.invT + gumbel_f32(pick_word(w, static_cast<uint32_t>(arg_t) & 3u));
                }
                t0 = __shfl_sync(0xffffffffu, t0, src);
            }
            if (lane == 0) { s_seed[warp] = t0; s_qn[warp] = 0; }
        }
        __syncthreads();
        float seed = s_seed[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) seed = fmaxf(seed, s_seed[w]);
        const float pub = key_score(__ldcg(&P.row_thr[row]));
        if (tid == 0 && seed > -INFINITY) atomicMax(&P.row_thr[row], score_key(seed));
        const float best0 = fmaxf(seed, pub);
        float thr = best0 > -INFINITY ? best0 - cand_delta(best0) : -INFINITY;
        float zthr = thr - kGumbelMax;  // an element can reach thr only if z / T >= zthr
        int2* q = s_q + warp * kQCap;
        volatile int* qn = s_qn + warp;

        // score one queued candidate (all lanes busy); updates tt / thr
        auto score_one = [&](int2 ent) {
            const int v = ent.x;
            const float zb = __int_as_float(ent.y);
            if (v == excl || zb + kGumbelMax < thr) return;
            const uint4 w = gumbel_block(nk, static_cast<uint32_t>(v) >> 2, static_cast<uint32_t>(j));
            const uint32_t word = pick_word(w, static_cast<uint32_t>(v) & 3u);
            if (zb + gumbel_fast(word) < thr - 1e-3f) return;
            const float score = zb + gumbel_f32(word);
            if (score >= thr) {
                top2_push(tt, score, v);
                thr = fmaxf(thr, tt.s1 - cand_delta(tt.s1));
            }
        };

        // ---- pass B: sum of exponentials; candidates go to the warp's queue
        const float msc = m_t * P.sc;
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < kNV; ++i) {
            const int off = (i * kThreads + tid) * EPV;
            const int e0 = v0 + off;
            const int nv = min(EPV, v1 - e0);
            float z[EPV];
            if (nv > 0) {
                float x[EPV];
                unpack<BF16>(raw[i], x);
                const unsigned pb = pen_bits<PENALTY, EPV>(s_bm, off);
                if (nv == EPV) {
                    float acc = 0.0f;
#pragma unroll
                    for (int e = 0; e < EPV; ++e) {
                        z[e] = transform_f32<SOFTCAP, PENALTY>(x[e], (pb >> e) & 1u, P);
                        acc += ex2_approx(fmaf(z[e], P.sc, -msc));
                    }
                    s += acc;
                } else {
#pragma unroll
                    for (int e = 0; e < EPV; ++e) {
                        z[e] = transform_f32<SOFTCAP, PENALTY>(x[e], (pb >> e) & 1u, P);
                        if (e < nv) s += ex2_approx(fmaf(z[e], P.sc, -msc));
                    }
                }
                if (vmax[i] * P.invT >= zthr) {
                    unsigned msk = 0u;
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        if (e < nv && z[e] * P.invT >= zthr) msk |= 1u << e;
                    if (msk != 0u) {
                        int slot = atomicAdd(&s_qn[warp], __popc(msk));
#pragma unroll
                        for (int e = 0; e < EPV; ++e)
                            if ((msk >> e) & 1u) q[slot++] = make_int2(e0 + e, __float_as_int(z[e] * P.invT));
                    }
                }
            }
            __syncwarp();
            int n = *qn;
            if (n >= 32) {
                do {
                    score_one(q[n - 32 + lane]);
                    n -= 32;
                } while (n >= 32);
#pragma unroll
                for (int off2 = 16; off2 > 0; off2 >>= 1) thr = fmaxf(thr, __shfl_xor_sync(0xffffffffu, thr, off2));
                zthr = thr - kGumbelMax;
                __syncwarp();
                if (lane == 0) *qn = n;
                __syncwarp();
            }
        }
        {
            const int n = *qn;
            if (lane < n) score_one(q[lane]);
        }
        if (!(m_t > -INFINITY)) s = 0.0f;
        // ---- CTA reduction of (max, sum) and candidates
        m_c = m_t;
        s_c = s;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, m_c, off);
            const float so = __shfl_xor_sync(0xffffffffu, s_c, off);
            ms_merge(m_c, s_c, mo, so, P.sc);
        }
        tt = top2_warp_reduce(tt);
    } else {
        tt = top2_warp_reduce(gt);
    }
    if (lane == 0) { s_m[warp] = m_c; s_s[warp] = s_c; s_t[warp] = tt; }
    __syncthreads();
    if (warp == 0) {
        float m = lane < kWarps ? s_m[lane] : -INFINITY;
        float s = lane < kWarps ? s_s[lane] : 0.0f;
        Top2 t = lane < kWarps ? s_t[lane] : top2_empty();
#pragma unroll
        for (int off = 4; off > 0; off >>= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, m, off);
            const float so = __shfl_xor_sync(0xffffffffu, s, off);
            ms_merge(m, s, mo, so, P.sc);
            t = top2_merge(t, top2_shfl_xor(t, off));
        }
        if (lane == 0) {
            st_partial(P.part + static_cast<size_t>(row) * P.nchunk + c, m, s, t);
            if (!GREEDY && t.s1 > -INFINITY) atomicMax(&P.row_thr[row], score_key(t.s1));
            __threadfence();
            const unsigned prev = atomicAdd(&P.row_ticket[row], 1u);
            s_last = prev == static_cast<unsigned>(P.nchunk - 1);
        }
    }
    __syncthreads();
    if (!s_last || warp != 0) return;
    __threadfence();

    // ---- last CTA of the row: merge the chunks (warp 0)
    if (lane == 0) { P.row_ticket[row] = 0u; P.row_thr[row] = 0u; }
    const Partial* pr = P.part + static_cast<size_t>(row) * P.nchunk;
    double M = -INFINITY;
    for (int cc = lane; cc < P.nchunk; cc += 32) M = fmax(M, static_cast<double>(__ldcg(&pr[cc].m)));
    M = warp_max_f64(M);
    double S = 0.0;
    Top2 t = top2_empty();
    for (int cc = lane; cc < P.nchunk; cc += 32) {
        const Partial p = ldcg_partial(pr + cc);
        if (!GREEDY && p.m > -INFINITY) S += static_cast<double>(p.s) * exp((static_cast<double>(p.m) - M) / P.Td);
        t = top2_merge(t, p.t);
    }
    S = warp_sum_f64(S);
    t = top2_warp_reduce(t);
    // leave the workspace zeroed for the next call (any shape may reuse it)
    __syncwarp();
    for (int cc = lane; cc < P.nchunk; cc += 32) st_zero(const_cast<Partial*>(pr) + cc);
    const double lse = GREEDY ? 0.0 : M / P.Td + log(S);
    if (!GREEDY && !(S > 0.0 && S < INFINITY && M < INFINITY) && lane == 0)
        raise_status(P.status, SPECNG_DEV_NONFINITE);

    // fp64 re-score of the (up to) two candidates from the raw logits
    const int nw = PENALTY ? s_nwin : 0;
    const bool pen1 = PENALTY && t.i1 >= 0 ? warp_in_window(t.i1, s_win, nw) : false;
    const bool pen2 = PENALTY && t.i2 >= 0 ? warp_in_window(t.i2, s_win, nw) : false;
    int winner = t.i1;
    if (lane == 0 && t.i1 >= 0) {
        const bool second = t.i2 >= 0 && t.s2 >= t.s1 - cand_delta(t.s1);
        double sc1, sc2 = -INFINITY;
        {
            const double z = transform_f64<SOFTCAP, PENALTY>(raw_logit_f64<BF16>(P.logits, row, P.V, t.i1), pen1, P);
            if constexpr (GREEDY) {
                sc1 = z;
            } else {
                const uint4 w = gumbel_block(nk, static_cast<uint32_t>(t.i1) >> 2, static_cast<uint32_t>(j));
                sc1 = z / P.Td + gumbel_f64(pick_word(w, static_cast<uint32_t>(t.i1) & 3u));
            }
        }
        if (second) {
            const double z = transform_f64<SOFTCAP, PENALTY>(raw_logit_f64<BF16>(P.logits, row, P.V, t.i2), pen2, P);
            if constexpr (GREEDY) {
                sc2 = z;
            } else {
                const uint4 w = gumbel_block(nk, static_cast<uint32_t>(t.i2) >> 2, static_cast<uint32_t>(j));
                sc2 = z / P.Td + gumbel_f64(pick_word(w, static_cast<uint32_t>(t.i2) & 3u));
            }
            if (better64(sc2, t.i2, sc1, t.i1)) winner = t.i2;
        }
    }
    winner = __shfl_sync(0xffffffffu, winner, 0);

    // accept test of the draft this row verifies, in fp64
    int accepted = 0;
    if (j < keff && dvalid) {
        if constexpr (GREEDY) {
            accepted = dnext == winner;
        } else {
            const bool pend = PENALTY ? warp_in_window(dnext, s_win, nw) : false;
            if (lane == 0) {
                const double zd = transform_f64<SOFTCAP, PENALTY>(raw_logit_f64<BF16>(P.logits, row, P.V, dnext), pend, P);
                const double p = exp(zd / P.Td - lse);
                const double q = dense ? static_cast<double>(P.q[(static_cast<size_t>(b) * P.K + j) * P.V + dnext]) : 1.0;
                const double u = accept_uniform_f64(nk, static_cast<uint32_t>(j + 1));
                accepted = u * q <= p;
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

    // ---- last row of the sequence: epilogue (warp 0)
    if (lane == 0) P.seq_ticket[b] = 0u;
    const RowRes* rs = P.rowres + static_cast<size_t>(b) * K1;
    int acc = 1;
    if (lane < keff) acc = __ldcg(&rs[lane].accepted);
    const unsigned rej = __ballot_sync(0xffffffffu, lane < keff && !acc);
    const int a = rej ? __ffs(rej) - 1 : keff;
    // a rejected draft outside [0, V) leaves the residual equal to p: the
    // row's own candidate (over all ids) is then the sample
    const int da = a < keff ? P.drafts[b * P.K + a] : -1;
    const bool need = dense && !GREEDY && a < keff && da >= 0 && da < P.V;
    const int y = need ? -1 : __ldcg(&rs[a].winner);
    __syncwarp();
    if (lane <= keff && !(need && lane == a)) st_zero(const_cast<RowRes*>(rs) + lane);
    if (lane < K1) P.out_tokens[static_cast<size_t>(b) * K1 + lane] = lane < a ? P.drafts[b * P.K + lane] : (lane == a ? y : -1);
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

// ---------------------------------------------------------------- K2
// Dense draft distributions: after a rejection at row a, sample from the
// residual max(0, p_a - q_a) by Gumbel-max over row a (logits and q read once
// more, for the rejected sequences only).

template <bool BF16, bool SOFTCAP, bool PENALTY>
__global__ void __launch_bounds__(kThreads, 2) verify_residual_kernel(const VerifyDev P) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    constexpr int CHUNK = chunk_elems<BF16>();
    __shared__ uint32_t s_bm[PENALTY ? CHUNK / 32 : 1];
    __shared__ int s_win[PENALTY ? SPECNG_MAX_REP_WINDOW : 1];
    __shared__ int s_nwin;
    __shared__ Top2 s_t[kWarps];
    __shared__ int s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K1 = P.K + 1;
    const int b = blockIdx.x / P.nchunk;
    const int c = blockIdx.x - b * P.nchunk;
    const int need = __ldcg(&P.seqres[b].need_residual);
    if (!need) return;
    const int a = __ldcg(&P.seqres[b].a);
    const int row = b * K1 + a;
    const float lse_f = static_cast<float>(__ldcg(&P.rowres[row].lse));
    const int v0 = c * CHUNK;
    const int v1 = min(P.V, v0 + CHUNK);
    const char* rowp = static_cast<const char*>(P.logits) +
                       static_cast<size_t>(row) * P.V * ElemTraits<BF16>::SIZE;
    const float* qrow = P.q + (static_cast<size_t>(b) * P.K + a) * P.V;
    NoiseKey nk = P.nk;
    nk.seq = static_cast<uint32_t>(b);

    if constexpr (PENALTY) build_window<CHUNK>(P, b, a, v0, v1, s_bm, s_win, &s_nwin);

    Top2 tt = top2_empty();
    float thr = -INFINITY;
    uint32_t cblk = 0xFFFFFFFFu;
    uint4 cw = make_uint4(0u, 0u, 0u, 0u);
    const float l2 = kLog2e;
#pragma unroll 2
    for (int i = 0; i < kNV; ++i) {
        const int off = (i * kThreads + tid) * EPV;
        const int e0 = v0 + off;
        const int nv = min(EPV, v1 - e0);
        if (nv <= 0) continue;
        const uint4 r = load_vec<BF16>(rowp, e0, v1, P.aligned);
        float x[EPV], qv[EPV];
        unpack<BF16>(r, x);
        if (P.aligned) {
#pragma unroll
            for (int h = 0; h < EPV / 4; ++h) {
                const float4 q4 = __ldcs(reinterpret_cast<const float4*>(qrow + e0) + h);
                qv[4 * h + 0] = q4.x; qv[4 * h + 1] = q4.y; qv[4 * h + 2] = q4.z; qv[4 * h + 3] = q4.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < EPV; ++e) qv[e] = e < nv ? qrow[e0 + e] : 0.0f;
        }
        const unsigned pb = pen_bits<PENALTY, EPV>(s_bm, off);
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            if (e >= nv) break;
            const float lp = transform_f32<SOFTCAP, PENALTY>(x[e], (pb >> e) & 1u, P) * P.invT - lse_f;
            if (lp + kGumbelMax < thr) continue;
            const float rsd = ex2_approx(lp * l2) - qv[e];
            if (!(rsd > 0.0f)) continue;
            const int v = e0 + e;
            const uint32_t blk = static_cast<uint32_t>(v) >> 2;
            if (blk != cblk) { cw = gumbel_block(nk, blk, static_cast<uint32_t>(a)); cblk = blk; }
            const float score = logf(rsd) + gumbel_f32(pick_word(cw, static_cast<uint32_t>(v) & 3u));
            if (score >= thr) {
                top2_push(tt, score, v);
                thr = fmaxf(thr, tt.s1 - cand_delta(tt.s1));
            }
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
            s_last = prev == static_cast<unsigned>(P.nchunk - 1);
        }
    }
    __syncthreads();
    if (!s_last || warp != 0) return;
    __threadfence();
    if (lane == 0) P.seq_ticket2[b] = 0u;
    const Partial* pr = P.part2 + static_cast<size_t>(b) * P.nchunk;
    Top2 t = top2_empty();
    for (int cc = lane; cc < P.nchunk; cc += 32) t = top2_merge(t, ldcg_partial(pr + cc).t);
    t = top2_warp_reduce(t);
    __syncwarp();
    for (int cc = lane; cc < P.nchunk; cc += 32) st_zero(const_cast<Partial*>(pr) + cc);
    const int nw = PENALTY ? s_nwin : 0;
    const bool pen1 = PENALTY && t.i1 >= 0 ? warp_in_window(t.i1, s_win, nw) : false;
    const bool pen2 = PENALTY && t.i2 >= 0 ? warp_in_window(t.i2, s_win, nw) : false;
    if (lane != 0) return;
    const double lse = __ldcg(&P.rowres[row].lse);
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
        const uint4 w = gumbel_block(nk, static_cast<uint32_t>(id) >> 2, static_cast<uint32_t>(a));
        const double score = log(rsd) + gumbel_f64(pick_word(w, static_cast<uint32_t>(id) & 3u));
        if (winner < 0 || better64(score, id, best, winner)) { best = score; winner = id; }
    }
    // all-zero residual (p <= q everywhere): sample from p, the row's bonus candidate
    if (winner < 0) winner = bonus;
    P.out_tokens[static_cast<size_t>(b) * K1 + a] = winner;
}

// Host-side launch of one dtype (defined in verify_bf16.cu / verify_f32.cu).
template <bool BF16>
cudaError_t launch_verify_dtype(const VerifyDev& P, bool greedy, bool softcap, bool penalty, bool dense,
                                cudaStream_t s);

}  // namespace specng
