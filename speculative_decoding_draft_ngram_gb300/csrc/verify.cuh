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

#include <cuda_bf16.h>

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

__device__ __forceinline__ unsigned warp_best_key(float best) {
    return __reduce_max_sync(0xffffffffu, best > -INFINITY ? score_key(best) : 0u);
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

constexpr int kQCap = 32 + 32 * 32;  // per-warp candidate queue (chunk offsets): a remainder + one stage

// Largest bf16 value <= f, as a packed pair (both halves).  NaN maps to +inf.
__device__ __forceinline__ uint32_t bf16x2_floor(float f) {
    uint32_t u = __float_as_uint(f);
    if (f != f) u = 0x7F800000u;
    uint32_t h = u >> 16;
    if ((u & 0x80000000u) && (u & 0xFFFFu) && (u & 0x7FFFFFFFu) < 0x7F800000u) h += 1u;  // negative: away from 0
    return h | (h << 16);
}

__device__ __forceinline__ __nv_bfloat162 as_bf162(uint32_t w) { return *reinterpret_cast<__nv_bfloat162*>(&w); }

// Maximum of the 8 bf16 values of a 16-byte vector (packed compares).
__device__ __forceinline__ float bf16x8_max(const uint4& r) {
    const __nv_bfloat162 a = __hmax2(__hmax2(as_bf162(r.x), as_bf162(r.y)), __hmax2(as_bf162(r.z), as_bf162(r.w)));
    const uint32_t w = *reinterpret_cast<const uint32_t*>(&a);
    return fmaxf(bf16lo(w), bf16hi(w));
}

// Bit e set when element e of the vector is >= the (packed) threshold t.
__device__ __forceinline__ unsigned bf16x8_ge_mask(const uint4& r, uint32_t t) {
    const __nv_bfloat162 th = as_bf162(t);
    const unsigned m0 = __hge2_mask(as_bf162(r.x), th), m1 = __hge2_mask(as_bf162(r.y), th);
    const unsigned m2 = __hge2_mask(as_bf162(r.z), th), m3 = __hge2_mask(as_bf162(r.w), th);
    return (m0 & 1u) | ((m0 >> 15) & 2u) | ((m1 & 1u) << 2) | ((m1 >> 13) & 8u) | ((m2 & 1u) << 4) |
           ((m2 >> 11) & 32u) | ((m3 & 1u) << 6) | ((m3 >> 9) & 128u);
}

// The same mask with fewer instructions: the high byte of each compared half
// is gathered with byte permutes, and the four 0xFF / 0x00 bytes of a word are
// turned into four bits by one multiply (the partial products of distinct
// bytes land on distinct bit positions, so nothing carries into bits 24..27).
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
// Persistent, warp-specialised streaming kernel.  One CTA per SM; the active
// row-chunks of the call (rows 0..k_eff of every sequence, V-chunks of
// CHUNK elements) are laid out row-major and split into equal contiguous
// ranges, one per CTA.  A producer warp walks its CTA's range and keeps up to
// kStages chunks in flight with cp.async.bulk into a shared-memory ring
// (full / empty mbarriers, bounded waits); sixteen consumer warps each take
// a 2 KB slice of every chunk.  A consumer warp keeps its Gumbel threshold
// across the consecutive chunks of one row, so only a row's first chunk
// needs a seed.  Each chunk leaves one partial (max, sum of exponentials,
// top-two candidates) in the workspace; the merge kernel combines them.

constexpr int kCWarps = 16;                    // consumer warps
constexpr int kPWarp = kCWarps;                // producer warp index
constexpr int kPThreads = (kCWarps + 1) * 32;  // 544
constexpr int kStages = 5;
constexpr int kVL = 4;                         // 16-byte vectors per lane per chunk

template <bool BF16>
__host__ __device__ constexpr int stage_bytes() { return chunk_elems<BF16>() * ElemTraits<BF16>::SIZE; }

template <bool PENALTY>
__host__ __device__ constexpr size_t k1_dyn_smem() {
    return static_cast<size_t>(kStages) * 32768 + static_cast<size_t>(kCWarps) * kQCap * sizeof(uint16_t) +
           (PENALTY ? static_cast<size_t>(kStages) * 2048 : 0);
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

// Bitmap of the penalised ids of row j that fall in [v0, v1); one warp builds it.
template <int CHUNK>
__device__ __forceinline__ void warp_build_bitmap(uint32_t* bm, const WindowView& wv, int j, int v0, int v1) {
    const int lane = threadIdx.x & 31;
    for (int t = lane; t < CHUNK / 32; t += 32) bm[t] = 0u;
    __syncwarp();
    const int n = wv.count(j);
    for (int t = lane; t < n; t += 32) {
        const int tok = wv.token(j, t);
        if (tok >= v0 && tok < v1) atomicOr(&bm[(tok - v0) >> 5], 1u << ((tok - v0) & 31));
    }
    __syncwarp();
}

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

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

struct StageMeta {
    int b, j, c, excl, seg_end;  // seg_end: the last chunk of this row in the CTA's range
    int cand;                    // the row's Gumbel candidates can be the emitted token
};

struct WarpPart {
    float m, s;
    Top2 t;
};

template <bool BF16, bool GREEDY, bool SOFTCAP, bool PENALTY>
__global__ void __launch_bounds__(kPThreads, 1) verify_stream_kernel(const VerifyDev P) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    constexpr int CHUNK = chunk_elems<BF16>();
    constexpr int SB = stage_bytes<BF16>();
    static_assert(SB == 32768 && SB == kCWarps * 32 * kVL * 16, "stage layout");
    extern __shared__ __align__(128) uint8_t s_dyn[];
    uint8_t* s_stage = s_dyn;
    uint16_t* s_q = reinterpret_cast<uint16_t*>(s_dyn + kStages * SB);
    uint32_t* s_bm = reinterpret_cast<uint32_t*>(s_dyn + kStages * SB + kCWarps * kQCap * sizeof(uint16_t));
    __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages];
    __shared__ StageMeta s_meta[kStages];
    __shared__ WarpPart s_slot[kStages][kCWarps];
    __shared__ int s_cnt[kStages];
    __shared__ unsigned s_rthr[kStages + 1];  // per-segment shared threshold (score_key; 0 = none)
    __shared__ int s_qn[kCWarps];
    __shared__ float s_cz[GREEDY ? 1 : kCWarps * 32];  // carried candidates: z / T
    __shared__ int s_cv[GREEDY ? 1 : kCWarps * 32];    // carried candidates: vocab id
    __shared__ long long s_wsum[kPThreads / 32];
    __shared__ int s_start[3];
    __shared__ int s_hwin[PENALTY ? SPECNG_MAX_REP_WINDOW : 1];
    __shared__ int s_pdrafts[SPECNG_MAX_K + 1];

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
        int b = s_start[0], j = s_start[1], c = s_start[2];
        int kb = 0;
        int keff = 0;
        int nh = 0;
        auto load_seq = [&](int bq) {
            keff = gate_keff(P, bq, &kb, true);
            if (lane < keff) {
                const int d = P.drafts[bq * P.K + lane];
                s_pdrafts[lane] = d;
                if (!(d >= 0 && d < P.V)) raise_status(P.status, SPECNG_DEV_TOKEN_OOR);
            }
            if constexpr (PENALTY) {
                int L = P.lens[bq];
                L = L < 0 ? 0 : (static_cast<int64_t>(L) > P.hist_stride ? static_cast<int>(P.hist_stride) : L);
                nh = L < P.W ? L : P.W;
                for (int t = lane; t < nh; t += 32) s_hwin[t] = P.hist[static_cast<size_t>(bq) * P.hist_stride + (L - nh) + t];
            }
            __syncwarp();
        };
        load_seq(b);
        bool ok = true;
        for (int n = 0; n < nwork && ok; ++n) {
            const int st = n % kStages;
            const int use = n / kStages;
            if (use >= 1) ok = mbar_wait_bounded(&s_empty[st], static_cast<unsigned>((use - 1) & 1));
            if (!ok) { if (lane == 0) raise_status(P.status, SPECNG_DEV_TIMEOUT); break; }
            const int v0 = c * CHUNK;
            const int v1 = min(P.V, v0 + CHUNK);
            if (lane == 0) {
                int excl = -1;
                // with dense q, row j < k_eff is sampled by the residual pass unless
                // its draft is invalid (the residual is then p itself)
                int cand = 1;
                if (!GREEDY && j < keff) {
                    const int d = s_pdrafts[j];
                    const bool valid = d >= 0 && d < P.V;
                    if (!dense && valid) excl = d;
                    if (dense && valid) cand = 0;
                }
                s_meta[st] = StageMeta{b, j, c, excl, (c == P.nchunk - 1 || n == nwork - 1) ? 1 : 0, cand};
            }
            if constexpr (PENALTY) {
                const WindowView wv{s_hwin, s_pdrafts, nh, P.W};
                warp_build_bitmap<CHUNK>(s_bm + st * (CHUNK / 32), wv, j, v0, v1);
            }
            __syncwarp();
            const char* src = static_cast<const char*>(P.logits) +
                              ((static_cast<size_t>(b) * K1 + j) * P.V + v0) * ElemTraits<BF16>::SIZE;
            if (P.aligned) {
                if (lane == 0) {
                    // the empty barrier already orders the consumers' reads of this stage
                    // before the copy that overwrites it
                    mbar_expect_tx(&s_full[st], static_cast<unsigned>(v1 - v0) * ElemTraits<BF16>::SIZE);
                    bulk_g2s(s_stage + st * SB, src, static_cast<unsigned>(v1 - v0) * ElemTraits<BF16>::SIZE, &s_full[st]);
                }
            } else {
                uint8_t* dst = s_stage + st * SB;
                for (int e = lane; e < v1 - v0; e += 32) {
                    if constexpr (BF16) reinterpret_cast<uint16_t*>(dst)[e] = reinterpret_cast<const uint16_t*>(src)[e];
                    else reinterpret_cast<uint32_t*>(dst)[e] = reinterpret_cast<const uint32_t*>(src)[e];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_full[st]);
            }
            // advance to the next row-chunk
            if (++c == P.nchunk) {
                c = 0;
                if (++j > keff) {
                    j = 0;
                    ++b;
                    if (n + 1 < nwork) load_seq(b);
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

    // ================= consumers =================
    // Per-lane accumulators live across the chunks of one row (a segment of
    // the CTA's range); warps combine them once, at the segment's last chunk.
    // The candidate threshold of a segment is shared by the CTA's consumer
    // warps through a small ring of shared-memory slots (order-preserving
    // keys, atomicMax): every warp prunes with the best score any warp found.
    float thr = -INFINITY;
    float m = -INFINITY, s = 0.0f, msc = 0.0f;
    Top2 tt = top2_empty();
    bool fresh = true;
    int seg = 0;
    uint16_t* q = s_q + warp * kQCap;
    int cn = 0;  // candidates carried from the segment's previous stage (s_cz / s_cv)
    if (lane == 0) s_qn[warp] = 0;
    __syncwarp();
    for (int n = 0; n < nwork; ++n) {
        const int st = n % kStages;
        if (!mbar_wait_bounded(&s_full[st], static_cast<unsigned>((n / kStages) & 1))) {
            if (lane == 0) raise_status(P.status, SPECNG_DEV_TIMEOUT);
            break;
        }
        const StageMeta mt = s_meta[st];
        const int row = mt.b * K1 + mt.j;
        const int j = mt.j;
        const int excl = mt.excl;
        const int v0 = mt.c * CHUNK;
        const int v1 = min(P.V, v0 + CHUNK);
        const uint4* stage = reinterpret_cast<const uint4*>(s_stage + st * SB);
        const uint32_t* bm = s_bm + (PENALTY ? st * (CHUNK / 32) : 0);
        NoiseKey nk = P.nk;
        nk.seq = static_cast<uint32_t>(mt.b);
        const int ubase = warp * (32 * kVL);  // first 16-byte vector of my slice
        unsigned* rth = &s_rthr[seg % (kStages + 1)];
        const RowPhilox rp = row_philox(nk, static_cast<uint32_t>(j));

        if constexpr (GREEDY) {
            // top two transformed values (lower id on ties) within cand_delta of
            // the best value any warp of the CTA has seen in this segment.  The
            // slice's maxima come first (packed compares), so the threshold is
            // already the warp's best before any element is pushed.
            uint4 rv[kVL];
            float vmx[kVL];
            float lmax = -INFINITY;
#pragma unroll
            for (int i = 0; i < kVL; ++i) {
                const int u = ubase + i * 32 + lane;
                const int off = u * EPV;
                const int nv = min(EPV, v1 - (v0 + off));
                rv[i] = stage[u];
                const unsigned pb = pen_bits<PENALTY, EPV>(bm, off);
                float vm = -INFINITY;
                if (BF16 && nv == EPV && pb == 0u) {
                    vm = bf16x8_max(rv[i]);
                    if constexpr (SOFTCAP) vm = transform_f32<true, false>(vm, false, P);
                } else if (nv > 0) {
                    float x[EPV];
                    unpack<BF16>(rv[i], x);
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        if (e < nv) vm = fmaxf(vm, transform_f32<SOFTCAP, PENALTY>(x[e], (pb >> e) & 1u, P));
                }
                vmx[i] = vm;
                lmax = fmaxf(lmax, vm);
            }
            const unsigned wk = warp_best_key(lmax);
            float gth = fmaxf(fmaxf(tt.s1, key_score(wk)), key_score(*reinterpret_cast<volatile unsigned*>(rth)));
            gth = gth > -INFINITY ? gth - cand_delta(gth) : -INFINITY;
#pragma unroll
            for (int i = 0; i < kVL; ++i) {
                const int u = ubase + i * 32 + lane;
                const int off = u * EPV;
                const int e0 = v0 + off;
                const int nv = min(EPV, v1 - e0);
                if (nv <= 0 || !(vmx[i] >= gth)) continue;
                const unsigned pb = pen_bits<PENALTY, EPV>(bm, off);
                float x[EPV];
                unpack<BF16>(rv[i], x);
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    if (e >= nv) break;
                    const float z = transform_f32<SOFTCAP, PENALTY>(x[e], (pb >> e) & 1u, P);
                    if (z >= gth) top2_push(tt, z, e0 + e);
                }
                gth = fmaxf(gth, tt.s1 - cand_delta(tt.s1));
            }
            const unsigned kw = warp_best_key(tt.s1);
            if (lane == 0 && kw != 0u) atomicMax(rth, kw);
        } else {
            const bool cand = mt.cand != 0;
            int seeded = -1;  // element already scored as this lane's seed
            if (fresh && cand && !(BF16 && !PENALTY && v0 + (ubase + (kVL - 1) * 32 + lane) * EPV + EPV <= v1)) {
                // ---- seed: every lane scores the largest element of its slice
                float zm = -INFINITY;
                int am = -1;
#pragma unroll
                for (int i = 0; i < kVL; ++i) {
                    const int u = ubase + i * 32 + lane;
                    const int off = u * EPV;
                    const int e0 = v0 + off;
                    const int nv = min(EPV, v1 - e0);
                    if (nv <= 0) continue;
                    float x[EPV];
                    unpack<BF16>(stage[u], x);
                    const unsigned pb = pen_bits<PENALTY, EPV>(bm, off);
#pragma unroll
                    for (int e = 0; e < EPV; ++e) {
                        if (e >= nv) break;
                        const float z = transform_f32<SOFTCAP, PENALTY>(x[e], (pb >> e) & 1u, P);
                        if (z > zm && e0 + e != excl) { zm = z; am = e0 + e; }
                    }
                }
                float t0 = -INFINITY;
                if (am >= 0) {
                    const uint4 w = gumbel_block_row(rp, static_cast<uint32_t>(am) >> 2);
                    t0 = zm * P.invT + gumbel_f32(pick_word(w, static_cast<uint32_t>(am) & 3u));
                    top2_push(tt, t0, am);
                    seeded = am;
                }
                const unsigned k0 = warp_best_key(t0);
                if (k0 != 0u) {
                    t0 = key_score(k0);
                    thr = t0 - cand_delta(t0);
                    if (lane == 0) atomicMax(rth, k0);
                }
            }
            // candidate threshold in raw-logit units: z / T >= thr - g_max  <=>  x >= xt
            float xt;
            uint32_t xt2;
            auto set_xt = [&]() {
                const float zt = (thr - kGumbelMax) * P.T;
                if constexpr (SOFTCAP) {
                    // shrink u by more than the fp32 error of c * tanh(x / c) before inverting:
                    // atanh is steep near |u| = 1
                    float u = zt * P.invcap;
                    u -= 1e-6f * fabsf(u) + 1e-7f;
                    xt = u > 1.0f ? INFINITY : (u <= -1.0f ? -INFINITY : P.cap * atanhf(fminf(u, 1.0f - 1e-7f)));
                } else {
                    xt = zt;
                }
                xt -= 1e-5f * (1.0f + fabsf(xt));  // slack for the rounding of the transform
                xt2 = bf16x2_floor(xt);
            };
            // adopt the best score another warp published for this segment
            auto sync_thr = [&]() {
                const float best = key_score(*reinterpret_cast<volatile unsigned*>(rth));
                if (best > -INFINITY) {
                    const float t1 = best - cand_delta(best);
                    if (t1 > thr) { thr = t1; set_xt(); }
                }
            };
            if (cand) {
                set_xt();
                sync_thr();
            } else {
                xt = INFINITY;
                xt2 = 0x7F807F80u;
            }
            // ---- one pass over the slice: all four 16-byte vectors are loaded first; the
            //      online maximum and the 32 exponentials (packed fp32x2 arithmetic) form one
            //      independent block; candidate masks are formed only for the vectors whose
            //      maximum reaches the threshold
            uint4 rv[kVL];
#pragma unroll
            for (int i = 0; i < kVL; ++i) rv[i] = stage[ubase + i * 32 + lane];
            const int off0 = ubase * EPV + lane * EPV;  // chunk offset of vector 0's element 0
            const bool fast = v0 + (ubase + (kVL - 1) * 32 + lane) * EPV + EPV <= v1;  // four full vectors
            unsigned pmk = 0u;  // penalised elements of the slice (bit 8 i + e)
            if constexpr (PENALTY) {
#pragma unroll
                for (int i = 0; i < kVL; ++i) pmk |= pen_bits<PENALTY, EPV>(bm, off0 + i * 32 * EPV) << (8 * i);
            }
            unsigned msk = 0u;  // bit 8 i + e: element e of vector i
            if (fast) {
                float rmx[kVL];  // raw maxima
#pragma unroll
                for (int i = 0; i < kVL; ++i) {
                    if constexpr (BF16) {
                        rmx[i] = bf16x8_max(rv[i]);
                    } else {
                        rmx[i] = fmaxf(fmaxf(__uint_as_float(rv[i].x), __uint_as_float(rv[i].y)),
                                       fmaxf(__uint_as_float(rv[i].z), __uint_as_float(rv[i].w)));
                    }
                }
                float vm = fmaxf(fmaxf(rmx[0], rmx[1]), fmaxf(rmx[2], rmx[3]));
                if constexpr (BF16 && !PENALTY) {
                    if (fresh && cand) {
                        // seed: score the slice's largest element (lowest id among equals); the
                        // transform is monotone, so it is also the largest transformed value
                        int am = -1;
#pragma unroll
                        for (int i = kVL - 1; i >= 0; --i) {
                            if (rmx[i] == vm) {
                                float x[EPV];
                                unpack<BF16>(rv[i], x);
                                int e = EPV - 1;
#pragma unroll
                                for (int k = EPV - 2; k >= 0; --k) e = x[k] == vm ? k : e;
                                am = v0 + off0 + i * 32 * EPV + e;
                            }
                        }
                        float t0 = -INFINITY;
                        if (am >= 0 && am != excl) {
                            const uint4 w = gumbel_block_row(rp, static_cast<uint32_t>(am) >> 2);
                            t0 = transform_f32<SOFTCAP, false>(vm, false, P) * P.invT +
                                 gumbel_f32(pick_word(w, static_cast<uint32_t>(am) & 3u));
                            top2_push(tt, t0, am);
                            seeded = am;
                        }
                        const unsigned k0 = warp_best_key(t0);
                        if (k0 != 0u) {
                            t0 = key_score(k0);
                            thr = t0 - cand_delta(t0);
                            if (lane == 0) atomicMax(rth, k0);
                            set_xt();
                        }
                        sync_thr();  // and adopt the best seed any warp has published
                    }
                }
                if constexpr (SOFTCAP) vm = transform_f32<true, false>(vm, false, P);
                if (vm > m) {
                    s = m > -INFINITY ? s * ex2_approx((m - vm) * P.sc) : 0.0f;
                    m = vm;
                    msc = m * P.sc;
                }
                float2 acc2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
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
                        acc2[i & 1] = __fadd2_rn(acc2[i & 1], make_float2(ex2_approx(t.x), ex2_approx(t.y)));
                    }
                }
                s += (acc2[0].x + acc2[0].y) + (acc2[1].x + acc2[1].y);
                if (cand) {
#pragma unroll
                    for (int i = 0; i < kVL; ++i) {
                        if (!(rmx[i] >= xt)) continue;
                        unsigned mi;
                        if constexpr (BF16) {
                            mi = bf16x8_ge_bits(rv[i], xt2);
                        } else {
                            mi = 0u;
                            mi |= static_cast<unsigned>(__uint_as_float(rv[i].x) >= xt);
                            mi |= static_cast<unsigned>(__uint_as_float(rv[i].y) >= xt) << 1;
                            mi |= static_cast<unsigned>(__uint_as_float(rv[i].z) >= xt) << 2;
                            mi |= static_cast<unsigned>(__uint_as_float(rv[i].w) >= xt) << 3;
                        }
                        msk |= mi << (8 * i);
                    }
                }
                if constexpr (PENALTY) {
                    // the few penalised elements: replace their terms by the penalised ones
                    // (and raise the maximum if a penalty below 1 lifted one above it); they
                    // are always queued, so scoring sees their exact values
                    unsigned pw = pmk;
                    while (pw != 0u) {
                        const int bit = __ffs(pw) - 1;
                        pw &= pw - 1u;
                        const int loc = off0 + (bit >> 3) * 32 * EPV + (bit & 7);
                        float xe;
                        if constexpr (BF16) {
                            xe = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(stage)[loc]) << 16);
                        } else {
                            xe = reinterpret_cast<const float*>(stage)[loc];
                        }
                        const float zu = transform_f32<SOFTCAP, false>(xe, false, P);
                        const float zp = transform_f32<SOFTCAP, true>(xe, true, P);
                        if (zp > m) {
                            s *= ex2_approx((m - zp) * P.sc);
                            m = zp;
                            msc = m * P.sc;
                        }
                        s += ex2_approx(fmaf(zp, P.sc, -msc)) - ex2_approx(fmaf(zu, P.sc, -msc));
                    }
                    if (cand) msk |= pmk;
                }
            } else {
                // partial vectors (a row's last chunk): exact transform element by element
#pragma unroll
                for (int i = 0; i < kVL; ++i) {
                    const int off = off0 + i * 32 * EPV;
                    const int e0 = v0 + off;
                    const int nv = min(EPV, v1 - e0);
                    if (nv <= 0) continue;
                    float x[EPV], z[EPV];
                    unpack<BF16>(rv[i], x);
                    const unsigned pb = pen_bits<PENALTY, EPV>(bm, off);
                    float vmx = -INFINITY;
#pragma unroll
                    for (int e = 0; e < EPV; ++e) {
                        z[e] = transform_f32<SOFTCAP, PENALTY>(x[e], (pb >> e) & 1u, P);
                        if (e < nv) vmx = fmaxf(vmx, z[e]);
                    }
                    if (vmx > m) {
                        s = m > -INFINITY ? s * ex2_approx((m - vmx) * P.sc) : 0.0f;
                        m = vmx;
                        msc = m * P.sc;
                    }
                    const float zthr = thr - kGumbelMax;
#pragma unroll
                    for (int e = 0; e < EPV; ++e) {
                        if (e < nv) {
                            if (m > -INFINITY) s += ex2_approx(fmaf(z[e], P.sc, -msc));
                            if (cand) msk |= static_cast<unsigned>(z[e] * P.invT >= zthr) << (8 * i + e);
                        }
                    }
                }
            }
            if (seeded >= 0) {
                const int so = seeded - v0 - off0;  // position of the seed in the slice
                const int si = so / (32 * EPV), se = so - si * 32 * EPV;
                if (se >= 0 && se < EPV) msk &= ~(1u << (8 * si + se));
            }
            if (cand) {
            // ---- queue the slice's candidates (chunk offsets of this stage)
            const unsigned cnt = __popc(msk);
            const int nq = static_cast<int>(__reduce_add_sync(0xffffffffu, cnt));
            if (msk != 0u) {
                int slot = atomicAdd(&s_qn[warp], static_cast<int>(cnt));
                while (msk != 0u) {
                    const int bit = __ffs(msk) - 1;
                    msk &= msk - 1u;
                    q[slot++] = static_cast<uint16_t>(off0 + (bit >> 3) * 32 * EPV + (bit & 7));
                }
            }
            __syncwarp();
            // ---- score full batches of 32 from [carried ++ queued]; the remainder is carried to
            //      the segment's next stage (as transformed value and id), and scored at its end
            const bool flush = mt.seg_end != 0;
            const int total = cn + nq;
            float* cz = s_cz + warp * 32;
            int* cv = s_cv + warp * 32;
            auto fetch = [&](int idx, float& zb, int& v) {
                if (idx < cn) {
                    zb = cz[idx];
                    v = cv[idx];
                } else {
                    const int loc = static_cast<int>(q[idx - cn]);
                    float x;
                    if constexpr (BF16) {
                        x = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(stage)[loc]) << 16);
                    } else {
                        x = reinterpret_cast<const float*>(stage)[loc];
                    }
                    const bool pen = PENALTY && ((bm[loc >> 5] >> (loc & 31)) & 1u);
                    zb = transform_f32<SOFTCAP, PENALTY>(x, pen, P) * P.invT;
                    v = v0 + loc;
                }
            };
            int base = 0;
            while (total - base >= 32 || (flush && base < total)) {
                const int idx = base + lane;
                float zb = -INFINITY;
                int v = 0;
                if (idx < total) fetch(idx, zb, v);
                const bool live = idx < total && v != excl && zb + kGumbelMax >= thr;
                if (__any_sync(0xffffffffu, live)) {
                    const uint32_t word = pick_word(gumbel_block_row(rp, static_cast<uint32_t>(v) >> 2),
                                                    static_cast<uint32_t>(v) & 3u);
                    if (live && gumbel_may_reach(word, thr - zb)) {
                        const float score = zb + gumbel_f32(word);
                        if (score >= thr) {
                            top2_push(tt, score, v);
                            thr = fmaxf(thr, tt.s1 - cand_delta(tt.s1));
                        }
                    }
                }
                base += 32;
            }
            const int rem = total - base;  // < 32; 0 after a flush
            if (rem > 0) {
                float zc = 0.0f;
                int vc = 0;
                if (lane < rem) fetch(base + lane, zc, vc);
                __syncwarp();
                if (lane < rem) {
                    cz[lane] = zc;
                    cv[lane] = vc;
                }
            }
            cn = rem > 0 ? rem : 0;
            __syncwarp();
            if (lane == 0) s_qn[warp] = 0;
            __syncwarp();
            // share the warp's best score with the CTA, adopt the CTA's best
            const unsigned kw = warp_best_key(tt.s1);
            if (kw != 0u) {
                const float bw = key_score(kw);
                thr = fmaxf(thr, bw - cand_delta(bw));
                if (lane == 0) atomicMax(rth, kw);
            }
            }  // cand
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
                if (lane == 0) {
                    // keyed by the segment's last chunk; a written partial is never all-zero
                    st_partial(P.part + static_cast<size_t>(row) * P.nchunk + mt.c, GREEDY ? 0.0f : cm,
                               GREEDY ? 1.0f : cs, ct);
                    s_cnt[st] = 0;
                    *rth = 0u;  // every warp is past this segment: the slot is free
                }
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
    }
}

// ---------------------------------------------------------------- K3
// One warp per row: combine the row's chunk partials (log-sum-exp, sampled
// candidate), run the accept test of the draft it verifies; the last row of
// a sequence to finish runs the epilogue (tokens, kv_len, EMA).

template <bool BF16, bool GREEDY, bool SOFTCAP, bool PENALTY>
__global__ void __launch_bounds__(256) verify_merge_kernel(const VerifyDev P) {
    const int lane = threadIdx.x & 31;
    const int K1 = P.K + 1;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= P.B * K1) return;
    const int b = row / K1, j = row - b * K1;
    int kb;
    const int keff = gate_keff(P, b, &kb, false);
    if (j > keff) return;
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
    // other slots are all-zero (a written partial never is).  A lane holds at
    // most a few of them (chunks <= 32 for V <= 2^18 bf16 / 2^17 fp32).
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
                    const uint4 w = gumbel_block(nk, static_cast<uint32_t>(id) >> 2, static_cast<uint32_t>(j));
                    sc[h] = z / P.Td + gumbel_f64(pick_word(w, static_cast<uint32_t>(id) & 3u));
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

// ---------------------------------------------------------------- K2
// Dense draft distributions: after a rejection at row a, sample from the
// residual max(0, p_a - q_a) by Gumbel-max over row a (the logits of row a
// read once more and q_a read at the candidates only, for the rejected
// sequences).  log r_v <= log p_v = z_v / T - lse, so an element can beat
// the threshold only if z_v / T - lse + g_max reaches it.  The threshold
// starts from the exact residual score of the row's bonus sample (when its
// residual is positive) and is shared by the CTA's warps and, through the
// workspace, by the CTAs of the row.

// log max(0, p - q) for log p = lp, in fp32 without cancellation: for q > 0,
// p - q = q (e^(lp - ln q) - 1), and expm1 keeps the relative accuracy when
// p and q are close.  -inf when the residual is zero.
__device__ __forceinline__ float log_residual(float lp, float q) {
    if (!(q > 0.0f)) return lp;
    const float d = lp - logf(q);
    if (!(d > 0.0f)) return -INFINITY;
    return logf(q) + logf(expm1f(d));
}

template <bool BF16, bool SOFTCAP, bool PENALTY>
__global__ void __launch_bounds__(kThreads, 2) verify_residual_kernel(const VerifyDev P) {
    constexpr int EPV = ElemTraits<BF16>::EPV;
    constexpr int CHUNK = chunk_elems<BF16>();
    __shared__ uint32_t s_bm[PENALTY ? CHUNK / 32 : 1];
    __shared__ int s_win[PENALTY ? SPECNG_MAX_REP_WINDOW : 1];
    __shared__ int s_nwin;
    __shared__ Top2 s_t[kWarps];
    __shared__ int s_last;
    __shared__ unsigned s_thr;
    __shared__ uint16_t s_q2[kWarps * 32 * kNV * EPV];  // per-warp candidate queues (chunk offsets)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K1 = P.K + 1;
    const int b = blockIdx.x / P.nchunk;
    const int c = blockIdx.x - b * P.nchunk;
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
            const unsigned pb = pen_bits<PENALTY, EPV>(s_bm, off);
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
                t0 = lr + gumbel_f32(pick_word(gumbel_block_row(rp, static_cast<uint32_t>(im) >> 2),
                                               static_cast<uint32_t>(im) & 3u));
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
    // ---- candidates: log r_v <= lp_v, so lp_v + g_max must reach the threshold.  They
    //      are compacted per warp (chunk offsets), then scored 32 at a time, so the
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
            const unsigned pb = pen_bits<PENALTY, EPV>(s_bm, off);
#pragma unroll
            for (int e = 0; e < EPV; ++e)
                if (e < nv && !(lp_of(x[e], (pb >> e) & 1u) + kGumbelMax < thr) && v0 + off + e != seeded) mi |= 1u << e;
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
        const float lp = lp_of(x, pen);
        const float lr = in && !(lp + kGumbelMax < thr) ? log_residual(lp, qv) : -INFINITY;
        const bool live = lr > -INFINITY;
        if (__any_sync(0xffffffffu, live)) {
            const uint32_t word = pick_word(gumbel_block_row(rp, static_cast<uint32_t>(v) >> 2),
                                            static_cast<uint32_t>(v) & 3u);
            if (live && gumbel_may_reach(word, thr - lr - 1e-4f)) {
                const float score = lr + gumbel_f32(word);
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
            s_last = prev == static_cast<unsigned>(P.nchunk - 1);
        }
    }
    __syncthreads();
    if (!s_last || warp != 0) return;
    __threadfence();
    if (lane == 0) {
        P.seq_ticket2[b] = 0u;
        P.row_thr[row] = 0u;  // leave the workspace zeroed
    }
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
