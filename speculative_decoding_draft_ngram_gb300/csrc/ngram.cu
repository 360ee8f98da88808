// N-gram table update / draft kernels, the history append and the Philox
// diagnostic kernel (sm_103a).
#include "ngram.cuh"

namespace specng {

namespace {

constexpr int kNgThreads = 256;

// Exclusive prefix over the per-sequence counts of new positions, shared by
// both update phases.  Position i of sequence b is new when
// max(indexed_b, 1) <= i < min(lens_b, stride): position 0 has no context.
struct NewRange {
    long long* pref;  // [B + 1]
    int* lo;          // [B]
};

__device__ void build_new_range(const NgramDev& T, const int32_t* lens, int64_t stride,
                                long long* s_pref, int* s_lo, int* s_hi, bool flag) {
    __shared__ long long s_warp[kNgThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // each thread owns up to 2 consecutive sequences (B <= 512)
    long long n[2] = {0, 0};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int b = 2 * tid + h;
        if (b < T.B) {
            const int idx = T.indexed[0][b];
            int L = lens[b];
            if (L < 0) L = 0;
            if (static_cast<int64_t>(L) > stride) L = static_cast<int>(stride);
            if (flag && L < idx) raise_status(T.status, SPECNG_DEV_HIST_SHRANK);
            const int lo = idx > 1 ? idx : 1;
            s_lo[b] = lo;
            s_hi[b] = L;
            n[h] = L > lo ? L - lo : 0;
        }
    }
    long long v = n[0] + n[1];
    long long incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    long long base = 0;
    for (int w = 0; w < warp; ++w) base += s_warp[w];
    const long long excl = base + incl - v;
    if (2 * tid < T.B) s_pref[2 * tid] = excl;
    if (2 * tid + 1 < T.B) s_pref[2 * tid + 1] = excl + n[0];
    if (tid == kNgThreads - 1) s_pref[T.B] = base + incl;
    __syncthreads();
}

__device__ __forceinline__ int seq_of(const long long* s_pref, int B, long long f) {
    int lo = 0, hi = B;  // largest b with s_pref[b] <= f
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_pref[mid] <= f) lo = mid; else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ bool tok_ok(int t, int V) { return t >= 0 && t < V; }

__global__ void __launch_bounds__(kNgThreads) ngram_count_kernel(const NgramDev T, const int32_t* hist,
                                                                 int64_t stride, const int32_t* lens) {
    __shared__ long long s_pref[SPECNG_NGRAM_MAX_B + 1];
    __shared__ int s_lo[SPECNG_NGRAM_MAX_B], s_hi[SPECNG_NGRAM_MAX_B];
    build_new_range(T, lens, stride, s_pref, s_lo, s_hi, blockIdx.x == 0);
    const long long total = s_pref[T.B];
    for (long long f = static_cast<long long>(blockIdx.x) * kNgThreads + threadIdx.x; f < total;
         f += static_cast<long long>(gridDim.x) * kNgThreads) {
        const int b = seq_of(s_pref, T.B, f);
        const int i = s_lo[b] + static_cast<int>(f - s_pref[b]);
        const int32_t* h = hist + static_cast<size_t>(b) * stride;
        const int c = h[i], t1 = h[i - 1];
        if (!tok_ok(c, T.V) || !tok_ok(t1, T.V)) { raise_status(T.status, SPECNG_DEV_TOKEN_OOR); continue; }
        int64_t slot = find_or_insert(T.bi_pair, T.mask, key_bi_pair(b, t1, c));
        if (slot < 0) {
            raise_status(T.status, SPECNG_DEV_TABLE_FULL);
        } else {
            unsigned* v = reinterpret_cast<unsigned*>(&T.bi_pair[slot].y);
            atomicAdd(v, 1u);
            atomicMax(v + 1, static_cast<unsigned>(i));
        }
        if (i >= 2) {
            const int t2 = h[i - 2];
            if (!tok_ok(t2, T.V)) { raise_status(T.status, SPECNG_DEV_TOKEN_OOR); continue; }
            slot = find_or_insert(T.tri_pair, T.mask, key_tri_pair(b, t2, t1, c));
            if (slot < 0) {
                raise_status(T.status, SPECNG_DEV_TABLE_FULL);
            } else {
                unsigned* v = reinterpret_cast<unsigned*>(&T.tri_pair[slot].y);
                atomicAdd(v, 1u);
                atomicMax(v + 1, static_cast<unsigned>(i));
            }
        }
    }
}

__device__ __forceinline__ void push_best(const NgramDev& T, const ulonglong2* pairs, ulonglong2* ctxs,
                                          uint64_t pair_key, uint64_t ctx_key, int c) {
    // the context's home slot does not depend on the pair's value: start its
    // fetch into L2 now, so its probe below does not wait on HBM again
    asm volatile("prefetch.global.L2 [%0];" ::"l"(&ctxs[mix64(ctx_key) & T.mask]));
    uint64_t pv;
    if (!find_value(pairs, T.mask, pair_key, &pv)) return;  // insert failed in the count phase
    uint64_t count = pv & 0xFFFFFFFFull;
    const uint64_t last = pv >> 32;
    if (count > kCountMax) { raise_status(T.status, SPECNG_DEV_COUNT_SAT); count = kCountMax; }
    const int64_t slot = find_or_insert(ctxs, T.mask, ctx_key);
    if (slot < 0) { raise_status(T.status, SPECNG_DEV_TABLE_FULL); return; }
    atomicMax(&ctxs[slot].y, static_cast<unsigned long long>(pack_best(count, last, static_cast<uint64_t>(c))));
}

__global__ void __launch_bounds__(kNgThreads) ngram_best_kernel(const NgramDev T, const int32_t* hist,
                                                                int64_t stride, const int32_t* lens) {
    __shared__ long long s_pref[SPECNG_NGRAM_MAX_B + 1];
    __shared__ int s_lo[SPECNG_NGRAM_MAX_B], s_hi[SPECNG_NGRAM_MAX_B];
    build_new_range(T, lens, stride, s_pref, s_lo, s_hi, false);
    const long long total = s_pref[T.B];
    for (long long f = static_cast<long long>(blockIdx.x) * kNgThreads + threadIdx.x; f < total;
         f += static_cast<long long>(gridDim.x) * kNgThreads) {
        const int b = seq_of(s_pref, T.B, f);
        const int i = s_lo[b] + static_cast<int>(f - s_pref[b]);
        const int32_t* h = hist + static_cast<size_t>(b) * stride;
        const int c = h[i], t1 = h[i - 1];
        if (!tok_ok(c, T.V) || !tok_ok(t1, T.V)) continue;
        push_best(T, T.bi_pair, T.bi_ctx, key_bi_pair(b, t1, c), key_bi_ctx(b, t1), c);
        if (i >= 2) {
            const int t2 = h[i - 2];
            if (!tok_ok(t2, T.V)) continue;
            push_best(T, T.tri_pair, T.tri_ctx, key_tri_pair(b, t2, t1, c), key_tri_ctx(b, t2, t1), c);
        }
    }
    // the lengths indexed now go to the second buffer (every block of this
    // launch reads the first); the next launch copies them over
    if (blockIdx.x == 0) {
        for (int b = threadIdx.x; b < T.B; b += kNgThreads) {
            const int idx = T.indexed[0][b];
            T.indexed[1][b] = s_hi[b] > idx ? s_hi[b] : idx;
        }
    }
}

// The indexed lengths of ngram_update take effect (second buffer to first).
// The kernels keep no state on the host, so a captured step replays right.
__global__ void ngram_indexed_kernel(const NgramDev T) {
    for (int b = threadIdx.x; b < T.B; b += blockDim.x) T.indexed[0][b] = T.indexed[1][b];
}

__device__ void draft_one(const NgramDev& T, int b, const int32_t* h, int L, int max_k, const int32_t* k_limit,
                          const int32_t* fallback, int32_t* out_drafts, int32_t* out_k);

__global__ void __launch_bounds__(kNgThreads) ngram_draft_kernel(const NgramDev T, const int32_t* hist, int64_t stride,
                                                                 const int32_t* lens, int max_k, const int32_t* k_limit,
                                                                 const int32_t* fallback, int32_t* out_drafts,
                                                                 int32_t* out_k) {
    const int b = blockIdx.x * kNgThreads + threadIdx.x;
    if (b >= T.B) return;
    int L = lens[b];
    if (L < 0) L = 0;
    if (static_cast<int64_t>(L) > stride) L = static_cast<int>(stride);
    draft_one(T, b, hist + static_cast<size_t>(b) * stride, L, max_k, k_limit, fallback, out_drafts, out_k);
}

__global__ void ngram_clear_kernel(const NgramDev T) {
    const uint64_t slots = T.mask + 1;
    const ulonglong2 empty = make_ulonglong2(kEmptyKey, 0ull);
    for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < slots;
         i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        T.tri_pair[i] = empty;
        T.bi_pair[i] = empty;
        T.tri_ctx[i] = empty;
        T.bi_ctx[i] = empty;
    }
    if (blockIdx.x == 0) {
        for (int b = threadIdx.x; b < T.B; b += blockDim.x) { T.indexed[0][b] = 0; T.indexed[1][b] = 0; }
    }
}

__global__ void spec_append_kernel(int32_t* hist, int64_t stride, int32_t* lens, int64_t cap, const int32_t* out_tokens,
                                   const int32_t* out_accept, int B, int K, unsigned* status) {
    pdl_wait();  // the verify kernels' tokens
    pdl_trigger();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int a = out_accept[b];
    if (a < 0 || a > K) { raise_status(status, SPECNG_DEV_BAD_K); return; }
    const int L = lens[b];
    if (L < 0 || static_cast<int64_t>(L) + a + 1 > cap) { raise_status(status, SPECNG_DEV_HIST_OVERFLOW); return; }
    int32_t* h = hist + static_cast<size_t>(b) * stride + L;
    const int32_t* t = out_tokens + static_cast<size_t>(b) * (K + 1);
    for (int i = 0; i <= a; ++i) h[i] = t[i];
    lens[b] = L + a + 1;
}

// Chained trigram -> bigram drafts of sequence b (one thread), as ngram_draft_kernel.
__device__ void draft_one(const NgramDev& T, int b, const int32_t* h, int L, int max_k, const int32_t* k_limit,
                          const int32_t* fallback, int32_t* out_drafts, int32_t* out_k) {
    int kmax = max_k;
    if (k_limit != nullptr) {
        const int kl = k_limit[b];
        kmax = kl < 0 ? 0 : (kl < kmax ? kl : kmax);
    }
    int c2 = L >= 2 ? h[L - 2] : -1;
    int c1 = L >= 1 ? h[L - 1] : -1;
    if ((L >= 2 && !tok_ok(c2, T.V)) || (L >= 1 && !tok_ok(c1, T.V))) raise_status(T.status, SPECNG_DEV_TOKEN_OOR);
    if (!tok_ok(c2, T.V)) c2 = -1;
    if (!tok_ok(c1, T.V)) c1 = -1;
    int n = 0;
    int32_t* out = out_drafts + static_cast<size_t>(b) * max_k;
    while (n < kmax && c1 >= 0) {
        int tok = -1;
        uint64_t v;
        if (c2 >= 0 && find_value(T.tri_ctx, T.mask, key_tri_ctx(b, c2, c1), &v)) tok = best_token_if(v, T.min_count);
        if (tok < 0 && find_value(T.bi_ctx, T.mask, key_bi_ctx(b, c1), &v)) tok = best_token_if(v, T.min_count);
        if (tok < 0) break;
        out[n++] = tok;
        c2 = c1;
        c1 = tok;
    }
    if (fallback != nullptr) {
        const int32_t* fb = fallback + static_cast<size_t>(b) * max_k;
        for (; n < kmax; ++n) out[n] = fb[n];
    }
    for (int t = n; t < max_k; ++t) out[t] = -1;
    out_k[b] = n;
}

// The same drafts as draft_one, by a whole warp: at every draft position the
// trigram probe (lane 0) and the bigram probe (lane 1) are in flight together,
// so a position costs one probe latency, not two.
__device__ void draft_warp(const NgramDev& T, int b, const int32_t* h, int L, int max_k, const int32_t* k_limit,
                           const int32_t* fallback, int32_t* out_drafts, int32_t* out_k) {
    const int lane = threadIdx.x & 31;
    int kmax = max_k;
    if (k_limit != nullptr) {
        const int kl = k_limit[b];
        kmax = kl < 0 ? 0 : (kl < kmax ? kl : kmax);
    }
    int c2 = L >= 2 ? h[L - 2] : -1;
    int c1 = L >= 1 ? h[L - 1] : -1;
    if (lane == 0 && ((L >= 2 && !tok_ok(c2, T.V)) || (L >= 1 && !tok_ok(c1, T.V))))
        raise_status(T.status, SPECNG_DEV_TOKEN_OOR);
    if (!tok_ok(c2, T.V)) c2 = -1;
    if (!tok_ok(c1, T.V)) c1 = -1;
    int n = 0;
    int32_t* out = out_drafts + static_cast<size_t>(b) * max_k;
    while (n < kmax && c1 >= 0) {  // warp-uniform
        int tok = -1;
        uint64_t v;
        if (lane == 0 && c2 >= 0 && find_value(T.tri_ctx, T.mask, key_tri_ctx(b, c2, c1), &v))
            tok = best_token_if(v, T.min_count);
        if (lane == 1 && find_value(T.bi_ctx, T.mask, key_bi_ctx(b, c1), &v)) tok = best_token_if(v, T.min_count);
        const int tt = __shfl_sync(0xffffffffu, tok, 0), tb = __shfl_sync(0xffffffffu, tok, 1);
        tok = tt >= 0 ? tt : tb;
        if (tok < 0) break;
        if (lane == 0) out[n] = tok;
        ++n;
        c2 = c1;
        c1 = tok;
    }
    int nf = n;
    if (fallback != nullptr) {
        const int32_t* fb = fallback + static_cast<size_t>(b) * max_k;
        for (int t = n + lane; t < kmax; t += 32) out[t] = fb[t];
        nf = n > kmax ? n : kmax;
    }
    for (int t = nf + lane; t < max_k; t += 32) out[t] = -1;
    if (lane == 0) out_k[b] = nf;
}

// One step's commit for every sequence, one warp per sequence: append the
// emitted tokens (spec_append), index the new positions (ngram_update: pair
// counts, then the contexts' best continuations) and draft the next step
// (ngram_draft).  A sequence's keys belong to it alone, so the warp needs no
// other sequence's work: __syncwarp orders its phases.  The tokens around the
// appended positions are kept in shared memory, and each pair's count and
// latest position are updated by one 64-bit compare-and-swap whose result
// feeds the context's best continuation at once: the state a lane produces is
// never above the pair's final state, and pack_best grows with the count, so
// the context's atomic maximum ends at what the final state gives.
constexpr int kTailTok = SPECNG_MAX_K + 3;  // the two tokens before the appended ones, then those

__global__ void __launch_bounds__(kNgThreads) spec_commit_kernel(const NgramDev T, int32_t* hist,
                                                                 int64_t stride, int32_t* lens, int64_t cap,
                                                                 const int32_t* out_tokens, const int32_t* out_accept,
                                                                 int K, int max_k, const int32_t* k_limit,
                                                                 const int32_t* fallback, int32_t* out_drafts,
                                                                 int32_t* out_k) {
    __shared__ int s_tail[kNgThreads / 32][kTailTok];
    pdl_wait();  // the verify kernels' tokens
    pdl_trigger();
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int b = blockIdx.x * (kNgThreads / 32) + wib;
    if (b >= T.B) return;
    int32_t* h = hist + static_cast<size_t>(b) * stride;
    int* tail = s_tail[wib];
    // ---- append
    int L = lens[b];
    const int a = out_accept[b];
    const int L0 = L;       // first appended position (tail[2 + t] holds position L0 + t)
    bool appended = false;  // the tail holds positions L0 - 2 .. L0 + a
    if (a < 0 || a > K) {
        if (lane == 0) raise_status(T.status, SPECNG_DEV_BAD_K);
    } else if (L < 0 || static_cast<int64_t>(L) + a + 1 > cap) {
        if (lane == 0) raise_status(T.status, SPECNG_DEV_HIST_OVERFLOW);
    } else {
        if (lane <= a) {
            const int t = out_tokens[static_cast<size_t>(b) * (K + 1) + lane];
            h[L + lane] = t;
            tail[2 + lane] = t;
        }
        if (lane < 2) tail[lane] = L - 2 + lane >= 0 ? h[L - 2 + lane] : -1;
        L += a + 1;
        if (lane == 0) lens[b] = L;
        appended = true;
    }
    __syncwarp();
    // ---- index positions [max(indexed, 1), L)
    if (L < 0) L = 0;
    if (static_cast<int64_t>(L) > stride) L = static_cast<int>(stride);
    const int idx = T.indexed[0][b];  // this warp alone reads and writes entry b
    if (L < idx && lane == 0) raise_status(T.status, SPECNG_DEV_HIST_SHRANK);
    const int lo = idx > 1 ? idx : 1;
    auto tok_at = [&](int i) {  // the token at position i (the appended ones and the two before from shared memory)
        return (appended && i >= L0 - 2 && i - (L0 - 2) < a + 3) ? tail[i - (L0 - 2)] : h[i];
    };
    // half-warps: the bigram pairs on lanes 0..15, the trigram pairs on lanes 16..31,
    // so the two probe chains of a position run side by side
    const bool tri = lane >= 16;
    for (int i = lo + (lane & 15); i < L; i += 16) {
        if (tri && i < 2) continue;
        const int c = tok_at(i), t1 = tok_at(i - 1), t2 = tri ? tok_at(i - 2) : 0;
        if (!tok_ok(c, T.V) || !tok_ok(t1, T.V) || (tri && !tok_ok(t2, T.V))) {
            raise_status(T.status, SPECNG_DEV_TOKEN_OOR);
            continue;
        }
        ulonglong2* tab = tri ? T.tri_pair : T.bi_pair;
        ulonglong2* ctxs = tri ? T.tri_ctx : T.bi_ctx;
        const uint64_t ctx_key = tri ? key_tri_ctx(b, t2, t1) : key_bi_ctx(b, t1);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(&ctxs[mix64(ctx_key) & T.mask]));
        const int64_t slot = find_or_insert(tab, T.mask, tri ? key_tri_pair(b, t2, t1, c) : key_bi_pair(b, t1, c));
        if (slot < 0) {
            raise_status(T.status, SPECNG_DEV_TABLE_FULL);
            continue;
        }
        // count:32 | last:32, both at once
        unsigned long long* vp = &tab[slot].y;
        unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(vp), nxt;
        for (;;) {
            const uint64_t cnt = (cur & 0xFFFFFFFFull) + 1ull;
            const uint64_t lst = (cur >> 32) > static_cast<uint64_t>(i) ? (cur >> 32) : static_cast<uint64_t>(i);
            nxt = (lst << 32) | (cnt & 0xFFFFFFFFull);
            const unsigned long long prev = atomicCAS(vp, cur, nxt);
            if (prev == cur) break;
            cur = prev;
        }
        uint64_t count = nxt & 0xFFFFFFFFull;
        if (count > kCountMax) { raise_status(T.status, SPECNG_DEV_COUNT_SAT); count = kCountMax; }
        const int64_t cs = find_or_insert(ctxs, T.mask, ctx_key);
        if (cs < 0) { raise_status(T.status, SPECNG_DEV_TABLE_FULL); continue; }
        atomicMax(&ctxs[cs].y, static_cast<unsigned long long>(pack_best(count, nxt >> 32, static_cast<uint64_t>(c))));
    }
    __syncwarp();
    if (lane == 0) T.indexed[0][b] = L > idx ? L : idx;
    // ---- the next step's drafts
    draft_warp(T, b, h, L, max_k, k_limit, fallback, out_drafts, out_k);
}

__global__ void philox_kernel(const uint4* ctr, uint32_t k0, uint32_t k1, uint4* out, int64_t n) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        out[i] = philox4x32_10(ctr[i], k0, k1);
}

}  // namespace

cudaError_t launch_ngram_update(const NgramDev& T, const int32_t* hist, int64_t stride,
                                const int32_t* lens, int grid, cudaStream_t s) {
    ngram_count_kernel<<<grid, kNgThreads, 0, s>>>(T, hist, stride, lens);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ngram_best_kernel<<<grid, kNgThreads, 0, s>>>(T, hist, stride, lens);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ngram_indexed_kernel<<<1, kNgThreads, 0, s>>>(T);
    return cudaGetLastError();
}

cudaError_t launch_ngram_draft(const NgramDev& T, const int32_t* hist, int64_t stride, const int32_t* lens,
                               int max_k, const int32_t* k_limit, const int32_t* fallback, int32_t* out_drafts,
                               int32_t* out_k, cudaStream_t s) {
    const int grid = (T.B + kNgThreads - 1) / kNgThreads;
    ngram_draft_kernel<<<grid, kNgThreads, 0, s>>>(T, hist, stride, lens, max_k, k_limit, fallback, out_drafts,
                                                   out_k);
    return cudaGetLastError();
}

cudaError_t launch_ngram_clear(const NgramDev& T, cudaStream_t s) {
    const uint64_t slots = T.mask + 1;
    uint64_t blocks = (slots + 255) / 256;
    if (blocks > 65536) blocks = 65536;
    ngram_clear_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(T);
    return cudaGetLastError();
}

cudaError_t launch_spec_append(int32_t* hist, int64_t stride, int32_t* lens, int64_t cap, const int32_t* out_tokens,
                               const int32_t* out_accept, int B, int K, unsigned* status, cudaStream_t s) {
    return launch_chained(spec_append_kernel, dim3((B + 127) / 128), dim3(128), 0, s, hist, stride, lens, cap, out_tokens,
                          out_accept, B, K, status);
}

cudaError_t launch_spec_commit(const NgramDev& T, int32_t* hist, int64_t stride, int32_t* lens,
                               int64_t cap, const int32_t* out_tokens, const int32_t* out_accept, int K, int max_k,
                               const int32_t* k_limit, const int32_t* fallback, int32_t* out_drafts, int32_t* out_k,
                               cudaStream_t s) {
    const int per = kNgThreads / 32;
    return launch_chained(spec_commit_kernel, dim3((T.B + per - 1) / per), dim3(kNgThreads), 0, s, T, hist, stride,
                          lens, cap, out_tokens, out_accept, K, max_k, k_limit, fallback, out_drafts, out_k);
}

cudaError_t launch_philox(const uint32_t* ctr, uint64_t seed, uint32_t* out, int64_t n, cudaStream_t s) {
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    philox_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(reinterpret_cast<const uint4*>(ctr),
                                                                static_cast<uint32_t>(seed),
                                                                static_cast<uint32_t>(seed >> 32),
                                                                reinterpret_cast<uint4*>(out), n);
    return cudaGetLastError();
}

}  // namespace specng
