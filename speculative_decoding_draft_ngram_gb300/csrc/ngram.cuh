// N-gram table kernels (sm_103a).
//
// AX Engine page, "Core Technical Architecture & Methods": bigram and
// trigram tables are built at runtime and predict up to 4 draft tokens per
// step.  The best continuation of a context is the most frequent one, equal
// counts going to the most recent occurrence; lookups try the trigram
// context first and fall back to the bigram context.
//
// Layout: four open-addressed, linearly probed tables of 16-byte slots
// {key, value} in HBM, keyed per sequence:
//   trigram pair   key = b:9 | t2:18 | t1:18 | c:18   value = count:32 | last:32
//   bigram pair    key = b:9 | t1:18 | c:18           value = count:32 | last:32
//   trigram ctx    key = b:9 | t2:18 | t1:18          value = best (packed)
//   bigram ctx     key = b:9 | t1:18                  value = best (packed)
// with EMPTY = ~0 (no real key has its top bit set).  A context's packed
// best is count:22 | last:24 | token:18; as counts and latest positions only
// grow, the atomic maximum over every update of its pairs is the maximum
// over its pairs, whatever the order of the updates.  So an update is two
// kernels: count the new pairs (atomicAdd / atomicMax), then push each
// touched pair's packed value into its context (atomicMax).
#pragma once

#include "common.cuh"

namespace specng {

constexpr uint64_t kEmptyKey = ~0ull;

struct NgramDev {
    ulonglong2* tri_pair;
    ulonglong2* bi_pair;
    ulonglong2* tri_ctx;
    ulonglong2* bi_ctx;
    uint64_t mask;            // slots - 1 (slots a power of two)
    int32_t* indexed[2];      // per-sequence indexed length; [1]: ngram_update's new lengths until copied to [0]
    int B, V;
    unsigned* status;
    uint64_t min_count;       // a context drafts only a best continuation seen this often (>= 1)
};

__device__ __forceinline__ uint64_t key_tri_pair(uint64_t b, uint64_t t2, uint64_t t1, uint64_t c) {
    return (b << 54) | (t2 << 36) | (t1 << 18) | c;
}
__device__ __forceinline__ uint64_t key_bi_pair(uint64_t b, uint64_t t1, uint64_t c) {
    return (b << 36) | (t1 << 18) | c;
}
__device__ __forceinline__ uint64_t key_tri_ctx(uint64_t b, uint64_t t2, uint64_t t1) {
    return (b << 36) | (t2 << 18) | t1;
}
__device__ __forceinline__ uint64_t key_bi_ctx(uint64_t b, uint64_t t1) { return (b << 18) | t1; }

constexpr uint64_t kCountMax = (1ull << 22) - 1;

__device__ __forceinline__ uint64_t pack_best(uint64_t count, uint64_t last, uint64_t token) {
    return (count << 42) | (last << 18) | token;
}
__device__ __forceinline__ int best_token(uint64_t v) { return static_cast<int>(v & 0x3FFFFull); }
// The best continuation's token when its count reaches min_count, else -1.
__device__ __forceinline__ int best_token_if(uint64_t v, uint64_t min_count) {
    return (v >> 42) >= min_count ? best_token(v) : -1;
}

// Slot holding key (inserted if absent), or -1 when the table is full.
__device__ __forceinline__ int64_t find_or_insert(ulonglong2* tab, uint64_t mask, uint64_t key) {
    uint64_t slot = mix64(key) & mask;
    for (uint64_t probe = 0; probe <= mask; ++probe) {
        unsigned long long* kp = &tab[slot].x;
        const uint64_t k = *reinterpret_cast<volatile unsigned long long*>(kp);
        if (k == key) return static_cast<int64_t>(slot);
        if (k == kEmptyKey) {
            const uint64_t prev = atomicCAS(kp, kEmptyKey, key);
            if (prev == kEmptyKey || prev == key) return static_cast<int64_t>(slot);
        }
        slot = (slot + 1) & mask;
    }
    return -1;
}

// Value stored under key, or false when absent (read-only probe).
__device__ __forceinline__ bool find_value(const ulonglong2* tab, uint64_t mask, uint64_t key, uint64_t* val) {
    uint64_t slot = mix64(key) & mask;
    for (uint64_t probe = 0; probe <= mask; ++probe) {
        const ulonglong2 e = __ldcg(&tab[slot]);
        if (e.x == key) { *val = e.y; return true; }
        if (e.x == kEmptyKey) return false;
        slot = (slot + 1) & mask;
    }
    return false;
}

cudaError_t launch_ngram_update(const NgramDev& T, const int32_t* hist, int64_t stride,
                                const int32_t* lens, int grid, cudaStream_t s);
cudaError_t launch_ngram_draft(const NgramDev& T, const int32_t* hist, int64_t stride, const int32_t* lens,
                               int max_k, const int32_t* k_limit, const int32_t* fallback, int32_t* out_drafts,
                               int32_t* out_k, cudaStream_t s);
cudaError_t launch_ngram_clear(const NgramDev& T, cudaStream_t s);
cudaError_t launch_spec_append(int32_t* hist, int64_t stride, int32_t* lens, int64_t cap, const int32_t* out_tokens,
                               const int32_t* out_accept, int B, int K, unsigned* status, cudaStream_t s);
cudaError_t launch_spec_commit(const NgramDev& T, int32_t* hist, int64_t stride, int32_t* lens,
                               int64_t cap, const int32_t* out_tokens, const int32_t* out_accept, int K, int max_k,
                               const int32_t* k_limit, const int32_t* fallback, int32_t* out_drafts, int32_t* out_k,
                               cudaStream_t s);
cudaError_t launch_philox(const uint32_t* ctr, uint64_t seed, uint32_t* out, int64_t n, cudaStream_t s);

}  // namespace specng
