// KV block pool bookkeeping and the device decode-step counter (sm_103a).
//
// [AX] "Core Technical Architecture & Methods": the KV cache grows inside
// preallocated buffers and a speculation rollback only moves the sequence
// length (spec_verify's kv_len update); the scheduler recovers memory blocks.
// Here the preallocated buffer is a pool of fixed-size blocks: a stack of free
// block ids and, per sequence, a table of its blocks in position order.  A
// kernel either only takes blocks from the stack or only returns them, so the
// stack needs one atomic counter and no lock.
#include "kv.cuh"

#include "common.cuh"

namespace specng {

namespace {

constexpr int kKvThreads = 256;

__device__ __forceinline__ int blocks_for(int len, int bs) {
    if (len < 0) len = 0;
    return static_cast<int>((static_cast<long long>(len) + bs - 1) / bs);
}

// Every block free: the stack holds num_blocks - 1, ..., 0 from the bottom, so
// blocks are handed out in increasing id order; every table row empty.
__global__ void kv_init_kernel(KvDev K) {
    const long long n = static_cast<long long>(K.B) * K.max_blocks;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        K.table[i] = -1;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < K.num_blocks;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        K.free_stack[i] = K.num_blocks - 1 - static_cast<int>(i);
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < K.B;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        K.nblocks[i] = 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) *K.free_top = K.num_blocks;
}

// Sequence b takes blocks until it holds enough for kv_len[b] + extra
// positions (one thread per sequence; blocks come off the stack top).
__global__ void kv_reserve_kernel(KvDev K, const int32_t* kv_len, int extra) {
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < K.B; b += gridDim.x * blockDim.x) {
    int want = blocks_for(kv_len[b] + extra, K.block_size);
    if (want > K.max_blocks) {
        raise_status(K.status, SPECNG_DEV_KV_SHORT);
        want = K.max_blocks;
    }
    int have = K.nblocks[b];
    int32_t* row = K.table + static_cast<size_t>(b) * K.max_blocks;
    while (have < want) {
        const int slot = atomicSub(K.free_top, 1) - 1;
        if (slot < 0) {
            atomicAdd(K.free_top, 1);  // the pool is empty: give the slot back
            raise_status(K.status, SPECNG_DEV_KV_SHORT);
            break;
        }
        row[have++] = K.free_stack[slot];
    }
    K.nblocks[b] = have;
    }
}

// Blocks of sequence b past the ones its kv_len[b] positions need go back to
// the stack (drop == nullptr), or all its blocks when drop[b] != 0 (release).
__global__ void kv_return_kernel(KvDev K, const int32_t* kv_len, const int32_t* drop) {
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < K.B; b += gridDim.x * blockDim.x) {
    const int have = K.nblocks[b];
    const int keep = drop != nullptr ? (drop[b] != 0 ? 0 : have) : min(have, blocks_for(kv_len[b], K.block_size));
    int32_t* row = K.table + static_cast<size_t>(b) * K.max_blocks;
    for (int n = keep; n < have; ++n) {
        const int slot = atomicAdd(K.free_top, 1);
        K.free_stack[slot] = row[n];
        row[n] = -1;
    }
    K.nblocks[b] = keep;
    }
}

__global__ void step_advance_kernel(uint64_t* step) { *step += 1; }

unsigned grid_for(long long n) {
    const long long g = (n + kKvThreads - 1) / kKvThreads;
    return static_cast<unsigned>(g < 1 ? 1 : (g > 4096 ? 4096 : g));
}

}  // namespace

cudaError_t launch_kv_init(const KvDev& K, cudaStream_t s) {
    long long n = static_cast<long long>(K.B) * K.max_blocks;
    if (K.num_blocks > n) n = K.num_blocks;
    kv_init_kernel<<<grid_for(n), kKvThreads, 0, s>>>(K);
    return cudaGetLastError();
}

cudaError_t launch_kv_reserve(const KvDev& K, const int32_t* kv_len, int extra, cudaStream_t s) {
    kv_reserve_kernel<<<grid_for(K.B), kKvThreads, 0, s>>>(K, kv_len, extra);
    return cudaGetLastError();
}

cudaError_t launch_kv_trim(const KvDev& K, const int32_t* kv_len, cudaStream_t s) {
    kv_return_kernel<<<grid_for(K.B), kKvThreads, 0, s>>>(K, kv_len, nullptr);
    return cudaGetLastError();
}

cudaError_t launch_kv_release(const KvDev& K, const int32_t* done, cudaStream_t s) {
    kv_return_kernel<<<grid_for(K.B), kKvThreads, 0, s>>>(K, nullptr, done);
    return cudaGetLastError();
}

cudaError_t launch_step_advance(uint64_t* step, cudaStream_t s) {
    step_advance_kernel<<<1, 1, 0, s>>>(step);
    return cudaGetLastError();
}

}  // namespace specng
