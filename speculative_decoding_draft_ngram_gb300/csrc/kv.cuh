// KV block pool bookkeeping and the device decode-step counter (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

#include "specng.h"

namespace specng {

// Device view of a specng_kv_pool plus the status word.
struct KvDev {
    int32_t* free_stack;  // [num_blocks]: free block ids at [0, *free_top)
    int32_t* free_top;
    int32_t* table;       // [B, max_blocks]
    int32_t* nblocks;     // [B]
    int num_blocks, B, max_blocks, block_size;
    unsigned* status;
};

cudaError_t launch_kv_init(const KvDev& K, cudaStream_t s);
cudaError_t launch_kv_reserve(const KvDev& K, const int32_t* kv_len, int extra, cudaStream_t s);
cudaError_t launch_kv_trim(const KvDev& K, const int32_t* kv_len, cudaStream_t s);
cudaError_t launch_kv_release(const KvDev& K, const int32_t* done, cudaStream_t s);
cudaError_t launch_step_advance(uint64_t* step, cudaStream_t s);

}  // namespace specng
