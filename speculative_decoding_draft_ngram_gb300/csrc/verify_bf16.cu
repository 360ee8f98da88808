// Instantiation and dispatch of the spec_verify kernels for bf16 logits.
#include "verify.cuh"

namespace specng {

namespace {

int sm_count() {
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

template <bool G, bool C, bool R>
cudaError_t launch_k1_k3(const VerifyDev& P, cudaStream_t s) {
    // K1: one persistent CTA per SM; the staging ring lives in dynamic shared memory
    constexpr size_t smem = k1_dyn_smem<R>();
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(verify_stream_kernel<true, G, C, R>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    verify_stream_kernel<true, G, C, R><<<sm_count(), kPThreads, smem, s>>>(P);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // K3: one warp per row
    const unsigned rows = static_cast<unsigned>(P.B) * static_cast<unsigned>(P.K + 1);
    verify_merge_kernel<true, G, C, R><<<(rows + 7) / 8, 256, 0, s>>>(P);
    return cudaGetLastError();
}

template <bool C, bool R>
cudaError_t launch_k2(const VerifyDev& P, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>(P.B) * static_cast<unsigned>(P.nchunk);
    verify_residual_kernel<true, C, R><<<grid, kThreads, 0, s>>>(P);
    return cudaGetLastError();
}

template <bool G>
cudaError_t k1_cr(const VerifyDev& P, bool c, bool r, cudaStream_t s) {
    if (c) return r ? launch_k1_k3<G, true, true>(P, s) : launch_k1_k3<G, true, false>(P, s);
    return r ? launch_k1_k3<G, false, true>(P, s) : launch_k1_k3<G, false, false>(P, s);
}

}  // namespace

template <>
cudaError_t launch_verify_dtype<true>(const VerifyDev& P, bool greedy, bool softcap, bool penalty, bool dense,
                                     cudaStream_t s) {
    cudaError_t e = greedy ? k1_cr<true>(P, softcap, penalty, s) : k1_cr<false>(P, softcap, penalty, s);
    if (e != cudaSuccess || !dense || greedy) return e;
    if (softcap) return penalty ? launch_k2<true, true>(P, s) : launch_k2<true, false>(P, s);
    return penalty ? launch_k2<false, true>(P, s) : launch_k2<false, false>(P, s);
}

}  // namespace specng
