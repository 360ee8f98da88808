// Instantiation and dispatch of the spec_verify kernels for f32 logits.
#include "verify.cuh"

namespace specng {

namespace {

template <bool G, bool C, bool R>
cudaError_t launch_k1(const VerifyDev& P, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>(P.B) * static_cast<unsigned>(P.K + 1) * static_cast<unsigned>(P.nchunk);
    verify_stream_kernel<false, G, C, R><<<grid, kThreads, 0, s>>>(P);
    return cudaGetLastError();
}

template <bool C, bool R>
cudaError_t launch_k2(const VerifyDev& P, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>(P.B) * static_cast<unsigned>(P.nchunk);
    verify_residual_kernel<false, C, R><<<grid, kThreads, 0, s>>>(P);
    return cudaGetLastError();
}

template <bool G>
cudaError_t k1_cr(const VerifyDev& P, bool c, bool r, cudaStream_t s) {
    if (c) return r ? launch_k1<G, true, true>(P, s) : launch_k1<G, true, false>(P, s);
    return r ? launch_k1<G, false, true>(P, s) : launch_k1<G, false, false>(P, s);
}

}  // namespace

template <>
cudaError_t launch_verify_dtype<false>(const VerifyDev& P, bool greedy, bool softcap, bool penalty, bool dense,
                                     cudaStream_t s) {
    cudaError_t e = greedy ? k1_cr<true>(P, softcap, penalty, s) : k1_cr<false>(P, softcap, penalty, s);
    if (e != cudaSuccess || !dense || greedy) return e;
    if (softcap) return penalty ? launch_k2<true, true>(P, s) : launch_k2<true, false>(P, s);
    return penalty ? launch_k2<false, true>(P, s) : launch_k2<false, false>(P, s);
}

}  // namespace specng
