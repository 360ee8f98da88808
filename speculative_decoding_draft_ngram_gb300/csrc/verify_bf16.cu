// Instantiation of the spec_verify kernels for bf16 logits (one translation
// unit per dtype, so the two compile in parallel).
#include "verify.cuh"

namespace specng {

template <>
cudaError_t launch_verify_dtype<true>(const VerifyDev& P, bool greedy, bool softcap, bool penalty, bool dense,
                                     cudaStream_t s) {
    return launch_verify_impl<true>(P, greedy, softcap, penalty, dense, s);
}

}  // namespace specng
