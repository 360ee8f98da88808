// Instantiation of the spec_verify kernels for f32 logits (one translation
// unit per dtype, so the two compile in parallel).
#include "verify.cuh"

namespace specng {

template <>
cudaError_t launch_verify_dtype<false>(const VerifyDev& P, bool greedy, bool softcap, bool penalty, bool dense,
                                     cudaStream_t s) {
    return launch_verify_impl<false>(P, greedy, softcap, penalty, dense, s);
}

}  // namespace specng
