// kf_decode_tc_fp8.cu -- FP8 E4M3-cache instantiations of the tensor-core
// decode kernel (kf_decode_tc.cuh).
#include "kf_decode_tc.cuh"

namespace kf {

cudaError_t launch_decode_tc_fp8(const DecodeParams &p, cudaStream_t stream, void *encode) {
    tc::StepParams sp = {};
    return tc::launch_any<false, true>(p, sp, stream, encode);
}

cudaError_t launch_decode_step_tc_fp8(const DecodeParams &p, const StepArgs &a, cudaStream_t stream,
                                      void *encode) {
    return tc::launch_any<true, true>(p, tc::step_params(a), stream, encode);
}

}  // namespace kf
