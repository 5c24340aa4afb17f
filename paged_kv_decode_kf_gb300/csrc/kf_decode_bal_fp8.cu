// kf_decode_bal_fp8.cu -- FP8 E4M3-cache instantiations of the
// balanced-schedule decode step (kf_decode_bal.cuh).
#include "kf_decode_bal.cuh"

namespace kf {

cudaError_t decode_bal_resident_fp8(int head_dim, int num_q_heads, int num_kv_heads, int *resident) {
    return tc::bal_resident<true>(head_dim, num_q_heads, num_kv_heads, resident);
}

cudaError_t launch_decode_step_bal_fp8(const DecodeParams &p, const StepArgs &a, int ctas,
                                       cudaStream_t stream, void *encode) {
    return tc::launch_bal<true>(p, tc::step_params(a), ctas, stream, encode);
}

}  // namespace kf
