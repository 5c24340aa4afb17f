// kf_decode_bal.cu -- bf16-cache instantiations of the balanced-schedule
// decode step (kf_decode_bal.cuh).
#include "kf_decode_bal.cuh"

namespace kf {

cudaError_t decode_bal_resident(int head_dim, int num_q_heads, int num_kv_heads, int *resident) {
    return tc::bal_resident<false>(head_dim, num_q_heads, num_kv_heads, resident);
}

cudaError_t launch_decode_step_bal(const DecodeParams &p, const StepArgs &a, int ctas, cudaStream_t stream,
                                   void *encode) {
    return tc::launch_bal<false>(p, tc::step_params(a), ctas, stream, encode);
}

}  // namespace kf
