// kf_decode_tc.cu -- bf16-cache instantiations of the tensor-core decode
// kernel (kf_decode_tc.cuh) and the shape queries the planner uses.
#include "kf_decode_tc.cuh"

namespace kf {

void decode_tc_shape(int num_kv_heads, int head_dim, int block_size, bool kv8, int *hpc_out,
                     int *ctas_per_sm) {
    (void)block_size;
    const int hpc = tc::heads_per_cta(num_kv_heads);
    const int smem = kv8 ? tc::smem_bytes<true>(head_dim, hpc) : tc::smem_bytes<false>(head_dim, hpc);
    const int per_sm = 228 * 1024;  // shared memory per SM, 1 KiB of it reserved per CTA
    int c = per_sm / (smem + 1024);
    if (c > 8) c = 8;
    if (c < 1) c = 1;
    *hpc_out = hpc;
    *ctas_per_sm = c;
}

int decode_tc_ring_bytes(int num_kv_heads, int head_dim, bool kv8) {
    const int hpc = tc::heads_per_cta(num_kv_heads);
    const int smem = kv8 ? tc::smem_bytes<true>(head_dim, hpc) : tc::smem_bytes<false>(head_dim, hpc);
    return smem - 1024 - 16 * 8;  // minus alignment slack and the largest barrier block
}

// One wait that nothing completes: an mbarrier expecting one arrival that
// never comes, polled with the kernels' bounded wait at a short limit (2^16
// polls); when it gives up, the error word gets KF_DEVERR_TIMEOUT and the
// kernel returns like the decode kernels do.
__global__ void wait_check_kernel(unsigned int *err) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = tc::smem_u32(&bar);
    if (threadIdx.x != 0) return;
    tc::mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (!tc::mbar_wait(b, 0, 1u << 16)) raise_error(err, KF_DEVERR_TIMEOUT);
}

cudaError_t launch_wait_check(unsigned int *err, cudaStream_t stream) {
    wait_check_kernel<<<1, 32, 0, stream>>>(err);
    return cudaGetLastError();
}

cudaError_t launch_decode_tc(const DecodeParams &p, cudaStream_t stream, void *encode) {
    tc::StepParams sp = {};
    return tc::launch_any<false, false>(p, sp, stream, encode);
}

cudaError_t launch_decode_step_tc(const DecodeParams &p, const StepArgs &a, cudaStream_t stream,
                                  void *encode) {
    return tc::launch_any<true, false>(p, tc::step_params(a), stream, encode);
}

}  // namespace kf
