// kf_static.cu -- kf_decode_step for callers that cannot allocate device memory.
//
// Some callers of a decode step are not allowed to call cudaMalloc: serving
// runtimes whose device memory is carved up once, at start-up, by their own
// pool allocator; plugin-style hosts that hand a library only the input and
// output buffers of each call; and tight decode loops that cannot pay for
// cudaMalloc's implicit device synchronisation. kf_decode_step needs a scratch
// workspace (partials and merge counters). This file gives those callers a
// variant whose scratch is a fixed-size array in the library's own device
// memory, so the call itself allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU on which the
// library's device code is loaded holds it until the process exits. In host
// code its name is only a host-side stand-in, so its device address is taken
// with cudaGetSymbolAddress, once per device (and again if that device's
// context is torn down and created anew), with that device current.
#include <mutex>

#include "kf_internal.cuh"

namespace kf {
namespace {

// Scratch of kf_decode_step_static, shared by every call on a device.
static __device__ __align__(256) unsigned char g_step_scratch[KF_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
struct ScratchAddress {
    void *ptr = nullptr;
    unsigned long long ctx_id = 0;  // the context `ptr` was looked up in
};
ScratchAddress g_scratch[kMaxDevices];

// Device address of the scratch array on the current device (set up on the
// first call for that device, and again in a new context of it: a device
// reset reloads the module, which may place the array elsewhere).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    ScratchAddress &s = g_scratch[dev];
    if (s.ptr == nullptr || s.ctx_id != current_context_id()) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_step_scratch);
        if (e != cudaSuccess) return e;
        s.ptr = p;
        s.ctx_id = current_context_id();
    }
    *out = s.ptr;
    return cudaSuccess;
}

}  // namespace
}  // namespace kf

extern "C" kf_status kf_decode_step_static(
    const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
    const int32_t *block_tables, int bt_stride, const int32_t *context_lens_before,
    int max_context_len, int batch, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int64_t num_blocks, float scale, int num_splits, void *out,
    kf_dtype out_dtype, float *lse_out, kf_stream_t stream) {
    if (batch < 0 || num_splits < 0 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1)
        return KF_ERR_INVALID;
    if (batch == 0) return KF_OK;
    const bool uses = num_splits != 1;  // the split rule with S > 1, or the balanced schedule
    // Scratch beyond the array is refused here; a size of 0 (shapes the step
    // does not support, or a device that cannot be queried) is left to
    // kf_decode_step's own checks, so both calls report the same status.
    if (uses && kf_decode_step_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                              num_splits) > (size_t)KF_STATIC_SCRATCH_BYTES)
        return KF_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if (kf::scratch_address(&scratch) != cudaSuccess) return KF_ERR_CUDA;
    // The merge counters must start at zero, and the array keeps whatever the
    // previous call left: the step clears them on this call's stream once every
    // argument has passed its checks, so a refused call queues no work.
    return kf::decode_step_clearing_counters(
        q, k_new, v_new, k_cache, v_cache, block_tables, bt_stride, context_lens_before,
        max_context_len, batch, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
        num_splits, uses ? scratch : nullptr, uses ? (size_t)KF_STATIC_SCRATCH_BYTES : 0, out,
        out_dtype, lse_out, stream);
}
