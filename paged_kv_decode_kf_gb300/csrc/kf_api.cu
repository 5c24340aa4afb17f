// kf_api.cu -- the extern "C" surface declared in include/kf.h.
//
// Host-side argument checks, the per-device error word, the split planner
// and dispatch to the kernels. No call allocates device memory: the error
// word is a __device__ variable of this library (one per device that loads
// it), and all buffers are the caller's.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <queue>
#include <vector>

#include "kf_internal.cuh"

namespace kf {

// The device error word (KF_DEVERR_* bits). Host code obtains its device
// address with cudaGetSymbolAddress, once per device.
static __device__ unsigned int g_error_word;

unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    unsigned long long ctx_id = 0;  // context the facts below were taken in
    int sm_count = 0;
    unsigned int *err = nullptr;
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];
void *g_encode_fn = nullptr;
bool g_encode_tried = false;

// Per-device facts, set up on first use with that device current (and again
// in a new context of that device).
cudaError_t device_info(DeviceInfo **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &d = g_devices[dev];
    // a context torn down and created again (cudaDeviceReset) reloads the
    // module, so the address is looked up again in a new context
    if (!d.ready || d.ctx_id != current_context_id()) {
        d.ready = false;
        e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.err), g_error_word);
        if (e != cudaSuccess) return e;
        d.ctx_id = current_context_id();
        d.ready = true;
    }
    *out = &d;
    return cudaSuccess;
}

// cuTensorMapEncodeTiled from the driver, without linking libcuda.
void *encode_fn() {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode_tried) {
        g_encode_tried = true;
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode_fn = fn;
    }
    return g_encode_fn;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_dims(int head_dim, int block_size) {
    return (head_dim == 64 || head_dim == 128) && (block_size == 16 || block_size == 32);
}

bool supported_group(int num_q_heads, int num_kv_heads) {
    if (num_kv_heads < 1 || num_q_heads % num_kv_heads != 0) return false;
    const int g = num_q_heads / num_kv_heads;
    return g == 1 || g == 2 || g == 4 || g == 8;
}

kf_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KF_OK : KF_ERR_CUDA; }

// ----------------------------------------------------------------------------
// Balanced schedule of the decode step (num_splits = KF_SPLITS_BALANCED):
// P CTAs per KV-head group, one wave. Workspace: [batch, Hkv] counters, then
// 2P + batch partial slots of [Hq, D] o (two per CTA, one per request for a
// request inside one CTA that merges with extra partials), then as many of
// [Hq] lse.
// ----------------------------------------------------------------------------
struct BalLayout {
    size_t ctr, o, lse, total;  // byte offsets of the three parts, and the size
};

BalLayout bal_layout(int ctas, int batch, int num_q_heads, int num_kv_heads, int head_dim) {
    const auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t slots = 2 * (size_t)ctas + (size_t)batch;
    BalLayout l;
    l.ctr = 0;
    l.o = al((size_t)batch * num_kv_heads * 4);
    l.lse = l.o + al(slots * num_q_heads * head_dim * 4);
    l.total = l.lse + al(slots * num_q_heads * 4);
    return l;
}

// Upper bound of P over both cache types: CTAs per SM from the kernels'
// shared memory alone (registers can only lower it), times SMs, per group.
int bal_ctas_bound(int num_kv_heads, int head_dim, int sm_count) {
    int hpc = 1, c16 = 1, c8 = 1;
    decode_tc_shape(num_kv_heads, head_dim, 16, false, &hpc, &c16);
    decode_tc_shape(num_kv_heads, head_dim, 16, true, &hpc, &c8);
    const int groups = num_kv_heads / hpc;
    return std::max(1, std::max(c16, c8) * sm_count / groups);
}

// ----------------------------------------------------------------------------
// Split planner: a model of the decode kernel's schedule. Work units are
// (request, KV-head group, split) CTAs launched split-fastest. While CTAs are
// still queued, every slot is busy and each CTA streams at the fair share of
// HBM bandwidth; the hardware hands a freed slot the next CTA in launch order
// (simulated with a heap of slot finish times). Once the queue is empty the
// remaining CTAs drain, each at min(its own in-flight-bytes limit, bandwidth
// / CTAs still running). A CTA pays a fixed start-up; an empty CTA only its
// zero-fill; the merge reads and writes S partial rows per output row.
// Constants were fitted to measured GB300 sweeps of split count on the five
// workloads of the test suite.
// ----------------------------------------------------------------------------
constexpr double kHbmBytesPerUs = 7.2e6;   // sustained read bandwidth of the decode stream
constexpr double kLatencyUs = 3.0;         // loaded DRAM round trip seen by one CTA's ring
constexpr double kCtaStartUs = 1.5;        // CTA start-up: table, q, first loads in flight
constexpr double kEmptyCtaUs = 0.25;       // CTA that only writes its empty partial
constexpr double kLaunchUs = 3.0;          // one kernel launch

double model_time(int S, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                  int block_size, int64_t n_max, const int64_t *n_blocks, int heads_per_cta,
                  int slots, double ring_bytes, double elem_bytes) {
    const int64_t chunk = std::max<int64_t>(1, (n_max + S - 1) / S);
    const int groups = (num_kv_heads + heads_per_cta - 1) / heads_per_cta;
    const double bytes_per_block = 2.0 * block_size * heads_per_cta * head_dim * elem_bytes;
    const double fair = kHbmBytesPerUs / slots;                // bytes/us per CTA, all slots busy
    const double cap = std::max(fair, ring_bytes / kLatencyUs);  // one CTA alone
    std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
    for (int i = 0; i < slots; ++i) free_at.push(0.0);
    double queue_empty_at = 0.0;
    int64_t empties = 0;
    for (int b = 0; b < batch; ++b) {
        const int64_t nb = n_blocks ? n_blocks[b] : n_max;
        for (int g = 0; g < groups; ++g) {
            for (int s = 0; s < S; ++s) {
                const int64_t lo = (int64_t)s * chunk;
                const int64_t cnt = std::max<int64_t>(0, std::min(nb, lo + chunk) - lo);
                if (cnt == 0) {
                    ++empties;
                    continue;
                }
                const double start = free_at.top();
                free_at.pop();
                free_at.push(start + kCtaStartUs + cnt * bytes_per_block / fair);
                queue_empty_at = start;
            }
        }
    }
    // drain: remaining bytes of the CTAs still running when the queue empties
    std::vector<double> rem;
    while (!free_at.empty()) {
        const double end = free_at.top();
        free_at.pop();
        if (end > queue_empty_at) rem.push_back((end - queue_empty_at) * fair);
    }
    std::sort(rem.begin(), rem.end());
    double t = queue_empty_at, done = 0.0;
    const size_t n = rem.size();
    for (size_t i = 0; i < n; ++i) {
        const double rate = std::min(cap, kHbmBytesPerUs / (double)(n - i));
        t += (rem[i] - done) / rate;
        done = rem[i];
    }
    // the merge: with one split there is none (the single-launch step writes its
    // rows directly; a separate merge of one slot is a copy the caller can skip)
    const double rows = (double)batch * num_q_heads;
    const double merge_bytes = rows * (S * (head_dim + 1) * 4.0 * 2.0 + head_dim * 4.0);
    const double merge_us = S > 1 ? merge_bytes / kHbmBytesPerUs + kLaunchUs : 0.0;
    return t + empties * kEmptyCtaUs / slots + kLaunchUs + merge_us;
}

}  // namespace

int decode_impl() {
    // read per call so a process can compare the two kernels
    const char *s = getenv("KF_DECODE_IMPL");
    return (s && strcmp(s, "simt") == 0) ? 1 : 0;
}

// Which multi-query kernel serves a call: 0 = mma.sync (kf_multiquery.cu), 1 =
// tcgen05 with one 128-row query tile per CTA, 2 = tcgen05 with two tiles and
// 128-token KV tiles, 3 = tcgen05 on CTA pairs (head_dim 128 only; opt-in: it
// measured slower than 2 on the chunked-prefill and cascade workloads). By rows
// per KV head (max_query_len x group): up to 128 -> 1, more -> 2. Even 8-32 rows (speculative verify of 2-8 tokens at G = 4,
// HBM-bound) stream KV faster through the one-tile tcgen05 kernel (5.1 TB/s on
// 64 requests of ~3.8K tokens) than through the mma.sync kernel (4.2 TB/s),
// the padded rows notwithstanding. KF_MQ_IMPL = "mma", "tc05", "tc05w" or
// "tc05p" forces one (read per call, so a process can compare them; "tc05w"
// needs more than 128 rows, and "tc05p" head_dim 128 -- otherwise the default
// for the shape runs).
int multiquery_kernel(int max_query_len, int group, int head_dim) {
    const int64_t rows = (int64_t)max_query_len * group;
    const int wide = rows > 128 ? 2 : 1;
    const char *s = getenv("KF_MQ_IMPL");
    if (s && strcmp(s, "mma") == 0) return 0;
    if (s && strcmp(s, "tc05") == 0) return 1;
    if (s && strcmp(s, "tc05w") == 0) return rows > 128 ? 2 : 1;
    if (s && strcmp(s, "tc05p") == 0) return head_dim == 128 ? 3 : wide;
    return wide;
}

}  // namespace kf

using namespace kf;

extern "C" {

const char *kf_status_string(kf_status s) {
    switch (s) {
        case KF_OK: return "ok";
        case KF_ERR_INVALID: return "invalid argument";
        case KF_ERR_UNSUPPORTED: return "unsupported shape";
        case KF_ERR_CUDA: return "CUDA error";
        case KF_ERR_DEVICE: return "a kernel recorded a device error";
    }
    return "unknown status";
}

int kf_version(void) { return 100; }

kf_status kf_append_kv(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                       const int32_t *block_tables, int bt_stride,
                       const int32_t *context_lens_before, int batch, int num_kv_heads,
                       int head_dim, int block_size, int64_t num_blocks, kf_stream_t stream) {
    if (batch < 0 || num_kv_heads < 1 || bt_stride < 1 || num_blocks < 1 || head_dim < 1 ||
        block_size < 1)
        return KF_ERR_INVALID;
    if (batch == 0) return KF_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !block_tables || !context_lens_before)
        return KF_ERR_INVALID;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return KF_ERR_INVALID;
    if (!supported_dims(head_dim, block_size)) return KF_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return KF_ERR_CUDA;
    return from_cuda(launch_append(
        static_cast<const uint16_t *>(k_new), static_cast<const uint16_t *>(v_new),
        static_cast<uint16_t *>(k_cache), static_cast<uint16_t *>(v_cache), block_tables,
        bt_stride, context_lens_before, batch, num_kv_heads, head_dim, block_size, num_blocks,
        dev->err, reinterpret_cast<cudaStream_t>(stream)));
}

kf_status kf_append_kv_fp8(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                           const float *k_scale, const float *v_scale, const int32_t *block_tables,
                           int bt_stride, const int32_t *context_lens_before, int batch,
                           int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                           kf_stream_t stream) {
    if (batch < 0 || num_kv_heads < 1 || bt_stride < 1 || num_blocks < 1 || head_dim < 1 ||
        block_size < 1)
        return KF_ERR_INVALID;
    if (batch == 0) return KF_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !block_tables || !context_lens_before ||
        !k_scale || !v_scale)
        return KF_ERR_INVALID;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return KF_ERR_INVALID;
    if (!supported_dims(head_dim, block_size)) return KF_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return KF_ERR_CUDA;
    return from_cuda(launch_append_fp8(
        static_cast<const uint16_t *>(k_new), static_cast<const uint16_t *>(v_new),
        static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache), k_scale, v_scale,
        block_tables, bt_stride, context_lens_before, batch, num_kv_heads, head_dim, block_size,
        num_blocks, dev->err, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

kf_status attention_impl(const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, int bt_stride, const int32_t *context_lens,
                         int max_context_len, int batch, int num_q_heads, int num_kv_heads,
                         int head_dim, int block_size, int64_t num_blocks, float scale,
                         int num_splits, float *out_partial, float *lse_partial,
                         const float *k_scale, const float *v_scale, bool kv8, kf_stream_t stream) {
    if (batch < 0 || num_splits < 1 || bt_stride < 1 || num_blocks < 1 || max_context_len < 0 ||
        num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 || !isfinite(scale))
        return KF_ERR_INVALID;
    if (batch == 0) return KF_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out_partial ||
        !lse_partial || (kv8 && (!k_scale || !v_scale)))
        return KF_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out_partial))
        return KF_ERR_INVALID;
    if (!supported_dims(head_dim, block_size) || !supported_group(num_q_heads, num_kv_heads))
        return KF_ERR_UNSUPPORTED;
    if (batch > 65535 || num_splits > 65535) return KF_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return KF_ERR_CUDA;

    DecodeParams p;
    p.q = static_cast<const uint16_t *>(q);
    p.k_cache = static_cast<const uint16_t *>(k_cache);
    p.v_cache = static_cast<const uint16_t *>(v_cache);
    p.block_tables = block_tables;
    p.ctx_lens = context_lens;
    p.out_partial = out_partial;
    p.lse_partial = lse_partial;
    p.err = dev->err;
    p.num_blocks = num_blocks;
    p.bt_stride = bt_stride;
    p.max_context_len = max_context_len;
    p.batch = batch;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.block_size = block_size;
    p.num_splits = num_splits;
    const int64_t n_max = ((int64_t)max_context_len + block_size - 1) / block_size;
    p.chunk_blocks = (int)std::max<int64_t>(1, (n_max + num_splits - 1) / num_splits);
    p.scale_log2 = scale * 1.4426950408889634f;
    p.k_scale = kv8 ? k_scale : nullptr;
    p.v_scale = kv8 ? v_scale : nullptr;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!kv8 && decode_impl() == 1) return from_cuda(launch_decode_simt(p, st));
    void *fn = encode_fn();
    if (!fn) return KF_ERR_CUDA;
    return from_cuda(kv8 ? launch_decode_tc_fp8(p, st, fn) : launch_decode_tc(p, st, fn));
}

}  // namespace

extern "C" {

kf_status kf_paged_decode_attention(const void *q, const void *k_cache, const void *v_cache,
                                    const int32_t *block_tables, int bt_stride,
                                    const int32_t *context_lens, int max_context_len, int batch,
                                    int num_q_heads, int num_kv_heads, int head_dim,
                                    int block_size, int64_t num_blocks, float scale,
                                    int num_splits, float *out_partial, float *lse_partial,
                                    kf_stream_t stream) {
    return attention_impl(q, k_cache, v_cache, block_tables, bt_stride, context_lens,
                          max_context_len, batch, num_q_heads, num_kv_heads, head_dim, block_size,
                          num_blocks, scale, num_splits, out_partial, lse_partial, nullptr, nullptr,
                          false, stream);
}

kf_status kf_paged_decode_attention_fp8(const void *q, const void *k_cache, const void *v_cache,
                                        const float *k_scale, const float *v_scale,
                                        const int32_t *block_tables, int bt_stride,
                                        const int32_t *context_lens, int max_context_len,
                                        int batch, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, int64_t num_blocks,
                                        float scale, int num_splits, float *out_partial,
                                        float *lse_partial, kf_stream_t stream) {
    return attention_impl(q, k_cache, v_cache, block_tables, bt_stride, context_lens,
                          max_context_len, batch, num_q_heads, num_kv_heads, head_dim, block_size,
                          num_blocks, scale, num_splits, out_partial, lse_partial, k_scale,
                          v_scale, true, stream);
}

kf_status kf_paged_multiquery_attention(const void *q, const int32_t *q_start, const void *k_cache,
                                        const void *v_cache, const int32_t *block_tables,
                                        int bt_stride, const int32_t *context_lens, int causal,
                                        int max_context_len, int max_query_len, int batch,
                                        int num_q_tokens, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, int64_t num_blocks,
                                        float scale, int num_splits, float *out_partial,
                                        float *lse_partial, kf_stream_t stream) {
    if (batch < 0 || num_q_tokens < 0 || num_splits < 1 || bt_stride < 1 || num_blocks < 1 ||
        max_context_len < 0 || max_query_len < 0 || num_q_heads < 1 || num_kv_heads < 1 ||
        head_dim < 1 || block_size < 1 || !isfinite(scale) || (causal != 0 && causal != 1))
        return KF_ERR_INVALID;
    if (batch == 0 || num_q_tokens == 0) return KF_OK;
    if (!q || !q_start || !k_cache || !v_cache || !block_tables || !context_lens || !out_partial ||
        !lse_partial)
        return KF_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out_partial))
        return KF_ERR_INVALID;
    if (head_dim != 128 && head_dim != 64) return KF_ERR_UNSUPPORTED;
    if (!supported_dims(head_dim, block_size) || !supported_group(num_q_heads, num_kv_heads))
        return KF_ERR_UNSUPPORTED;
    if (num_splits > 65535) return KF_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return KF_ERR_CUDA;
    MqParams p;
    p.q = static_cast<const uint16_t *>(q);
    p.q_start = q_start;
    p.k_cache = static_cast<const uint16_t *>(k_cache);
    p.v_cache = static_cast<const uint16_t *>(v_cache);
    p.block_tables = block_tables;
    p.ctx_lens = context_lens;
    p.out_partial = out_partial;
    p.lse_partial = lse_partial;
    p.err = dev->err;
    p.num_blocks = num_blocks;
    p.bt_stride = bt_stride;
    p.max_context_len = max_context_len;
    p.max_query_len = max_query_len;
    p.batch = batch;
    p.num_q_tokens = num_q_tokens;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.block_size = block_size;
    p.num_splits = num_splits;
    const int64_t n_max = ((int64_t)max_context_len + block_size - 1) / block_size;
    p.chunk_blocks = (int)std::max<int64_t>(1, (n_max + num_splits - 1) / num_splits);
    p.causal = causal;
    p.q_tiles = 1;
    p.scale_log2 = scale * 1.4426950408889634f;
    void *fn = encode_fn();
    if (!fn) return KF_ERR_CUDA;
    const int which = multiquery_kernel(max_query_len, num_q_heads / num_kv_heads, head_dim);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = which == 3   ? launch_multiquery_tc05p(p, st, fn)
                          : which == 2 ? launch_multiquery_tc05w(p, st, fn)
                          : which == 1 ? launch_multiquery_tc05(p, st, fn)
                                       : launch_multiquery(p, st, fn);
    if (e == cudaErrorInvalidValue) return KF_ERR_UNSUPPORTED;
    return from_cuda(e);
}

size_t kf_decode_step_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                     int num_splits) {
    if (batch < 0 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || num_splits < 0) return 0;
    if (num_splits == KF_SPLITS_BALANCED) {
        if (!supported_dims(head_dim, 16) || !supported_group(num_q_heads, num_kv_heads)) return 0;
        DeviceInfo *dev = nullptr;
        if (device_info(&dev) != cudaSuccess) return 0;
        return bal_layout(bal_ctas_bound(num_kv_heads, head_dim, dev->sm_count), batch, num_q_heads,
                          num_kv_heads, head_dim)
            .total;
    }
    const size_t rows = (size_t)batch * num_q_heads;
    const auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    return al((size_t)num_splits * rows * head_dim * 4) + al((size_t)num_splits * rows * 4) +
           al((size_t)batch * num_kv_heads * 4);
}

}  // extern "C"

namespace {

// Shared DecodeParams of the two step schedules.
DecodeParams step_decode_params(const void *q, const void *k_cache, const void *v_cache,
                                const int32_t *block_tables, int bt_stride,
                                const int32_t *context_lens_before, int max_context_len, int batch,
                                int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                int64_t num_blocks, float scale, int num_splits, const float *k_scale,
                                const float *v_scale, bool kv8, unsigned int *err) {
    DecodeParams p;
    p.q = static_cast<const uint16_t *>(q);
    p.k_cache = static_cast<const uint16_t *>(k_cache);
    p.v_cache = static_cast<const uint16_t *>(v_cache);
    p.block_tables = block_tables;
    p.ctx_lens = context_lens_before;
    p.out_partial = nullptr;
    p.lse_partial = nullptr;
    p.err = err;
    p.num_blocks = num_blocks;
    p.bt_stride = bt_stride;
    p.max_context_len = max_context_len;
    p.batch = batch;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.block_size = block_size;
    p.num_splits = num_splits;
    const int64_t n_max = ((int64_t)max_context_len + block_size - 1) / block_size;
    p.chunk_blocks = num_splits > 0 ? (int)std::max<int64_t>(1, (n_max + num_splits - 1) / num_splits) : 1;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.k_scale = kv8 ? k_scale : nullptr;
    p.v_scale = kv8 ? v_scale : nullptr;
    return p;
}

// The decode step on the balanced schedule (arguments checked by step_impl).
kf_status bal_step(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                   const int32_t *block_tables, int bt_stride, const int32_t *context_lens_before,
                   int max_context_len, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                   int block_size, int64_t num_blocks, float scale, void *workspace,
                   size_t workspace_bytes, void *out, kf_dtype out_dtype, float *lse_out,
                   const float *k_scale, const float *v_scale, bool kv8, const float *ex_o,
                   const float *ex_lse, int n_ex, bool clear_counters, kf_stream_t stream) {
    if (!workspace || !aligned16(workspace)) return KF_ERR_INVALID;
    DeviceInfo *dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return KF_ERR_CUDA;
    int hpc = 1, cps = 1, resident = 0;
    decode_tc_shape(num_kv_heads, head_dim, block_size, kv8, &hpc, &cps);
    const cudaError_t re = kv8 ? decode_bal_resident_fp8(head_dim, num_q_heads, num_kv_heads, &resident)
                               : decode_bal_resident(head_dim, num_q_heads, num_kv_heads, &resident);
    if (re == cudaErrorInvalidValue) return KF_ERR_UNSUPPORTED;
    if (re != cudaSuccess) return KF_ERR_CUDA;
    // one wave; no more CTAs than the batch can have 16-token stages.
    // KF_BAL_CTAS (CTAs per KV-head group, read per call) overrides it for tuning.
    int64_t ctas = std::max(1, resident * dev->sm_count / (num_kv_heads / hpc));
    if (const char *env = getenv("KF_BAL_CTAS")) {
        const int forced = atoi(env);
        if (forced > 0) ctas = std::min<int64_t>(forced, bal_ctas_bound(num_kv_heads, head_dim, dev->sm_count));
    }
    const int64_t stages_max = (int64_t)batch * (((int64_t)max_context_len + 15) / 16);
    ctas = std::max<int64_t>(1, std::min(ctas, stages_max));
    const BalLayout l = bal_layout((int)ctas, batch, num_q_heads, num_kv_heads, head_dim);
    if (!workspace || !aligned16(workspace) || workspace_bytes < l.total) return KF_ERR_INVALID;
    const DecodeParams p = step_decode_params(q, k_cache, v_cache, block_tables, bt_stride,
                                              context_lens_before, max_context_len, batch, num_q_heads,
                                              num_kv_heads, head_dim, block_size, num_blocks, scale, 0,
                                              k_scale, v_scale, kv8, dev->err);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    StepArgs a;
    a.k_new = static_cast<const uint16_t *>(k_new);
    a.v_new = static_cast<const uint16_t *>(v_new);
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.counters = reinterpret_cast<unsigned int *>(ws + l.ctr);
    a.ws_o = reinterpret_cast<float *>(ws + l.o);
    a.ws_lse = reinterpret_cast<float *>(ws + l.lse);
    a.out = out;
    a.lse_out = lse_out;
    a.out_dtype = (int)out_dtype;
    a.ex_o = n_ex > 0 ? ex_o : nullptr;
    a.ex_lse = n_ex > 0 ? ex_lse : nullptr;
    a.n_ex = n_ex;
    void *fn = encode_fn();
    if (!fn) return KF_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (clear_counters &&
        cudaMemsetAsync(a.counters, 0, (size_t)batch * num_kv_heads * 4, st) != cudaSuccess)
        return KF_ERR_CUDA;
    const cudaError_t e = kv8 ? launch_decode_step_bal_fp8(p, a, (int)ctas, st, fn)
                              : launch_decode_step_bal(p, a, (int)ctas, st, fn);
    if (e == cudaErrorInvalidValue) return KF_ERR_UNSUPPORTED;
    return from_cuda(e);
}

kf_status step_impl(const void *q, const void *k_new, const void *v_new, void *k_cache,
                    void *v_cache, const int32_t *block_tables, int bt_stride,
                    const int32_t *context_lens_before, int max_context_len, int batch,
                    int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                    int64_t num_blocks, float scale, int num_splits, void *workspace,
                    size_t workspace_bytes, void *out, kf_dtype out_dtype, float *lse_out,
                    const float *k_scale, const float *v_scale, bool kv8, const float *ex_o,
                    const float *ex_lse, int n_ex, bool clear_counters, kf_stream_t stream) {
    if (batch < 0 || num_splits < 0 || bt_stride < 1 || num_blocks < 1 || max_context_len < 0 ||
        num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 || !isfinite(scale) ||
        (out_dtype != KF_BF16 && out_dtype != KF_F32) || n_ex < 0)
        return KF_ERR_INVALID;
    if (batch == 0) return KF_OK;
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !block_tables || !context_lens_before ||
        !out || (kv8 && (!k_scale || !v_scale)) ||
        (n_ex > 0 && (!ex_o || !ex_lse || !aligned16(ex_o))))
        return KF_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
        !aligned16(v_cache) || !aligned16(out))
        return KF_ERR_INVALID;
    if (!supported_dims(head_dim, block_size) || !supported_group(num_q_heads, num_kv_heads))
        return KF_ERR_UNSUPPORTED;
    if (batch > 65535 || num_splits > 65535) return KF_ERR_UNSUPPORTED;
    if (num_splits == KF_SPLITS_BALANCED)
        return bal_step(q, k_new, v_new, k_cache, v_cache, block_tables, bt_stride, context_lens_before,
                        max_context_len, batch, num_q_heads, num_kv_heads, head_dim, block_size,
                        num_blocks, scale, workspace, workspace_bytes, out, out_dtype, lse_out, k_scale,
                        v_scale, kv8, ex_o, ex_lse, n_ex, clear_counters, stream);
    const size_t need = kf_decode_step_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                      num_splits);
    const bool counted = num_splits > 1 || n_ex > 0;  // some group merges: counters needed
    if (counted && (!workspace || !aligned16(workspace) || workspace_bytes < need))
        return KF_ERR_INVALID;
    // the last CTA of a group merges in its shared-memory ring: S x rows x 4 bytes must fit
    int hpc = 1, cps = 1;
    decode_tc_shape(num_kv_heads, head_dim, block_size, kv8, &hpc, &cps);
    const int R = hpc * (num_q_heads / num_kv_heads);
    if (((int64_t)num_splits + n_ex) * R * 4 + 8 * R > decode_tc_ring_bytes(num_kv_heads, head_dim, kv8))
        return KF_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return KF_ERR_CUDA;

    DecodeParams p;
    p.q = static_cast<const uint16_t *>(q);
    p.k_cache = static_cast<const uint16_t *>(k_cache);
    p.v_cache = static_cast<const uint16_t *>(v_cache);
    p.block_tables = block_tables;
    p.ctx_lens = context_lens_before;
    p.out_partial = nullptr;
    p.lse_partial = nullptr;
    p.err = dev->err;
    p.num_blocks = num_blocks;
    p.bt_stride = bt_stride;
    p.max_context_len = max_context_len;
    p.batch = batch;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.block_size = block_size;
    p.num_splits = num_splits;
    const int64_t n_max = ((int64_t)max_context_len + block_size - 1) / block_size;
    p.chunk_blocks = (int)std::max<int64_t>(1, (n_max + num_splits - 1) / num_splits);
    p.scale_log2 = scale * 1.4426950408889634f;
    p.k_scale = kv8 ? k_scale : nullptr;
    p.v_scale = kv8 ? v_scale : nullptr;

    const size_t rows = (size_t)batch * num_q_heads;
    const auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    StepArgs a;
    a.k_new = static_cast<const uint16_t *>(k_new);
    a.v_new = static_cast<const uint16_t *>(v_new);
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.ws_o = counted ? reinterpret_cast<float *>(ws) : nullptr;
    a.ws_lse = counted ? reinterpret_cast<float *>(ws + al((size_t)num_splits * rows * head_dim * 4)) : nullptr;
    a.counters = counted ? reinterpret_cast<unsigned int *>(
                                      ws + al((size_t)num_splits * rows * head_dim * 4) +
                                      al((size_t)num_splits * rows * 4))
                                : nullptr;
    a.out = out;
    a.lse_out = lse_out;
    a.out_dtype = (int)out_dtype;
    a.ex_o = n_ex > 0 ? ex_o : nullptr;
    a.ex_lse = n_ex > 0 ? ex_lse : nullptr;
    a.n_ex = n_ex;
    void *fn = encode_fn();
    if (!fn) return KF_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (clear_counters && a.counters &&
        cudaMemsetAsync(a.counters, 0, (size_t)batch * num_kv_heads * 4, st) != cudaSuccess)
        return KF_ERR_CUDA;
    return from_cuda(kv8 ? launch_decode_step_tc_fp8(p, a, st, fn) : launch_decode_step_tc(p, a, st, fn));
}


}  // namespace

extern "C" {

kf_status kf_decode_step(const void *q, const void *k_new, const void *v_new, void *k_cache,
                         void *v_cache, const int32_t *block_tables, int bt_stride,
                         const int32_t *context_lens_before, int max_context_len, int batch,
                         int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         int64_t num_blocks, float scale, int num_splits, void *workspace,
                         size_t workspace_bytes, void *out, kf_dtype out_dtype, float *lse_out,
                         kf_stream_t stream) {
    return step_impl(q, k_new, v_new, k_cache, v_cache, block_tables, bt_stride,
                     context_lens_before, max_context_len, batch, num_q_heads, num_kv_heads,
                     head_dim, block_size, num_blocks, scale, num_splits, workspace,
                     workspace_bytes, out, out_dtype, lse_out, nullptr, nullptr, false, nullptr,
                     nullptr, 0, false, stream);
}

kf_status kf_decode_step_merge_partials(const void *q, const void *k_new, const void *v_new,
                                        void *k_cache, void *v_cache, const int32_t *block_tables,
                                        int bt_stride, const int32_t *context_lens_before,
                                        int max_context_len, int batch, int num_q_heads,
                                        int num_kv_heads, int head_dim, int block_size,
                                        int64_t num_blocks, float scale, int num_splits,
                                        const float *extra_out_partial,
                                        const float *extra_lse_partial, int num_extra,
                                        void *workspace, size_t workspace_bytes, void *out,
                                        kf_dtype out_dtype, float *lse_out, kf_stream_t stream) {
    return step_impl(q, k_new, v_new, k_cache, v_cache, block_tables, bt_stride,
                     context_lens_before, max_context_len, batch, num_q_heads, num_kv_heads,
                     head_dim, block_size, num_blocks, scale, num_splits, workspace,
                     workspace_bytes, out, out_dtype, lse_out, nullptr, nullptr, false,
                     extra_out_partial, extra_lse_partial, num_extra, false, stream);
}

kf_status kf_decode_step_fp8(const void *q, const void *k_new, const void *v_new, void *k_cache,
                             void *v_cache, const float *k_scale, const float *v_scale,
                             const int32_t *block_tables, int bt_stride,
                             const int32_t *context_lens_before, int max_context_len, int batch,
                             int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                             int64_t num_blocks, float scale, int num_splits, void *workspace,
                             size_t workspace_bytes, void *out, kf_dtype out_dtype,
                             float *lse_out, kf_stream_t stream) {
    return step_impl(q, k_new, v_new, k_cache, v_cache, block_tables, bt_stride,
                     context_lens_before, max_context_len, batch, num_q_heads, num_kv_heads,
                     head_dim, block_size, num_blocks, scale, num_splits, workspace,
                     workspace_bytes, out, out_dtype, lse_out, k_scale, v_scale, true, nullptr,
                     nullptr, 0, false, stream);
}

}  // extern "C"

namespace kf {

// kf_decode_step with the workspace's merge counters cleared on the stream
// after every argument check, right before the launch (the scratch of
// kf_decode_step_static keeps the previous call's contents).
kf_status decode_step_clearing_counters(const void *q, const void *k_new, const void *v_new,
                                        void *k_cache, void *v_cache, const int32_t *block_tables,
                                        int bt_stride, const int32_t *context_lens_before,
                                        int max_context_len, int batch, int num_q_heads,
                                        int num_kv_heads, int head_dim, int block_size,
                                        int64_t num_blocks, float scale, int num_splits,
                                        void *workspace, size_t workspace_bytes, void *out,
                                        kf_dtype out_dtype, float *lse_out, kf_stream_t stream) {
    return step_impl(q, k_new, v_new, k_cache, v_cache, block_tables, bt_stride,
                     context_lens_before, max_context_len, batch, num_q_heads, num_kv_heads,
                     head_dim, block_size, num_blocks, scale, num_splits, workspace,
                     workspace_bytes, out, out_dtype, lse_out, nullptr, nullptr, false, nullptr,
                     nullptr, 0, true, stream);
}

}  // namespace kf


namespace {

int choose_splits(int batch, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                  int max_context_len, const int32_t *context_lens_host, int num_sms, bool kv8) {
    if (batch < 1 || max_context_len < 0 || num_sms < 1 || block_size < 1 ||
        !supported_dims(head_dim, block_size) || !supported_group(num_q_heads, num_kv_heads))
        return -1;
    const int64_t n_max = ((int64_t)max_context_len + block_size - 1) / block_size;
    if (n_max <= 1) return 1;
    std::vector<int64_t> nb;
    if (context_lens_host) {
        nb.resize(batch);
        for (int b = 0; b < batch; ++b) {
            const int64_t L = std::max<int32_t>(0, context_lens_host[b]);
            nb[b] = std::min<int64_t>((L + block_size - 1) / block_size, n_max);
        }
    }
    int hpc = 1, cps = 1;
    double ring = 32768.0;
    if (!kv8 && decode_impl() == 1) {
        hpc = 1;
        cps = 8;
    } else {
        decode_tc_shape(num_kv_heads, head_dim, block_size, kv8, &hpc, &cps);
        ring = decode_tc_ring_bytes(num_kv_heads, head_dim, kv8);
    }
    const int slots = num_sms * cps;
    static const int cands[] = {1,   2,   3,   4,   5,   6,   7,   8,   10,  12,  14,  16,
                                20,  24,  28,  32,  40,  48,  56,  64,  80,  96,  112, 128,
                                160, 192, 224, 256, 320, 384, 448, 512, 640, 768, 896, 1024};
    int best = 1;
    double best_t = 1e300;
    for (int S : cands) {
        if (S > n_max) break;
        const double t = model_time(S, batch, num_q_heads, num_kv_heads, head_dim, block_size,
                                    n_max, nb.empty() ? nullptr : nb.data(), hpc, slots, ring,
                                    kv8 ? 1.0 : 2.0);
        if (t < best_t * 0.995) {  // prefer fewer splits unless clearly faster
            best_t = t;
            best = S;
        }
    }
    return best;
}

}  // namespace

extern "C" {

int kf_choose_num_splits_for(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                             int block_size, int max_context_len,
                             const int32_t *context_lens_host, int num_sms) {
    return choose_splits(batch, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                         context_lens_host, num_sms, false);
}

int kf_choose_num_splits(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                         int block_size, int max_context_len, const int32_t *context_lens_host,
                         int device) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return -1;
    return choose_splits(batch, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                         context_lens_host, sms, false);
}

int kf_choose_num_splits_fp8(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                             int block_size, int max_context_len,
                             const int32_t *context_lens_host, int num_sms) {
    return choose_splits(batch, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                         context_lens_host, num_sms, true);
}

kf_status kf_merge_partials(const float *out_partial, const float *lse_partial,
                            int num_partials, int batch, int num_q_heads, int head_dim,
                            void *out, kf_dtype out_dtype, float *lse_out, kf_stream_t stream) {
    if (num_partials < 1 || batch < 0 || num_q_heads < 1 ||
        (out_dtype != KF_BF16 && out_dtype != KF_F32))
        return KF_ERR_INVALID;
    if (batch == 0) return KF_OK;
    if (!out_partial || !lse_partial || !out) return KF_ERR_INVALID;
    if (!aligned16(out_partial) || !aligned16(out)) return KF_ERR_INVALID;
    if (head_dim != 64 && head_dim != 128) return KF_ERR_UNSUPPORTED;
    return from_cuda(launch_merge(out_partial, lse_partial, num_partials, batch, num_q_heads,
                                  head_dim, out, (int)out_dtype, lse_out,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

kf_status kf_get_device_error(unsigned int *flags, kf_stream_t stream) {
    if (!flags) return KF_ERR_INVALID;
    DeviceInfo *dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return KF_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    unsigned int word = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KF_ERR_CUDA;
    if (cudaMemcpy(&word, dev->err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return KF_ERR_CUDA;
    if (word != 0 && cudaMemset(dev->err, 0, sizeof word) != cudaSuccess) return KF_ERR_CUDA;
    *flags = word;
    return word ? KF_ERR_DEVICE : KF_OK;
}

kf_status kf_check_bounded_wait(kf_stream_t stream) {
    DeviceInfo *dev = nullptr;
    if (device_info(&dev) != cudaSuccess) return KF_ERR_CUDA;
    return from_cuda(launch_wait_check(dev->err, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
