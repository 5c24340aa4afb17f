// kf_mq_tc05.cuh -- pieces shared by the tcgen05 multi-query kernels: packed
// fp32 arithmetic for the softmax, warp-uniform bounded waits, and the 5-D
// tensor map whose box is one cache block of one head.
#pragma once

#include "kf_decode_tc.cuh"
#include "kf_tc05.cuh"

namespace kf {
namespace mq5 {

using namespace tc;

// Packed two-lane fp32 operations (f32x2 forms of sm_100 and later), the
// three-input max and the hardware base-2 exponential (flushes subnormal
// results to zero; exp2(-inf) = 0).
__device__ __forceinline__ float2 fma_f32x2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 add_f32x2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// All lanes of the warp see the same outcome of a bounded wait.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// ----------------------------------------------------------------------------
// Thread-block clusters
// ----------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// One arrival on an mbarrier of any CTA of the cluster (`caddr` from map_to),
// with the default (CTA-scope release) semantics: a cluster-scope release
// costs a memory barrier per arrival, and what the arrivals here publish --
// TMEM written under tcgen05 fences, shared memory the pair's MMAs read
// through the async proxy after a proxy fence -- needs no generic-memory
// ordering beyond the CTA.
__device__ __forceinline__ void arrive_cluster(uint32_t caddr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}

// Bounded wait on a local barrier whose arrivals may come from other CTAs.
__device__ __forceinline__ bool wait_cl(uint32_t bar, uint32_t parity) { return mbar_wait(bar, parity); }

__device__ __forceinline__ bool warp_wait_cl(uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, wait_cl(bar, parity));
}

// All threads of every CTA of the cluster.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 4-D view of a [num_blocks, bs, Hkv, D] bf16 cache: (d % 64, slot % 8,
// head * D/64 + d / 64, 8-slot group) -- the head stride is twice the
// 64-element stride, so (head, half) is one dimension, and the blocks' 8-slot
// groups follow one another at one stride, so (block, slot / 8) is one too
// (group = block * bs/8 + slot / 8) -- with a box of one block of one head:
// bs * D * 2 bytes at group coordinate block * bs/8, landing as 8-token atoms of
// 128-byte rows (token t, half c at (t / 8) * 1024 * D/64 + c * 1024 + (t % 8) * 128).
inline bool encode_block_map(tc::EncodeFn fn, CUtensorMap *map, const void *cache, const MqParams &p) {
    const int halves = p.head_dim / 64;
    const cuuint64_t row = (cuuint64_t)p.num_kv_heads * p.head_dim * 2;  // bytes between slots
    const cuuint64_t dims[4] = {64, 8, (cuuint64_t)p.num_kv_heads * halves,
                                (cuuint64_t)p.num_blocks * (p.block_size / 8)};
    const cuuint64_t strides[3] = {row, 128, 8 * row};
    const cuuint32_t box[4] = {64, 8, (cuuint32_t)halves, (cuuint32_t)p.block_size / 8};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(cache), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace mq5
}  // namespace kf
