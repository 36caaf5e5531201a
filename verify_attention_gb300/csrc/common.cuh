// common.cuh -- device helpers shared by the fp8kv kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/fp8kv.h"

namespace fp8kv {

// Device status word of this translation unit (bits FP8KV_DEV_*); each .cu
// file has its own copy and a host reader, OR-ed by fp8kv_device_status.
static __device__ unsigned int g_status;

__device__ __forceinline__ void flag(unsigned int bits) { atomicOr(&g_status, bits); }

// ------------------------------------------------------------------ E4M3

// Two fp32 values -> two E4M3FN codes (lo in bits 0..7, hi in bits 8..15):
// round to nearest even, saturating to +-448 (infinities included) by the
// hardware conversion; NaN inputs become 0x7F with their own sign bit.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    uint32_t out = r;
    uint32_t bl = __float_as_uint(lo), bh = __float_as_uint(hi);
    if ((bl & 0x7fffffffu) > 0x7f800000u) out = (out & 0xff00u) | 0x7fu | ((bl >> 24) & 0x80u);
    if ((bh & 0x7fffffffu) > 0x7f800000u) out = (out & 0x00ffu) | ((0x7fu | ((bh >> 24) & 0x80u)) << 8);
    return out;
}

// Two E4M3 codes (bits 0..15) -> f16x2, exact (every E4M3 value is an f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t codes) {
    uint32_t r;
    uint16_t c = (uint16_t)codes;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(c));
    return r;
}

// Two E4M3 codes (bits 0..15) -> two fp32 values, exact.
__device__ __forceinline__ void e4m3x2_to_f32x2(uint32_t codes, float& lo, float& hi) {
    const uint32_t h = e4m3x2_to_f16x2(codes);
    lo = __half2float(__ushort_as_half((unsigned short)(h & 0xffffu)));
    hi = __half2float(__ushort_as_half((unsigned short)(h >> 16)));
}

// f16x2 -> two E4M3 codes (bits 0..7 from the low half), round to nearest
// even, saturating; no NaN sign fix-up (for operands, not stored bytes).
__device__ __forceinline__ uint32_t f16x2_to_e4m3x2(uint32_t h) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
    return r;
}

__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h) {
    return make_float2(__half2float(__ushort_as_half((unsigned short)(h & 0xffffu))),
                       __half2float(__ushort_as_half((unsigned short)(h >> 16))));
}

__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t sub_f16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Eight bf16 values (one 16-byte chunk) -> eight E4M3 codes of x / scale,
// each with one fp32 IEEE division (the cache-insert encoding).
__device__ __forceinline__ uint2 e4m3_encode8(uint4 x, float scale) {
    uint2 o;
    o.x = e4m3x2(__fdiv_rn(bf16_lo(x.x), scale), __fdiv_rn(bf16_hi(x.x), scale)) |
          (e4m3x2(__fdiv_rn(bf16_lo(x.y), scale), __fdiv_rn(bf16_hi(x.y), scale)) << 16);
    o.y = e4m3x2(__fdiv_rn(bf16_lo(x.z), scale), __fdiv_rn(bf16_hi(x.z), scale)) |
          (e4m3x2(__fdiv_rn(bf16_lo(x.w), scale), __fdiv_rn(bf16_hi(x.w), scale)) << 16);
    return o;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// 2^x on the special-function unit (the hardware ex2 instruction).
__device__ __forceinline__ float ex2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// ------------------------------------------------------------ tensor core

// D += A * B, m16n8k16, fp32 accumulate; A row-major, B column-major.
__device__ __forceinline__ void mma_f16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D += A * B, m16n8k32, E4M3 x E4M3, fp32 accumulate; A row-major, B
// column-major; each register holds four consecutive k elements.
__device__ __forceinline__ void mma_e4m3(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------ mbarrier and TMA

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with parity `phase` of an mbarrier to complete.  Gives up
// after `limit_ns` of wall time (2 s unless a caller asks otherwise; sets
// FP8KV_DEV_WAIT_TIMEOUT and returns false) so a broken pipeline can never
// hang the GPU.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t phase, uint64_t limit_ns = 2000000000ull) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(phase)
        : "memory");
    if (ok) return true;
    const uint64_t start = globaltimer();
    while (true) {
        // suspends until the phase completes or 0.5 ms pass: no hot spinning
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
            : "=r"(ok)
            : "r"(bar), "r"(phase), "r"(500000u)
            : "memory");
        if (ok) return true;
        if (globaltimer() - start > limit_ns) {
            flag(FP8KV_DEV_WAIT_TIMEOUT);
            return false;
        }
    }
}

// Non-blocking test: has the phase with parity `phase` of an mbarrier completed?
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(phase)
        : "memory");
    return ok != 0;
}

// 3-D tiled TMA load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int x, int y, int z,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(tm), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from this CTA's shared memory to global memory, tracked as a bulk group.
__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk group has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue now; and, before touching any global input, wait until every
// kernel this one depends on has completed and its writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tm) : "memory");
}

}  // namespace fp8kv

// Host-side helpers (api.cu).
namespace fp8kv {
// Counts every kernel launch the library makes (api.cu; fp8kv_launch_count).
void count_launch();

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream is finishing; it must call pdl_wait()
// before reading anything that kernel may have written.  cluster_x > 1
// groups that many consecutive CTAs along x into one thread-block cluster.
template <typename... KArgs, typename... Args>
static inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                             cudaStream_t stream, int cluster_x, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x > 1 ? cluster_x : 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster_x > 1 ? 2 : 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e == cudaSuccess) count_launch();
    return e;
}

template <typename... KArgs, typename... Args>
static inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t stream, Args&&... args) {
    return launch_pdl_cluster(kernel, grid, block, smem, stream, 1, std::forward<Args>(args)...);
}

// ------------------------------------------------ thread-block clusters

// The address of the same shared-memory object in cluster CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, int rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from this CTA's shared memory to shared memory of a CTA of the cluster
// (`dst`, `mbar`: addresses from dsmem_addr); the copy's bytes complete a
// transaction on that CTA's mbarrier `mbar`.  The source must stay unchanged
// until the receiver has seen the bytes arrive.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "r"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}
// Split cluster barrier, executed by every thread of every CTA of the
// cluster (warp-aligned): arrive without ordering, then wait (acquire).
// A fence.mbarrier_init before the arrive publishes barrier initialisation.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

int launch_status();                    // FP8KV_OK or FP8KV_ERR_CUDA after a launch
int num_sms();                          // SM count of the current device
void set_dispatch(const char* text);    // per-thread record of the last dispatch
int status_insert(unsigned int* s, int clear);     // insert.cu
int status_attention(unsigned int* s, int clear);  // attention.cu

// OR this translation unit's status word into *s, optionally clearing it.
static inline int read_status(unsigned int* s, int clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(v)) != cudaSuccess) return FP8KV_ERR_CUDA;
    if (clear) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_status, &z, sizeof(z)) != cudaSuccess) return FP8KV_ERR_CUDA;
    }
    *s |= v;
    return FP8KV_OK;
}
}  // namespace fp8kv
