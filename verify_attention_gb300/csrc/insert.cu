// insert.cu -- E4M3 KV-cache insertion and the fused Q/K RMSNorm + RoPE +
// insert boundary.
//
// "quantize, store FP8" on cache write with the checkpoint's static per-tensor
// scalar k/v scales ("Laguna S 2.1 KV-cache precision decision", sections "What
// the official checkpoint requests" and "BF16 versus FP8 in concrete terms";
// "Laguna S 2.1 INT4 -- calibrated FP8 KV on Intel B70", section "Contract"),
// optionally at the Q/K norm + RoPE boundary (same page, "Initial optimization
// order", item 3).
//
// Both kernels are HBM-bound streaming kernels: every thread moves 16 B of
// bf16 in and 8 B of codes out with one vector load and one vector store.
#include "attention.cuh"
#include "common.cuh"

namespace fp8kv {

int status_insert(unsigned int* s, int clear) { return read_status(s, clear); }

// ------------------------------------------------------------- plain insert

// One thread per (token, head, 8-element chunk); it handles that chunk of K
// and of V.  Rows whose slot is negative are skipped.
template <bool FP8>
__global__ void __launch_bounds__(256) insert_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, const int64_t* __restrict__ slots,
    int T, int Hkv, const float* __restrict__ k_scale, const float* __restrict__ v_scale, int scale_stride,
    uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache, int64_t num_slots, int page_size) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)T * Hkv * 16) return;
    const int chunk = (int)(i & 15);
    const int64_t row = i >> 4;                 // t * Hkv + h
    const int64_t t = row / Hkv;
    const int h = (int)(row - t * Hkv);
    // every load is independent of the others: issue them all before the
    // first use, one memory round trip instead of two
    const int64_t slot = slots[t];
    const uint4 kx = k[i], vx = v[i];
    // one scale per tensor (stride 0) or per KV head (stride 1)
    const float ks = FP8 ? k_scale[scale_stride * h] : 1.f, vs = FP8 ? v_scale[scale_stride * h] : 1.f;
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (chunk == 0) flag(FP8KV_DEV_BAD_SLOT);
        return;
    }
    const int64_t page = slot / page_size, off = slot - page * page_size;
    const int64_t dst = ((page * Hkv + h) * page_size + off) * 128 + chunk * 8;  // element index
    if (FP8) {
        *reinterpret_cast<uint2*>(k_cache + dst) = e4m3_encode8(kx, ks);
        *reinterpret_cast<uint2*>(v_cache + dst) = e4m3_encode8(vx, vs);
    } else {
        *reinterpret_cast<uint4*>(k_cache + dst * 2) = kx;
        *reinterpret_cast<uint4*>(v_cache + dst * 2) = vx;
    }
}

// ---------------------------------------------------------- append insert

// The M new tokens of every sequence to positions L_b - M + m, through the
// block table (the slots an insert of the verifier's new rows would name).
// One thread per (sequence, row, head, 8-element chunk).
template <bool FP8>
__global__ void __launch_bounds__(256) append_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, const int32_t* __restrict__ seq_lens,
    const int32_t* __restrict__ block_table, int mpps, int B, int M, int Hkv, const float* __restrict__ k_scale,
    const float* __restrict__ v_scale, int scale_stride, uint8_t* __restrict__ k_cache,
    uint8_t* __restrict__ v_cache, int num_pages, int page_size) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * M * Hkv * 16) return;
    const int chunk = (int)(i & 15);
    const int64_t row = i >> 4;                 // (b * M + m) * Hkv + h
    const int h = (int)(row % Hkv);
    const int64_t bm = row / Hkv;
    const int b = (int)(bm / M), m = (int)(bm % M);
    const int L = seq_lens[b];
    const uint4 kx = k[i], vx = v[i];
    const float ks = FP8 ? k_scale[scale_stride * h] : 1.f, vs = FP8 ? v_scale[scale_stride * h] : 1.f;
    const int pos = L - M + m;
    if (L < M || (L + page_size - 1) / page_size > mpps) {
        if (chunk == 0) flag(FP8KV_DEV_BAD_SEQ_LEN);
        return;
    }
    const int page = block_table[(int64_t)b * mpps + pos / page_size];
    if (page < 0 || page >= num_pages) {
        if (chunk == 0) flag(FP8KV_DEV_BAD_SLOT);
        return;
    }
    const int64_t dst = (((int64_t)page * Hkv + h) * page_size + pos % page_size) * 128 + chunk * 8;
    if (FP8) {
        *reinterpret_cast<uint2*>(k_cache + dst) = e4m3_encode8(kx, ks);
        *reinterpret_cast<uint2*>(v_cache + dst) = e4m3_encode8(vx, vs);
    } else {
        *reinterpret_cast<uint4*>(k_cache + dst * 2) = kx;
        *reinterpret_cast<uint4*>(v_cache + dst * 2) = vx;
    }
}

int launch_append(const void* k, const void* v, const int32_t* seq_lens, const int32_t* block_table, int mpps, int B,
                  int M, int Hkv, const float* k_scale, const float* v_scale, int scale_stride, void* k_cache,
                  void* v_cache, int num_pages, int page_size, bool fp8, cudaStream_t s) {
    const int64_t items = (int64_t)B * M * Hkv * 16;
    const int64_t blocks = (items + 255) / 256;
    if (blocks > 0x7fffffff) return FP8KV_ERR_UNSUPPORTED;
    cudaError_t e = launch_pdl(fp8 ? append_kernel<true> : append_kernel<false>, dim3((unsigned)blocks), dim3(256), 0,
                               s, (const uint4*)k, (const uint4*)v, seq_lens, block_table, mpps, B, M, Hkv, k_scale,
                               v_scale, scale_stride, (uint8_t*)k_cache, (uint8_t*)v_cache, num_pages, page_size);
    return e == cudaSuccess ? FP8KV_OK : (cudaGetLastError(), FP8KV_ERR_CUDA);
}

// ------------------------------------------------ fused RMSNorm+RoPE+insert

// One warp per (token, head) row; heads 0..Hq-1 are Q rows, Hq..Hq+Hkv-1 are
// K rows (whose warp also encodes the V row of the same head).  Lane l holds
// elements 4l..4l+3; the RoPE partner of element k < 64 is k + 64, held by
// lane l ^ 16.  Every fp32 operation uses an explicitly rounded intrinsic so
// the result is bit-reproducible.
__global__ void __launch_bounds__(256) norm_rope_insert_kernel(
    const uint2* __restrict__ q, const uint2* __restrict__ k, const uint2* __restrict__ v,
    const int64_t* __restrict__ positions, const uint2* __restrict__ q_w, const uint2* __restrict__ k_w,
    float eps, const float4* __restrict__ cos_sin, int max_pos, uint2* __restrict__ q_out,
    const int64_t* __restrict__ slots, int T, int Hq, int Hkv, const float* __restrict__ k_scale,
    const float* __restrict__ v_scale, uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
    int64_t num_slots, int page_size) {
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int heads = Hq + Hkv;
    if (row >= (int64_t)T * heads) return;
    const int64_t t = row / heads;
    const int hh = (int)(row - t * heads);
    const bool is_q = hh < Hq;
    const int h = is_q ? hh : hh - Hq;

    const int64_t pos = positions[t];
    if (pos < 0 || pos >= max_pos) {
        if (lane == 0 && hh == 0) flag(FP8KV_DEV_BAD_POSITION);
        return;
    }
    int64_t slot = -1;
    if (!is_q) {
        slot = slots[t];
        if (slot < 0) return;
        if (slot >= num_slots) {
            if (lane == 0) flag(FP8KV_DEV_BAD_SLOT);
            return;
        }
    }

    const uint2 xr = is_q ? q[(t * Hq + h) * 32 + lane] : k[(t * Hkv + h) * 32 + lane];
    const uint2 wr = is_q ? q_w[lane] : k_w[lane];
    float x[4] = {bf16_lo(xr.x), bf16_hi(xr.x), bf16_lo(xr.y), bf16_hi(xr.y)};
    float w[4] = {bf16_lo(wr.x), bf16_hi(wr.x), bf16_lo(wr.y), bf16_hi(wr.y)};

    // sum of squares: fixed per-lane fma chain, then a fixed butterfly
    float part = __fmul_rn(x[0], x[0]);
    part = __fmaf_rn(x[1], x[1], part);
    part = __fmaf_rn(x[2], x[2], part);
    part = __fmaf_rn(x[3], x[3], part);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, off));
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(part, 128.0f), eps)));

    float y[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float n = __bfloat162float(__float2bfloat16_rn(__fmul_rn(x[j], r)));
        y[j] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(n, w[j])));
    }
    float yp[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) yp[j] = __shfl_xor_sync(0xffffffffu, y[j], 16);

    const int kf = (4 * lane) & 63;                  // frequency index of element 0
    const float4 c = cos_sin[pos * 32 + kf / 4];
    const float4 s = cos_sin[pos * 32 + 16 + kf / 4];
    const float cc[4] = {c.x, c.y, c.z, c.w}, ss[4] = {s.x, s.y, s.z, s.w};
    float o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float val;
        if (lane < 16) val = __fmaf_rn(y[j], cc[j], -__fmul_rn(yp[j], ss[j]));   // k < 64
        else val = __fmaf_rn(y[j], cc[j], __fmul_rn(yp[j], ss[j]));             // k + 64
        o[j] = __bfloat162float(__float2bfloat16_rn(val));
    }

    if (is_q) {
        q_out[(t * Hq + h) * 32 + lane] = make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
        return;
    }
    const float ks = *k_scale, vs = *v_scale;
    const int64_t page = slot / page_size, off = slot - page * page_size;
    const int64_t dst = ((page * Hkv + h) * page_size + off) * 128 + 4 * lane;
    const uint32_t kc = e4m3x2(__fdiv_rn(o[0], ks), __fdiv_rn(o[1], ks)) |
                        (e4m3x2(__fdiv_rn(o[2], ks), __fdiv_rn(o[3], ks)) << 16);
    const uint2 vr = v[(t * Hkv + h) * 32 + lane];
    const uint32_t vc = e4m3x2(__fdiv_rn(bf16_lo(vr.x), vs), __fdiv_rn(bf16_hi(vr.x), vs)) |
                        (e4m3x2(__fdiv_rn(bf16_lo(vr.y), vs), __fdiv_rn(bf16_hi(vr.y), vs)) << 16);
    *reinterpret_cast<uint32_t*>(k_cache + dst) = kc;
    *reinterpret_cast<uint32_t*>(v_cache + dst) = vc;
}

// ---------------------------------------------------- encoder sweep kernel

__global__ void __launch_bounds__(256) encode_bits_kernel(uint32_t first, uint64_t n, uint8_t* out) {
    const uint64_t i = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
    if (i >= n) return;
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float a = __uint_as_float(first + (uint32_t)(i + 2 * j));
        const float b = __uint_as_float(first + (uint32_t)(i + 2 * j + 1));
        w[j] = e4m3x2(a, b);
    }
    if (i + 8 <= n && ((reinterpret_cast<uintptr_t>(out + i) & 7) == 0)) {
        *reinterpret_cast<uint2*>(out + i) = make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
    } else {
        for (int j = 0; j < 8 && i + j < n; ++j) out[i + j] = (uint8_t)(w[j / 2] >> (8 * (j & 1)));
    }
}

// ------------------------------------------------ bounded-wait self-test

// One warp waits on an mbarrier that nothing ever arrives on: the wait gives
// up after limit_ns, sets FP8KV_DEV_WAIT_TIMEOUT and the kernel returns like
// any pipeline kernel whose wait ran out (no trap, the context stays usable).
__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_barrier_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) (void)mbar_wait(smem_u32(&bar), 0, limit_ns);
    __syncwarp();
}

}  // namespace fp8kv

using namespace fp8kv;

extern "C" int fp8kv_selftest_bounded_wait(unsigned int limit_us, void* stream) {
    if (limit_us == 0 || limit_us > 2000000u) return FP8KV_ERR_INVALID_ARG;
    bounded_wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint64_t)limit_us * 1000ull);
    count_launch();
    return launch_status();
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

static int cache_insert(const void* k, const void* v, const int64_t* slot_mapping, int T, int Hkv, int D,
                        const float* k_scale, const float* v_scale, int scale_stride, void* k_cache, void* v_cache,
                        int num_pages, int page_size, int cache_dtype, void* stream) {
    if (T < 0 || Hkv <= 0 || num_pages <= 0) return FP8KV_ERR_INVALID_ARG;
    if (cache_dtype != FP8KV_CACHE_E4M3 && cache_dtype != FP8KV_CACHE_BF16) return FP8KV_ERR_INVALID_ARG;
    if (D != 128) return FP8KV_ERR_UNSUPPORTED;
    if (page_size != 32 && page_size != 64) return FP8KV_ERR_UNSUPPORTED;
    if (T == 0) return FP8KV_OK;                                // nothing to do; no pointer is read
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return FP8KV_ERR_INVALID_ARG;
    if (cache_dtype == FP8KV_CACHE_E4M3 && (!k_scale || !v_scale)) return FP8KV_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return FP8KV_ERR_INVALID_ARG;
    const int64_t items = (int64_t)T * Hkv * 16;
    const int threads = 256;
    const int64_t blocks = (items + threads - 1) / threads;
    if (blocks > 0x7fffffff) return FP8KV_ERR_UNSUPPORTED;
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t num_slots = (int64_t)num_pages * page_size;
    cudaError_t e = launch_pdl(cache_dtype == FP8KV_CACHE_E4M3 ? insert_kernel<true> : insert_kernel<false>,
                               dim3((unsigned)blocks), dim3(threads), 0, s, (const uint4*)k, (const uint4*)v,
                               slot_mapping, T, Hkv, k_scale, v_scale, scale_stride, (uint8_t*)k_cache,
                               (uint8_t*)v_cache, num_slots, page_size);
    return e == cudaSuccess ? FP8KV_OK : (cudaGetLastError(), FP8KV_ERR_CUDA);
}

extern "C" int fp8kv_cache_insert(const void* k, const void* v, const int64_t* slot_mapping, int T,
                                  int Hkv, int D, const float* k_scale, const float* v_scale,
                                  void* k_cache, void* v_cache, int num_pages, int page_size,
                                  int cache_dtype, void* stream) {
    return cache_insert(k, v, slot_mapping, T, Hkv, D, k_scale, v_scale, 0, k_cache, v_cache, num_pages, page_size,
                        cache_dtype, stream);
}

extern "C" int fp8kv_cache_insert_per_head(const void* k, const void* v, const int64_t* slot_mapping, int T,
                                           int Hkv, int D, const float* k_scale, const float* v_scale,
                                           void* k_cache, void* v_cache, int num_pages, int page_size,
                                           void* stream) {
    return cache_insert(k, v, slot_mapping, T, Hkv, D, k_scale, v_scale, 1, k_cache, v_cache, num_pages, page_size,
                        FP8KV_CACHE_E4M3, stream);
}

extern "C" int fp8kv_qk_norm_rope_insert(const void* q, const void* k, const void* v,
                                         const int64_t* positions, const void* q_norm_w,
                                         const void* k_norm_w, float eps, const float* cos_sin,
                                         int max_pos, void* q_out, const int64_t* slot_mapping, int T,
                                         int Hq, int Hkv, int D, const float* k_scale,
                                         const float* v_scale, void* k_cache, void* v_cache,
                                         int num_pages, int page_size, void* stream) {
    if (T < 0 || Hq <= 0 || Hkv <= 0 || num_pages <= 0 || max_pos <= 0) return FP8KV_ERR_INVALID_ARG;
    if (!(eps >= 0.0f)) return FP8KV_ERR_INVALID_ARG;
    if (D != 128) return FP8KV_ERR_UNSUPPORTED;
    if (page_size != 32 && page_size != 64) return FP8KV_ERR_UNSUPPORTED;
    if (T == 0) return FP8KV_OK;                                // nothing to do; no pointer is read
    if (!q || !k || !v || !positions || !q_norm_w || !k_norm_w || !cos_sin || !q_out || !slot_mapping ||
        !k_scale || !v_scale || !k_cache || !v_cache)
        return FP8KV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_out) || !aligned16(cos_sin) ||
        !aligned16(q_norm_w) || !aligned16(k_norm_w) || !aligned16(k_cache) || !aligned16(v_cache))
        return FP8KV_ERR_INVALID_ARG;
    if (q == q_out) return FP8KV_ERR_INVALID_ARG;
    const int64_t warps = (int64_t)T * (Hq + Hkv);
    const int64_t blocks = (warps + 7) / 8;
    if (blocks > 0x7fffffff) return FP8KV_ERR_UNSUPPORTED;
    cudaError_t e = launch_pdl(norm_rope_insert_kernel, dim3((unsigned)blocks), dim3(256), 0, (cudaStream_t)stream,
                               (const uint2*)q, (const uint2*)k, (const uint2*)v, positions, (const uint2*)q_norm_w,
                               (const uint2*)k_norm_w, eps, (const float4*)cos_sin, max_pos, (uint2*)q_out,
                               slot_mapping, T, Hq, Hkv, k_scale, v_scale, (uint8_t*)k_cache, (uint8_t*)v_cache,
                               (int64_t)num_pages * page_size, page_size);
    return e == cudaSuccess ? FP8KV_OK : (cudaGetLastError(), FP8KV_ERR_CUDA);
}

extern "C" int fp8kv_e4m3_encode_bits(uint32_t first, size_t n, uint8_t* out, void* stream) {
    if (!out) return FP8KV_ERR_INVALID_ARG;
    if (n == 0) return FP8KV_OK;
    if ((uint64_t)first + n > (1ull << 32)) return FP8KV_ERR_INVALID_ARG;
    const uint64_t threads_needed = (n + 7) / 8;
    const uint64_t blocks = (threads_needed + 255) / 256;
    encode_bits_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(first, (uint64_t)n, out);
    count_launch();
    return launch_status();
}
