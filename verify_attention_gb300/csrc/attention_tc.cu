// attention_tc.cu -- paged verifier attention on the 5th-generation tensor
// cores (tcgen05), for M x G query rows per KV head in (48, 128]: the M = 12,
// G = 9 verifier of "Laguna S 2.1 INT4 -- calibrated FP8 KV on Intel B70"
// ("Contract": width 12; "Initial optimization order", item 2: exact M12 paged
// attention) over the E4M3 cache ("Laguna S 2.1 KV-cache precision decision",
// property table: scale/dequantize on read).
//
// One CTA per (partition, KV head, sequence), 8 warps:
//   warp 0     TMA producer: 64-key tiles of E4M3 K and V (one page of 64 or
//              two pages of 32) into a 4-deep staging ring; owns TMEM.
//   warp 1     MMA issuer (one thread): S = Q.K^T (M=128, N=64, K=128) into a
//              double-buffered TMEM tile, then O += P.V (M=128, N=128, K=64)
//              into TMEM; completion through tcgen05.commit -> mbarrier.
//   warps 2-3  converters: E4M3 -> f16 (exact) into 128B-swizzled smem tiles,
//              K as the K-major B operand, V as the MN-major B operand.
//   warps 4-7  softmax, one thread per query row: tcgen05.ld of the S row,
//              mask, online softmax (log2 domain, lazy O rescale when the row
//              maximum grows by more than 2^8), P as f16 written back over S
//              with tcgen05.st; it becomes the A operand of P.V straight from
//              TMEM.  Q lives in TMEM too (A operand of Q.K^T).
// TMEM: Q 64 columns, S/P 2 x 64, O 128 (512 allocated).
#include <mutex>
#include <set>
#include <utility>

#include "attention.cuh"
#include "common.cuh"
#include "tcgen05_tmem.cuh"

namespace fp8kv {

int status_attention_tc(unsigned int* s, int clear) { return read_status(s, clear); }

namespace tc {

constexpr int NK = 64;                          // keys per tile
constexpr int STAGES = 4;                       // E4M3 staging tiles
constexpr int STG_BYTES = 2 * NK * 128;         // K + V E4M3: 16 KiB
constexpr int F16_BYTES = 2 * NK * 256;         // K + V f16: 32 KiB
constexpr int SMEM = STAGES * STG_BYTES + 2 * F16_BYTES + 1024 + 512;
constexpr uint32_t TM_Q = 0, TM_S = 64, TM_O = 256, TM_COLS = 512;
constexpr int THREADS = 256;

// barrier slots
enum {
    B_STG_FULL = 0,
    B_STG_EMPTY = B_STG_FULL + STAGES,
    B_KV_FULL = B_STG_EMPTY + STAGES,
    B_KV_EMPTY = B_KV_FULL + 2,
    B_S_FULL = B_KV_EMPTY + 2,
    B_P_FULL = B_S_FULL + 2,
    B_O_DONE = B_P_FULL + 2,
    B_O_FINAL = B_O_DONE + 1,
    B_Q_READY = B_O_FINAL + 1,
    B_MMA_IDLE = B_Q_READY + 1,
    B_COUNT = B_MMA_IDLE + 1
};

// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2), sm_100
// descriptor version 1; offsets in bytes.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: D fp32, A and B f16, A K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major) {
    return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accum) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accum)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16 E4M3 codes (one 16-byte chunk) -> 16 f16 (two 16-byte chunks), exact.
__device__ __forceinline__ void widen_chunk(uint4 c, uint4& lo, uint4& hi) {
    lo.x = e4m3x2_to_f16x2(c.x);
    lo.y = e4m3x2_to_f16x2(c.x >> 16);
    lo.z = e4m3x2_to_f16x2(c.y);
    lo.w = e4m3x2_to_f16x2(c.y >> 16);
    hi.x = e4m3x2_to_f16x2(c.z);
    hi.y = e4m3x2_to_f16x2(c.z >> 16);
    hi.z = e4m3x2_to_f16x2(c.w);
    hi.w = e4m3x2_to_f16x2(c.w >> 16);
}

// Converts one staged E4M3 tile (64 rows x 128 B, 128B-swizzled) into the f16
// layout the MMA reads: two 64-column blocks (dims 0-63, 64-127) of 64 rows x
// 128 B, 128B-swizzled.  The same layout serves as the K-major K operand and
// the MN-major V operand.  Rows flagged in `zero_mask` (bit r) are written as
// zeros.  64 threads, 8 chunks each; the write order alternates so that each
// quarter-warp hits 8 distinct 16-byte bank groups.
__device__ __forceinline__ void convert_tile(const uint8_t* src, uint8_t* dst, int ct, uint64_t zero_mask) {
#pragma unroll 2
    for (int u = 0; u < 8; ++u) {
        const int i = ct + 64 * u;
        const int r = i >> 3, c = i & 7;
        uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
        if (!((zero_mask >> r) & 1)) {
            const uint4 code = *(const uint4*)(src + r * 128 + (((c ^ r) & 7) << 4));
            widen_chunk(code, lo, hi);
        }
        uint8_t* blk = dst + (c >> 2) * (NK * 128) + r * 128;
        const int c16 = 2 * (c & 3);
        if (c < 4) {
            *(uint4*)(blk + (((c16 ^ r) & 7) << 4)) = lo;
            *(uint4*)(blk + ((((c16 + 1) ^ r) & 7) << 4)) = hi;
        } else {
            *(uint4*)(blk + ((((c16 + 1) ^ r) & 7) << 4)) = hi;
            *(uint4*)(blk + (((c16 ^ r) & 7) << 4)) = lo;
        }
    }
}

template <int PS>
__global__ void __launch_bounds__(THREADS, 1) verify_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                              const __grid_constant__ CUtensorMap tm_v,
                                                              AttnParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* stg = smem;                                   // STAGES x 16 KiB
    uint8_t* f16buf = smem + STAGES * STG_BYTES;           // 2 x 32 KiB
    uint64_t* bars = (uint64_t*)(f16buf + 2 * F16_BYTES);
    uint32_t* tmem_slot = (uint32_t*)(bars + B_COUNT);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = P.seq_lens[b];
    if (L < P.M || L > P.max_seq_len || (L + PS - 1) / PS > P.mpps) {
        if (threadIdx.x == 0 && split == 0 && hk == 0) flag(FP8KV_DEV_BAD_SEQ_LEN);
        return;
    }
    const int lo0 = (P.window_left >= 0) ? max(0, L - P.M - P.window_left) : 0;
    const int first_page = lo0 / PS, last_page = (L - 1) / PS;
    const int nsplit_b = (last_page - first_page + P.split_pages) / P.split_pages;
    if (nsplit_b > P.num_splits) {
        if (threadIdx.x == 0 && split == 0) flag(FP8KV_DEV_BAD_SEQ_LEN);
        return;
    }
    if (split >= nsplit_b) return;
    const int page_begin = first_page + split * P.split_pages;
    const int n_pages = min(P.split_pages, last_page + 1 - page_begin);
    constexpr int PPT = NK / PS;                          // pages per tile
    const int n_tiles = (n_pages + PPT - 1) / PPT;
    const int k_begin = page_begin * PS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(B_STG_FULL + s), 1);
            mbar_init(bar(B_STG_EMPTY + s), 2);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_KV_FULL + s), 2);
            mbar_init(bar(B_KV_EMPTY + s), 1);
            mbar_init(bar(B_S_FULL + s), 1);
            mbar_init(bar(B_P_FULL + s), 4);
        }
        mbar_init(bar(B_O_DONE), 1);
        mbar_init(bar(B_O_FINAL), 1);
        mbar_init(bar(B_Q_READY), 4);
        mbar_init(bar(B_MMA_IDLE), 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        const uint64_t policy = policy_evict_first();
        const int32_t* bt = P.block_table + (int64_t)b * P.mpps + page_begin;
        int issued = 0;
        for (int base = 0; base < n_pages && ok; base += 32) {
            const int mine = (base + lane < n_pages) ? bt[base + lane] : 0;
            const int cnt = min(32, n_pages - base);
            for (int j = 0; j < cnt; ++j) {
                const int phys = __shfl_sync(0xffffffffu, mine, j);
                const int i = base + j;                   // page index in the partition
                const int t = i / PPT, pin = i % PPT;     // tile, page within the tile
                const int s = t % STAGES, use = t / STAGES;
                if (lane == 0) {
                    if (pin == 0) {
                        if (use > 0) ok = mbar_wait(bar(B_STG_EMPTY + s), (use - 1) & 1);
                        const int pages_here = min(PPT, n_pages - t * PPT);
                        if (ok) mbar_expect_tx(bar(B_STG_FULL + s), pages_here * PS * 128 * 2);
                    }
                    if (ok) {
                        const uint32_t dk = smem_u32(stg + s * STG_BYTES + pin * PS * 128);
                        const uint32_t dv = dk + NK * 128;
                        tma_load_3d(dk, &tm_k, 0, hk * PS, phys, bar(B_STG_FULL + s), policy);
                        tma_load_3d(dv, &tm_v, 0, hk * PS, phys, bar(B_STG_FULL + s), policy);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                issued = i + 1;
            }
        }
        if (lane == 0) {   // never leave with copies into this CTA's shared memory in flight
            const int t_issued = (issued + PPT - 1) / PPT;
            for (int t = max(0, t_issued - STAGES); t < t_issued; ++t)
                mbar_wait(bar(B_STG_FULL + t % STAGES), (t / STAGES) & 1);
        }
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_QK = idesc_f16(128, NK, false);
            constexpr uint32_t ID_PV = idesc_f16(128, 128, true);
            ok = mbar_wait(bar(B_Q_READY), 0);
            fence_after();
            for (int t = 0; t <= n_tiles && ok; ++t) {
                if (t < n_tiles) {
                    const int kb = t & 1;
                    ok = mbar_wait(bar(B_KV_FULL + kb), (t >> 1) & 1);
                    if (!ok) break;
                    fence_after();
                    const uint32_t kf = smem_u32(f16buf + kb * F16_BYTES);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t bd = sdesc(kf + (ks >> 2) * (NK * 128) + (ks & 3) * 32, 16, 1024);
                        mma_ts(tmem + TM_S + kb * 64, tmem + TM_Q + 8 * ks, bd, ID_QK, ks > 0);
                    }
                    mma_commit(bar(B_S_FULL + kb));
                }
                if (t >= 1) {
                    const int u = t - 1, ub = u & 1;
                    ok = mbar_wait(bar(B_P_FULL + ub), (u >> 1) & 1);
                    if (!ok) break;
                    fence_after();
                    const uint32_t vf = smem_u32(f16buf + ub * F16_BYTES + NK * 256);
#pragma unroll
                    for (int kk = 0; kk < NK / 16; ++kk) {
                        const uint64_t bd = sdesc(vf + kk * 2048, NK * 128, 1024);
                        mma_ts(tmem + TM_O, tmem + TM_S + ub * 64 + 8 * kk, bd, ID_PV, (u > 0 || kk > 0));
                    }
                    mma_commit(bar(B_O_DONE));
                    mma_commit(bar(B_KV_EMPTY + ub));
                    if (u == n_tiles - 1) mma_commit(bar(B_O_FINAL));
                }
            }
            // nothing the tensor cores still run may outlive the TMEM allocation
            mma_commit(bar(B_MMA_IDLE));
            mbar_wait(bar(B_MMA_IDLE), 0);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ---------------------------------------------------------- converters
        const int ct = threadIdx.x - 64;
        for (int t = 0; t < n_tiles; ++t) {
            const int s = t % STAGES, kb = t & 1;
            ok = mbar_wait(bar(B_STG_FULL + s), (t / STAGES) & 1);
            if (ok && t >= 2) ok = mbar_wait(bar(B_KV_EMPTY + kb), ((t >> 1) - 1) & 1);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            // rows of this tile outside every query row's range read as zeros
            // in V (stale or NaN bytes must not reach P.V); K needs no care
            // since those logits are masked
            const int k0 = k_begin + t * NK;
            const int pages_here = min(PPT, n_pages - t * PPT);
            const int zlo = max(0, min(NK, lo0 - k0));                       // rows [0, zlo) before every window
            const int zhi = max(0, min(min(NK, pages_here * PS), L - k0));   // rows [zhi, NK) past the end
            const uint64_t below = zlo >= 64 ? ~0ull : ((1ull << zlo) - 1);
            const uint64_t keep = zhi >= 64 ? ~0ull : ((1ull << zhi) - 1);
            const uint64_t zmask = below | ~keep;
            const uint8_t* src = stg + s * STG_BYTES;
            uint8_t* dst = f16buf + kb * F16_BYTES;
            convert_tile(src, dst, ct, 0);
            convert_tile(src + NK * 128, dst + NK * 256, ct, zmask);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(B_STG_EMPTY + s));
                mbar_arrive(bar(B_KV_FULL + kb));
            }
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        const int rr = min(r, P.R - 1);
        const int m = rr / P.G;
        const int p_r = L - P.M + m;
        const int lo_r = (P.window_left >= 0) ? max(0, p_r - P.window_left) : 0;
        float mult;
        {
            // Q row -> f16 with a power-of-two prescale putting the row maximum
            // in [2^14, 2^15) (exact for bf16 inputs), folded into the logit
            // multiplier with k_scale * sm_scale * log2(e)
            uint32_t qw[64];
            float amax = 0.f;
            const uint4* src = (const uint4*)(P.q + (((int64_t)b * P.M + m) * P.Hq + hk * P.G + rr % P.G) * 128);
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const uint4 w = (r < P.R) ? src[u] : make_uint4(0, 0, 0, 0);
                qw[4 * u] = w.x;
                qw[4 * u + 1] = w.y;
                qw[4 * u + 2] = w.z;
                qw[4 * u + 3] = w.w;
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(w.x)), fabsf(bf16_hi(w.x))),
                                         fmaxf(fabsf(bf16_lo(w.y)), fabsf(bf16_hi(w.y)))));
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(w.z)), fabsf(bf16_hi(w.z))),
                                         fmaxf(fabsf(bf16_lo(w.w)), fabsf(bf16_hi(w.w)))));
            }
            int e = 14;
            const uint32_t ab = __float_as_uint(amax);
            if (amax > 0.f && ((ab >> 23) & 0xff) != 0xff) {
                const int be = (int)((ab >> 23) & 0xff);
                e = be ? be - 127 : -127;
            }
            const int sh = max(-100, min(100, 14 - e));
            const float scale = ldexpf(1.0f, sh);
#pragma unroll
            for (int j = 0; j < 64; ++j) qw[j] = pack_f16x2(bf16_lo(qw[j]) * scale, bf16_hi(qw[j]) * scale);
            tmem_st_x64(lane_base + TM_Q, qw);
            tmem_wait_st();
            mult = (*P.k_scale) * P.sm_scale * 1.4426950408889634f * ldexpf(1.0f, -sh);
        }
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_Q_READY));

        // warp-uniform bounds: tiles strictly inside every row's range skip masking
        int pmin = p_r, lomax = lo_r;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            pmin = min(pmin, __shfl_xor_sync(0xffffffffu, pmin, off));
            lomax = max(lomax, __shfl_xor_sync(0xffffffffu, lomax, off));
        }
        float m_run = -INFINITY, l_run = 0.f;
        for (int t = 0; t < n_tiles; ++t) {
            const int sb = t & 1;
            ok = mbar_wait(bar(B_S_FULL + sb), (t >> 1) & 1);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            fence_after();
            uint32_t sv[64];
            tmem_ld_x64(lane_base + TM_S + sb * 64, sv);
            tmem_wait_ld();
            const int k0 = k_begin + t * NK;
            const bool need_mask = (k0 + NK - 1 > pmin) || (k0 < lomax);
            float smax = -INFINITY;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                float x = __uint_as_float(sv[j]);
                if (need_mask && (k0 + j > p_r || k0 + j < lo_r)) x = -INFINITY;
                sv[j] = __float_as_uint(x);
                smax = fmaxf(smax, x);
            }
            const float tmax = smax * mult;
            const bool rescale = (m_run != -INFINITY) && (tmax > m_run + 8.0f);
            if (__any_sync(0xffffffffu, rescale)) {
                // O rows of this warp hold P.V up to tile t-1: wait for it, then scale
                const bool okw = mbar_wait(bar(B_O_DONE), (t - 1) & 1);
                if (!__all_sync(0xffffffffu, okw)) { ok = false; break; }
                fence_after();
                const float alpha = rescale ? ex2(m_run - tmax) : 1.0f;
#pragma unroll 1
                for (int c = 0; c < 128; c += 32) {
                    uint32_t ov[32];
                    tmem_ld_x32(lane_base + TM_O + c, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
                    tmem_st_x32(lane_base + TM_O + c, ov);
                }
                tmem_wait_st();
                if (rescale) {
                    l_run *= alpha;
                    m_run = tmax;
                }
            }
            if (m_run == -INFINITY) m_run = tmax;           // first visible keys of this row
            float sum = 0.f;
            uint32_t pw[32];
            const float neg = (m_run == -INFINITY) ? 0.f : -m_run;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float x0 = __uint_as_float(sv[2 * j]), x1 = __uint_as_float(sv[2 * j + 1]);
                const float p0 = (x0 == -INFINITY) ? 0.f : ex2(fmaf(x0, mult, neg));
                const float p1 = (x1 == -INFINITY) ? 0.f : ex2(fmaf(x1, mult, neg));
                sum += p0 + p1;
                pw[j] = pack_f16x2(p0, p1);
            }
            l_run += sum;
            tmem_st_x32(lane_base + TM_S + sb * 64, pw);
            tmem_wait_st();
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_P_FULL + sb));
        }
        // ------------------------------------------------------------ epilogue
        if (ok) ok = mbar_wait(bar(B_O_FINAL), 0);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            fence_after();
            const float vs = *P.v_scale;
            const int64_t row_idx = ((int64_t)b * P.M + m) * P.Hq + hk * P.G + rr % P.G;
            const bool direct = nsplit_b == 1;
            const float f = direct ? vs / l_run : vs;
#pragma unroll 1
            for (int c = 0; c < 128; c += 32) {
                uint32_t ov[32];
                tmem_ld_x32(lane_base + TM_O + c, ov);
                tmem_wait_ld();
                if (r < P.R) {
                    if (direct) {
                        uint4* dst = (uint4*)(P.out + row_idx * 128 + c);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            dst[v4] = make_uint4(
                                pack_bf16x2(__uint_as_float(ov[8 * v4 + 0]) * f, __uint_as_float(ov[8 * v4 + 1]) * f),
                                pack_bf16x2(__uint_as_float(ov[8 * v4 + 2]) * f, __uint_as_float(ov[8 * v4 + 3]) * f),
                                pack_bf16x2(__uint_as_float(ov[8 * v4 + 4]) * f, __uint_as_float(ov[8 * v4 + 5]) * f),
                                pack_bf16x2(__uint_as_float(ov[8 * v4 + 6]) * f, __uint_as_float(ov[8 * v4 + 7]) * f));
                    } else {
                        float4* dst = (float4*)(P.ws_o + (row_idx * P.num_splits + split) * 128 + c);
#pragma unroll
                        for (int v4 = 0; v4 < 8; ++v4)
                            dst[v4] = make_float4(__uint_as_float(ov[4 * v4]) * f, __uint_as_float(ov[4 * v4 + 1]) * f,
                                                  __uint_as_float(ov[4 * v4 + 2]) * f,
                                                  __uint_as_float(ov[4 * v4 + 3]) * f);
                    }
                }
            }
            if (r < P.R && !direct) {
                P.ws_ml[(row_idx * P.num_splits + split) * 2] = m_run;
                P.ws_ml[(row_idx * P.num_splits + split) * 2 + 1] = l_run;
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TM_COLS) : "memory");
    }
}

}  // namespace tc

int launch_verify_tc(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& P, cudaStream_t s) {
    if (P.R > 128 || P.R <= 48) return FP8KV_ERR_UNSUPPORTED;
    if (P.page_size == 32 && (P.split_pages & 1)) return FP8KV_ERR_UNSUPPORTED;
    static std::mutex mu;
    static std::set<std::pair<int, const void*>> done;
    const void* kern = P.page_size == 32 ? (const void*)tc::verify_tc_kernel<32> : (const void*)tc::verify_tc_kernel<64>;
    {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return FP8KV_ERR_CUDA;
        std::lock_guard<std::mutex> lock(mu);
        if (!done.count({dev, kern})) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::SMEM) != cudaSuccess)
                return FP8KV_ERR_CUDA;
            done.insert({dev, kern});
        }
    }
    dim3 grid(P.num_splits, P.Hkv, P.B);
    if (P.page_size == 32)
        tc::verify_tc_kernel<32><<<grid, tc::THREADS, tc::SMEM, s>>>(tk, tv, P);
    else
        tc::verify_tc_kernel<64><<<grid, tc::THREADS, tc::SMEM, s>>>(tk, tv, P);
    return launch_status();
}

}  // namespace fp8kv
