// attention.cu -- exact paged decode / verifier attention over the FP8 (or
// BF16) KV cache, with split-KV partials and a log-sum-exp reduce kernel.
//
// Method: "exact q1/M12 paged attention" over the E4M3 cache with calibrated
// per-tensor scales ("Laguna S 2.1 INT4 -- calibrated FP8 KV on Intel B70",
// sections "Contract" and "Initial optimization order"); "scale/dequantize"
// on read ("Laguna S 2.1 KV-cache precision decision", property table); global
// and sliding-window layers, GQA with 8 KV heads of dimension 128 (same page,
// "BF16 versus FP8 in concrete terms"); page sizes 32 and 64 ("Laguna FP8 KV --
// replicated embedding win, page-32 build, and host boundary", section
// "Page-32 attention experiment").
//
// Kernel shape (one CTA per (partition, KV head, sequence)):
//  * a producer warp streams the (page, head) tiles of K and V -- each a
//    contiguous page_size x 128 block of the [page][head][slot][dim] cache --
//    into a ring of shared-memory stages with 3-D TMA loads (128-byte swizzle,
//    so the fragment reads below are bank-conflict free);
//  * consumer warps own 16 query rows each (the M x G rows of one KV head,
//    padded to 16) and run Q.K^T and P.V on the tensor cores (m16n8k16,
//    fp32 accumulate).  E4M3 codes are widened to f16 in registers (exact) and
//    Q is scaled by a per-row power of two into f16 range (exact for bf16);
//    the BF16 cache runs the same loop in bf16;
//  * online softmax in fp32 (log2 domain) with quad shuffles;
//  * when the M x G rows fit one row tile (decode), seven key groups of warps
//    split the pages of a partition, each with two or more stages in flight,
//    one CTA per SM (paged_decode_kernel); they are merged through shared
//    memory at the end;
//  * one partition per sequence writes bf16 output directly; otherwise each
//    partition writes (max, sum, unnormalised output) and attn_reduce_kernel
//    combines them (per row, over the partitions of that row's tile).
// More than 16 rows per KV head on an E4M3 cache go to the tcgen05 kernel
// (attention_tc.cu); this file also holds the plan, the reduce kernel and
// the C-ABI entry points.
#include <stdio.h>

#include "attention.cuh"
#include "common.cuh"

namespace fp8kv {

int status_attention(unsigned int* s, int clear) { return read_status(s, clear); }

constexpr int kMaxRowTiles = 9;          // M*G <= 144 on the mma.sync kernels
constexpr int kMaxM = 16384;             // query rows per sequence (prefill chunks; E4M3 cache)
// Bytes of K/V stages per CTA for several row tiles; for the decode shape
// (one row tile) the key groups, their stage budget and the register cap of
// the decode kernel.  Chosen by graph-timed sweeps on a 131072-token decode
// layer (key groups x stages, one CTA per SM): 4 x 1 at two CTAs per SM
// 4.24 TB/s, 4 x 3: 4.08, 5 x 2: 4.04, 6 x 2: 4.66, 7 x 2: 4.80.
constexpr int kStageBudget = 96 * 1024;
constexpr int kDecodeKeyGroups = 7;
constexpr int kDecodeStageBudget = 224 * 1024;
constexpr int kDecodeRegs = 200;

template <int PS, bool FP8>
struct Cfg {
    static constexpr int kElem = FP8 ? 1 : 2;
    static constexpr int kTileBytes = PS * 128 * kElem;          // one (page, head) tile
    static constexpr int kStageBytes = 2 * kTileBytes;           // K + V
    static constexpr int kStages = kStageBudget / kStageBytes;   // at 96 KiB: 12 / 6 / 6 / 3
    static int smem_bytes(int stages) { return stages * kStageBytes + 1024 /*align*/ + 512 /*barriers*/; }
};

// Visible key range of query row r (M*G rows per KV head, row = m*G + g).
struct RowPos {
    int p, lo;
};
__device__ __forceinline__ RowPos row_pos(int r, int R, int G, int L, int M, int wl) {
    if (r >= R) r = R - 1;                       // padding rows mirror the last row
    const int m = r / G;
    RowPos rp;
    rp.p = L - M + m;
    rp.lo = (wl >= 0) ? max(0, rp.p - wl) : 0;
    return rp;
}

// Smem byte offset of 16-byte chunk `ch` of row `row` in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t swz(int row, int ch) { return row * 128 + (((ch ^ row) & 7) << 4); }

template <int PS, bool FP8>
__device__ __forceinline__ void attention_body(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                               const AttnParams& P) {
    using C = Cfg<PS, FP8>;
    const int S = P.KW * P.SG;                                  // stages in use
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = (uint64_t*)(smem + S * C::kStageBytes);   // full[S], empty[S]

    const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_cons = P.NT * P.KW;
    const int SG = P.SG;
    pdl_launch_dependents();
    // barrier set-up reads no memory an earlier kernel may write: it overlaps
    // the tail of the previous kernel in the stream
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&bars[s]), 1);
            mbar_init(smem_u32(&bars[S + s]), P.NT);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_wait();
    const int L = P.seq_lens[b];
    if (L < P.M || L > P.max_seq_len || (L + PS - 1) / PS > P.mpps) {
        if (threadIdx.x == 0 && split == 0 && hk == 0) flag(FP8KV_DEV_BAD_SEQ_LEN);
        return;
    }
    const int lo0 = (P.window_left >= 0) ? max(0, L - P.M - P.window_left) : 0;
    const int first_page = lo0 / PS, last_page = (L - 1) / PS;
    const int nsplit_b = (last_page - first_page + P.split_pages) / P.split_pages;
    if (nsplit_b > P.num_splits) {   // cannot happen when L <= max_seq_len; never index past the plan
        if (threadIdx.x == 0 && split == 0) flag(FP8KV_DEV_BAD_SEQ_LEN);
        return;
    }
    if (split >= nsplit_b) return;
    const int page_begin = first_page + split * P.split_pages;
    const int n_pages = min(P.split_pages, last_page + 1 - page_begin);

    // Each key group owns SG consecutive stages.  Page i of this partition goes
    // to group i % KW, its j-th page (j = i / KW) to stage g*SG + j % SG, use
    // j / SG of that stage: every wait below is for the next phase of a barrier
    // only its own consumer advances, so a parity test can never pass early.

    if (warp == n_cons) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        const uint64_t policy = policy_evict_first();
        const int32_t* bt = P.block_table + (int64_t)b * P.mpps + page_begin;
        bool ok = true;
        if (PS == 32) {
            // Lane l < KW feeds key group l: its pages l, l + KW, ... in order,
            // each as soon as that group's next stage is free (polled, so that
            // no group waits for another), the lanes' copies going out in one
            // instruction.  One lane issuing every 4 KiB page in turn caps the
            // staging rate well below HBM's at this page size (at page 64 the
            // two ways measure the same on E4M3 and the serial one is faster
            // on BF16).
            const bool feeder = lane < P.KW;
            int nx = lane;                                  // next page of this lane's group
            int phys = (feeder && nx < n_pages) ? bt[nx] : 0;
            int phys_next = (feeder && nx + P.KW < n_pages) ? bt[nx + P.KW] : 0;
            uint64_t t_progress = globaltimer();
            uint32_t idle = 0;
            while (true) {
                const bool mine = feeder && nx < n_pages;
                if (!__any_sync(0xffffffffu, mine)) break;
                bool go = false;
                int s = 0;
                if (mine) {
                    const int jj = nx / P.KW, use = jj / SG;
                    s = lane * SG + jj % SG;
                    go = use == 0 || mbar_test(smem_u32(&bars[S + s]), (use - 1) & 1);
                }
                if (go) {
                    const uint32_t full = smem_u32(&bars[s]);
                    const uint32_t dk = smem_u32(smem + s * C::kStageBytes);
                    const uint32_t dv = dk + C::kTileBytes;
                    mbar_expect_tx(full, C::kStageBytes);
                    if (FP8) {
                        tma_load_3d(dk, &tm_k, 0, hk * PS, phys, full, policy);
                        tma_load_3d(dv, &tm_v, 0, hk * PS, phys, full, policy);
                    } else {
                        tma_load_3d(dk, &tm_k, 0, hk * PS, phys, full, policy);
                        tma_load_3d(dk + PS * 128, &tm_k, 64, hk * PS, phys, full, policy);
                        tma_load_3d(dv, &tm_v, 0, hk * PS, phys, full, policy);
                        tma_load_3d(dv + PS * 128, &tm_v, 64, hk * PS, phys, full, policy);
                    }
                    nx += P.KW;
                    phys = phys_next;
                    phys_next = (nx + P.KW < n_pages) ? bt[nx + P.KW] : 0;
                }
                if (__any_sync(0xffffffffu, go)) {
                    idle = 0;
                    t_progress = globaltimer();
                    continue;
                }
                if (globaltimer() - t_progress > 2000000000ull) {   // no stage freed for 2 s
                    if (lane == 0) flag(FP8KV_DEV_WAIT_TIMEOUT);
                    break;
                }
                __nanosleep(16u << min(idle++, 4u));
            }
            // Do not leave while copies into this CTA's shared memory are in
            // flight: each feeder waits for the last stages it filled.
            if (feeder) {
                const int k_issued = (nx - lane) / P.KW;           // pages this lane issued
                for (int j = max(0, k_issued - SG); j < k_issued; ++j)
                    mbar_wait(smem_u32(&bars[lane * SG + j % SG]), (j / SG) & 1);
            }
            return;
        }
        int issued = 0;
        // page ids 32 at a time, the next batch loaded while this one is issued
        int next = (lane < n_pages) ? bt[lane] : 0;
        for (int base = 0; base < n_pages && ok; base += 32) {
            const int mine = next;
            if (base + 32 < n_pages) next = (base + 32 + lane < n_pages) ? bt[base + 32 + lane] : 0;
            const int cnt = min(32, n_pages - base);
            for (int j = 0; j < cnt; ++j) {
                const int phys = __shfl_sync(0xffffffffu, mine, j);
                const int i = base + j;
                const int jj = i / P.KW, use = jj / SG;
                const int s = (i % P.KW) * SG + jj % SG;
                if (lane == 0) {
                    if (use > 0) ok = mbar_wait(smem_u32(&bars[S + s]), (use - 1) & 1);
                    if (ok) {
                        const uint32_t full = smem_u32(&bars[s]);
                        const uint32_t dk = smem_u32(smem + s * C::kStageBytes);
                        const uint32_t dv = dk + C::kTileBytes;
                        mbar_expect_tx(full, C::kStageBytes);
                        if (FP8) {
                            tma_load_3d(dk, &tm_k, 0, hk * PS, phys, full, policy);
                            tma_load_3d(dv, &tm_v, 0, hk * PS, phys, full, policy);
                        } else {
                            tma_load_3d(dk, &tm_k, 0, hk * PS, phys, full, policy);
                            tma_load_3d(dk + PS * 128, &tm_k, 64, hk * PS, phys, full, policy);
                            tma_load_3d(dv, &tm_v, 0, hk * PS, phys, full, policy);
                            tma_load_3d(dv + PS * 128, &tm_v, 64, hk * PS, phys, full, policy);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                ++issued;
            }
        }
        // Do not leave while copies into this CTA's shared memory are in flight.
        if (lane == 0) {
            for (int i = max(0, issued - P.KW * SG); i < issued; ++i) {
                const int jj = i / P.KW;
                mbar_wait(smem_u32(&bars[(i % P.KW) * SG + jj % SG]), (jj / SG) & 1);
            }
        }
        return;
    }
    if (warp > n_cons) return;

    // --------------------------------------------------------------- consumer
    const int rt = warp % P.NT, kg = warp / P.NT;
    const int g = lane >> 2, c = lane & 3;
    const int r0 = rt * 16 + g, r1 = r0 + 8;
    const RowPos rp0 = row_pos(r0, P.R, P.G, L, P.M, P.window_left);
    const RowPos rp1 = row_pos(r1, P.R, P.G, L, P.M, P.window_left);

    // Q fragments (A operand, 8 k-steps).  k-slot -> head-dim mapping:
    //   FP8 : k-step ks of thread c covers dims 32c + 4ks + {0,1 | 2,3}
    //   BF16: dims 16c + 4ks (ks < 4) or 64 + 16c + 4(ks-4)
    uint32_t qa[8][4];
    float mult[2];
    {
        float qf[2][32];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int r = hr ? r1 : r0;
#pragma unroll
            for (int j = 0; j < 32; ++j) qf[hr][j] = 0.f;
            if (r < P.R) {
                const int m = r / P.G, hq = hk * P.G + r % P.G;
                const uint4* src = (const uint4*)(P.q + (((int64_t)b * P.M + m) * P.Hq + hq) * 128);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int vec = FP8 ? (4 * c + u) : (u < 2 ? 2 * c + u : 8 + 2 * c + (u - 2));
                    const uint4 w = src[vec];
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        qf[hr][8 * u + 2 * e] = bf16_lo(ww[e]);
                        qf[hr][8 * u + 2 * e + 1] = bf16_hi(ww[e]);
                    }
                }
            }
        }
        const float log2e = 1.4426950408889634f;
        if (FP8) {
            const float ks = P.k_scale[P.scale_stride * hk];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                float amax = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(qf[hr][j]));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                // power-of-two prescale putting the row maximum in [2^14, 2^15)
                int e = 14;
                const uint32_t ab = __float_as_uint(amax);
                if (amax > 0.f && ((ab >> 23) & 0xff) != 0xff) {
                    const int be = (int)((ab >> 23) & 0xff);
                    e = be ? be - 127 : -127;
                }
                const int sh = max(-100, min(100, 14 - e));
                const float scale = ldexpf(1.0f, sh);
#pragma unroll
                for (int j = 0; j < 32; ++j) qf[hr][j] *= scale;
                mult[hr] = ks * P.sm_scale * log2e * ldexpf(1.0f, -sh);
            }
#pragma unroll
            for (int ks2 = 0; ks2 < 8; ++ks2) {
                qa[ks2][0] = pack_f16x2(qf[0][4 * ks2], qf[0][4 * ks2 + 1]);
                qa[ks2][1] = pack_f16x2(qf[1][4 * ks2], qf[1][4 * ks2 + 1]);
                qa[ks2][2] = pack_f16x2(qf[0][4 * ks2 + 2], qf[0][4 * ks2 + 3]);
                qa[ks2][3] = pack_f16x2(qf[1][4 * ks2 + 2], qf[1][4 * ks2 + 3]);
            }
        } else {
            mult[0] = mult[1] = P.sm_scale * log2e;
#pragma unroll
            for (int ks2 = 0; ks2 < 8; ++ks2) {
                qa[ks2][0] = pack_bf16x2(qf[0][4 * ks2], qf[0][4 * ks2 + 1]);
                qa[ks2][1] = pack_bf16x2(qf[1][4 * ks2], qf[1][4 * ks2 + 1]);
                qa[ks2][2] = pack_bf16x2(qf[0][4 * ks2 + 2], qf[0][4 * ks2 + 3]);
                qa[ks2][3] = pack_bf16x2(qf[1][4 * ks2 + 2], qf[1][4 * ks2 + 3]);
            }
        }
    }

    // warp-uniform bounds used to skip masking on interior chunks
    int pmin = min(rp0.p, rp1.p), lomax = max(rp0.lo, rp1.lo);
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
        pmin = min(pmin, __shfl_xor_sync(0xffffffffu, pmin, off));
        lomax = max(lomax, __shfl_xor_sync(0xffffffffu, lomax, off));
    }

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
    bool ok = true;

    for (int i = kg; i < n_pages; i += P.KW) {
        const int jj = i / P.KW;
        const int s = kg * SG + jj % SG;
        ok = mbar_wait(smem_u32(&bars[s]), (jj / SG) & 1);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const uint8_t* kt = smem + s * C::kStageBytes;
        const uint8_t* vt = kt + C::kTileBytes;
        const int kpage = (page_begin + i) * PS;

#pragma unroll 1
        for (int ch32 = 0; ch32 < PS / 32; ++ch32) {
            const int kfirst = kpage + 32 * ch32;
            // ---- S = Q K^T for 32 keys (4 n-tiles of 8 keys)
            float sacc[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
                const int row = 32 * ch32 + 8 * nt + g;
                if (FP8) {
                    const uint4 k0 = *(const uint4*)(kt + swz(row, 2 * c));
                    const uint4 k1 = *(const uint4*)(kt + swz(row, 2 * c + 1));
                    const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
                    for (int ks2 = 0; ks2 < 8; ++ks2)
                        mma_f16(sacc[nt], qa[ks2], e4m3x2_to_f16x2(kw[ks2]), e4m3x2_to_f16x2(kw[ks2] >> 16));
                } else {
                    const uint4 k0 = *(const uint4*)(kt + swz(row, 2 * c));
                    const uint4 k1 = *(const uint4*)(kt + swz(row, 2 * c + 1));
                    const uint4 k2 = *(const uint4*)(kt + PS * 128 + swz(row, 2 * c));
                    const uint4 k3 = *(const uint4*)(kt + PS * 128 + swz(row, 2 * c + 1));
                    mma_bf16(sacc[nt], qa[0], k0.x, k0.y);
                    mma_bf16(sacc[nt], qa[1], k0.z, k0.w);
                    mma_bf16(sacc[nt], qa[2], k1.x, k1.y);
                    mma_bf16(sacc[nt], qa[3], k1.z, k1.w);
                    mma_bf16(sacc[nt], qa[4], k2.x, k2.y);
                    mma_bf16(sacc[nt], qa[5], k2.z, k2.w);
                    mma_bf16(sacc[nt], qa[6], k3.x, k3.y);
                    mma_bf16(sacc[nt], qa[7], k3.z, k3.w);
                }
            }
            // ---- scale to log2 units, mask, online softmax
            const bool need_mask = (kfirst + 31 > pmin) || (kfirst < lomax);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float t = sacc[nt][e] * mult[e >> 1];
                    if (need_mask) {
                        const int key = kfirst + 8 * nt + 2 * c + (e & 1);
                        const RowPos& rp = (e >> 1) ? rp1 : rp0;
                        if (key > rp.p || key < rp.lo) t = -INFINITY;
                    }
                    sacc[nt][e] = t;
                }
            }
            float alpha[2];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                float tmax = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) tmax = fmaxf(tmax, fmaxf(sacc[nt][2 * hr], sacc[nt][2 * hr + 1]));
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
                const float mnew = fmaxf(mrow[hr], tmax);
                const float mref = (mnew == -INFINITY) ? 0.f : mnew;
                alpha[hr] = ex2(mrow[hr] - mref);
                mrow[hr] = mnew;
                float sum = 0.f;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    sacc[nt][2 * hr] = ex2(sacc[nt][2 * hr] - mref);
                    sacc[nt][2 * hr + 1] = ex2(sacc[nt][2 * hr + 1] - mref);
                    sum += sacc[nt][2 * hr] + sacc[nt][2 * hr + 1];
                }
                lrow[hr] = lrow[hr] * alpha[hr] + sum;
            }
            if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
                for (int i2 = 0; i2 < 16; ++i2) {
                    o[i2][0] *= alpha[0];
                    o[i2][1] *= alpha[0];
                    o[i2][2] *= alpha[1];
                    o[i2][3] *= alpha[1];
                }
            }
            // ---- O += P V  (2 k-steps of 16 keys)
            // keys outside every row's range (past the sequence end, or before
            // the first window) contribute exact zeros even if stale data there
            // is not finite
            const bool zero_v = (kfirst + 31 >= L) || (kfirst < lo0);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                uint32_t pa[4];
                if (FP8) {
                    pa[0] = pack_f16x2(sacc[2 * kk][0], sacc[2 * kk][1]);
                    pa[1] = pack_f16x2(sacc[2 * kk][2], sacc[2 * kk][3]);
                    pa[2] = pack_f16x2(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
                    pa[3] = pack_f16x2(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
                } else {
                    pa[0] = pack_bf16x2(sacc[2 * kk][0], sacc[2 * kk][1]);
                    pa[1] = pack_bf16x2(sacc[2 * kk][2], sacc[2 * kk][3]);
                    pa[2] = pack_bf16x2(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
                    pa[3] = pack_bf16x2(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
                }
                const int rA = 32 * ch32 + 16 * kk + 2 * c;   // keys rA, rA+1, rA+8, rA+9
                bool kz[4] = {false, false, false, false};
                if (zero_v) {
                    const int key = kpage + rA;
                    kz[0] = key >= L || key < lo0;
                    kz[1] = key + 1 >= L || key + 1 < lo0;
                    kz[2] = key + 8 >= L || key + 8 < lo0;
                    kz[3] = key + 9 >= L || key + 9 < lo0;
                }
                if (FP8) {
#pragma unroll
                    for (int T = 0; T < 4; ++T) {
                        const int chk = 2 * T + (g >> 2), wofs = (g & 3) * 4;
                        uint32_t w0 = *(const uint32_t*)(vt + swz(rA, chk) + wofs);
                        uint32_t w1 = *(const uint32_t*)(vt + swz(rA + 1, chk) + wofs);
                        uint32_t w8 = *(const uint32_t*)(vt + swz(rA + 8, chk) + wofs);
                        uint32_t w9 = *(const uint32_t*)(vt + swz(rA + 9, chk) + wofs);
                        if (kz[0]) w0 = 0;
                        if (kz[1]) w1 = 0;
                        if (kz[2]) w8 = 0;
                        if (kz[3]) w9 = 0;
                        const uint32_t a01 = prmt(w0, w1, 0x5140), b01 = prmt(w0, w1, 0x7362);
                        const uint32_t a89 = prmt(w8, w9, 0x5140), b89 = prmt(w8, w9, 0x7362);
                        mma_f16(o[4 * T + 0], pa, e4m3x2_to_f16x2(a01), e4m3x2_to_f16x2(a89));
                        mma_f16(o[4 * T + 1], pa, e4m3x2_to_f16x2(a01 >> 16), e4m3x2_to_f16x2(a89 >> 16));
                        mma_f16(o[4 * T + 2], pa, e4m3x2_to_f16x2(b01), e4m3x2_to_f16x2(b89));
                        mma_f16(o[4 * T + 3], pa, e4m3x2_to_f16x2(b01 >> 16), e4m3x2_to_f16x2(b89 >> 16));
                    }
                } else {
#pragma unroll
                    for (int T = 0; T < 8; ++T) {
                        const uint8_t* vh = vt + (T >> 2) * PS * 128;
                        const int chk = 2 * (T & 3) + (g >> 2), wofs = (g & 3) * 4;
                        uint32_t w0 = *(const uint32_t*)(vh + swz(rA, chk) + wofs);
                        uint32_t w1 = *(const uint32_t*)(vh + swz(rA + 1, chk) + wofs);
                        uint32_t w8 = *(const uint32_t*)(vh + swz(rA + 8, chk) + wofs);
                        uint32_t w9 = *(const uint32_t*)(vh + swz(rA + 9, chk) + wofs);
                        if (kz[0]) w0 = 0;
                        if (kz[1]) w1 = 0;
                        if (kz[2]) w8 = 0;
                        if (kz[3]) w9 = 0;
                        mma_bf16(o[2 * T + 0], pa, prmt(w0, w1, 0x5410), prmt(w8, w9, 0x5410));
                        mma_bf16(o[2 * T + 1], pa, prmt(w0, w1, 0x7632), prmt(w8, w9, 0x7632));
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars[S + s]));
    }

    // ------------------------------------------------------------ epilogue
    // all consumers are done with the stages (every issued copy was consumed),
    // so the ring is reused as the merge area: per (key group, row) 128 floats
    // of O, then m and l.
    asm volatile("bar.sync 1, %0;" ::"r"(n_cons * 32) : "memory");
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 1);
        lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 2);
    }
    constexpr int kRowStride = 132;   // floats
    float* mergef = (float*)smem;
    const int rows_pad = P.NT * 16;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int r = hr ? r1 : r0;
        float* dst = mergef + ((int64_t)kg * rows_pad + r) * kRowStride;
        if (FP8) {
#pragma unroll
            for (int T = 0; T < 4; ++T) {
                // n-tile 4T+i, column n -> dim 32T + 4n + i; this thread has n = 2c, 2c+1
                float4 lo4 = make_float4(o[4 * T + 0][2 * hr], o[4 * T + 1][2 * hr], o[4 * T + 2][2 * hr],
                                         o[4 * T + 3][2 * hr]);
                float4 hi4 = make_float4(o[4 * T + 0][2 * hr + 1], o[4 * T + 1][2 * hr + 1],
                                         o[4 * T + 2][2 * hr + 1], o[4 * T + 3][2 * hr + 1]);
                *(float4*)(dst + 32 * T + 8 * c) = lo4;
                *(float4*)(dst + 32 * T + 8 * c + 4) = hi4;
            }
        } else {
#pragma unroll
            for (int T = 0; T < 8; ++T) {
                // n-tile 2T+i, column n -> dim 16T + 2n + i
                *(float4*)(dst + 16 * T + 4 * c) = make_float4(o[2 * T][2 * hr], o[2 * T + 1][2 * hr],
                                                               o[2 * T][2 * hr + 1], o[2 * T + 1][2 * hr + 1]);
            }
        }
        if (c == 0) {
            dst[128] = mrow[hr];
            dst[129] = lrow[hr];
        }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(n_cons * 32) : "memory");
    if (!ok) return;

    const float vs = FP8 ? P.v_scale[P.scale_stride * hk] : 1.0f;
    const int tid = threadIdx.x;
    for (int item = tid; item < P.R * 32; item += n_cons * 32) {
        const int r = item >> 5, d4 = (item & 31) * 4;
        float mstar = -INFINITY;
        for (int k2 = 0; k2 < P.KW; ++k2) mstar = fmaxf(mstar, mergef[((int64_t)k2 * rows_pad + r) * kRowStride + 128]);
        float l = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (mstar != -INFINITY) {
            for (int k2 = 0; k2 < P.KW; ++k2) {
                const float* src = mergef + ((int64_t)k2 * rows_pad + r) * kRowStride;
                const float w = ex2(src[128] - mstar);
                l += w * src[129];
                const float4 v4 = *(const float4*)(src + d4);
                acc.x += w * v4.x;
                acc.y += w * v4.y;
                acc.z += w * v4.z;
                acc.w += w * v4.w;
            }
        }
        const int m = r / P.G, hq = hk * P.G + r % P.G;
        const int64_t row_idx = ((int64_t)b * P.M + m) * P.Hq + hq;
        if (nsplit_b == 1) {
            const float f = vs / l;
            *(uint2*)(P.out + row_idx * 128 + d4) =
                make_uint2(pack_bf16x2(acc.x * f, acc.y * f), pack_bf16x2(acc.z * f, acc.w * f));
        } else {
            float* wo = P.ws_o + (row_idx * P.num_splits + split) * 128 + d4;
            *(float4*)wo = make_float4(acc.x * vs, acc.y * vs, acc.z * vs, acc.w * vs);
            if (d4 == 0) {
                P.ws_ml[(row_idx * P.num_splits + split) * 2] = mstar;
                P.ws_ml[(row_idx * P.num_splits + split) * 2 + 1] = l;
            }
        }
    }
}

// Several row tiles (verifier rows on a BF16 cache, or more than 128 rows):
// up to ten warps, registers capped so that one CTA fits an SM.
template <int PS, bool FP8>
__global__ void __launch_bounds__(32 * (kMaxRowTiles + 1), 1) paged_attention_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, AttnParams P) {
    attention_body<PS, FP8>(tm_k, tm_v, P);
}

// One row tile (decode): a handful of key-group warps, each with two or more
// stages in flight, one CTA per SM; at most two warps per SM sub-partition,
// so the register cap can be high enough to keep every fragment resident.
template <int PS, bool FP8>
__global__ void __maxnreg__(kDecodeRegs) paged_decode_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, AttnParams P) {
    attention_body<PS, FP8>(tm_k, tm_v, P);
}

// One warp per output row (b, m, h): combine the partitions through their
// log-sum-exp.  Partials of the mma.sync kernels (F16 = false) are fp32
// unnormalised O_p * v_scale with (m_p, l_p):
//     O = sum_p 2^(m_p - m*) O_p / sum_p 2^(m_p - m*) l_p;
// those of the tensor-memory kernel (F16 = true) are f16 O_p / l_p in E4M3
// code units: O = v_scale * sum_p w_p O_p / sum_p w_p, w_p = 2^(m_p - m*) l_p.
// Longest-first order of the (sequence, partition) slots of a tcgen05 call
// with one row tile of R rows (q = b * num_splits + s): slots ranked by
// their number of 128-key tiles (in 63 classes of tiles_per_split), longest
// first, written to order[0 .. n) (n = slots that hold keys) and -1 after
// them.  One CTA.  Invalid sequence lengths hold no keys and are flagged as
// the attention kernel flags them.
__global__ void __launch_bounds__(512) lpt_order_kernel(const int32_t* __restrict__ seq_lens, int B, int M,
                                                        int R, int G, int mpps, int page_size, int window_left,
                                                        int split_pages, int num_splits, int max_seq_len,
                                                        int32_t* __restrict__ order) {
    __shared__ int count[64], start[64];
    pdl_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid < 64) count[tid] = 0;
    __syncthreads();
    pdl_wait();
    const int nslot = B * num_splits;
    const int tiles_per_split = split_pages * page_size / 128;
    auto cls = [&](int q) {
        const int b = q / num_splits, s = q % num_splits;
        const int L = seq_lens[b];
        if (L < M || L > max_seq_len || (L + page_size - 1) / page_size > mpps) {
            if (s == 0) flag(FP8KV_DEV_BAD_SEQ_LEN);
            return 0;
        }
        const int lo0 = (window_left >= 0) ? max(0, L - M - window_left) : 0;
        const int first_page = lo0 / page_size, last_page = (L - M + (R - 1) / G) / page_size;
        const int ns = (last_page - first_page + split_pages) / split_pages;
        if (ns > num_splits) {
            if (s == 0) flag(FP8KV_DEV_BAD_SEQ_LEN);
            return 0;
        }
        if (s >= ns) return 0;
        const int n_pages = min(split_pages, last_page + 1 - (first_page + s * split_pages));
        const int tiles = (n_pages * page_size + 127) / 128;
        return 1 + (tiles - 1) * 63 / tiles_per_split;
    };
    for (int q = tid; q < nslot; q += blockDim.x) {
        const int c = cls(q);
        if (c) atomicAdd(&count[c], 1);
    }
    __syncthreads();
    if (tid < 32) {
        // lane l: classes 63 - 2l and 62 - 2l, in that (descending) order
        const int c0 = 63 - 2 * lane, c1 = 62 - 2 * lane;
        const int n0 = count[c0], n1 = c1 > 0 ? count[c1] : 0;
        int incl = n0 + n1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += x;
        }
        start[c0] = incl - n0 - n1;
        if (c1 > 0) start[c1] = incl - n1;
        if (lane == 31) start[0] = incl;                 // slots with keys
    }
    __syncthreads();
    for (int j = start[0] + tid; j < nslot; j += blockDim.x) order[j] = -1;
    for (int q = tid; q < nslot; q += blockDim.x) {
        const int c = cls(q);
        if (c) order[atomicAdd(&start[c], 1)] = q;
    }
}

template <bool F16>
__global__ void __launch_bounds__(256) attn_reduce_kernel(const float* __restrict__ ws_o,
                                                          const float* __restrict__ ws_ml,
                                                          const int32_t* __restrict__ seq_lens, int B, int M,
                                                          int Hq, int G, int tile_rows, int mpps,
                                                          int page_size, int window_left, int split_pages,
                                                          int num_splits, int max_seq_len, const float* v_scale,
                                                          int scale_stride, uint16_t* out) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= (int64_t)B * M * Hq) return;
    const int b = (int)(row / ((int64_t)M * Hq));
    const int L = seq_lens[b];
    if (L < M || L > max_seq_len || (L + page_size - 1) / page_size > mpps) return;
    // the keys of this row's tile of tile_rows rows (row m * G + h % G of its
    // KV head), split into partitions exactly as the attention kernel did
    const int m = (int)(row / Hq % M), rk = m * G + (int)(row % Hq) % G;
    const int R0 = rk / tile_rows * tile_rows, RL = min(tile_rows, M * G - R0);
    const int lo0 = (window_left >= 0) ? max(0, L - M + R0 / G - window_left) : 0;
    const int first_page = lo0 / page_size, last_page = (L - M + (R0 + RL - 1) / G) / page_size;
    const int ns = (last_page - first_page + split_pages) / split_pages;
    if (ns <= 1 || ns > num_splits) return;
    const float* ml = ws_ml + row * num_splits * 2;
    const float* po = ws_o + row * num_splits * 128 + lane * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    if (F16) {
        const uint16_t* ph = (const uint16_t*)ws_o + row * num_splits * 128 + lane * 4;
        const float vs = v_scale[scale_stride * ((int)(row % Hq) / G)];   // this row's KV head
        if (ns <= 16) {
            // every load in flight at once: (max, sum) of partition j on lane j
            // and this lane's four dims of every partition; then the arithmetic
            const float2 mlj = lane < ns ? *(const float2*)(ml + 2 * lane) : make_float2(-INFINITY, 0.f);
            uint2 v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) v[u] = u < ns ? *(const uint2*)(ph + (int64_t)u * 128) : make_uint2(0, 0);
            float mstar = mlj.x;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) mstar = fmaxf(mstar, __shfl_xor_sync(0xffffffffu, mstar, off));
            const float w_l = (mlj.x == -INFINITY) ? 0.f : ex2(mlj.x - mstar) * mlj.y;
            den = w_l;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const float w = __shfl_sync(0xffffffffu, w_l, u);       // 0 past ns
                const float2 a2 = f16x2_to_f32x2(v[u].x), c2 = f16x2_to_f32x2(v[u].y);
                acc.x = fmaf(w, a2.x, acc.x);
                acc.y = fmaf(w, a2.y, acc.y);
                acc.z = fmaf(w, c2.x, acc.z);
                acc.w = fmaf(w, c2.y, acc.w);
            }
        } else {
            float mstar = -INFINITY;
            for (int s = lane; s < ns; s += 32) mstar = fmaxf(mstar, ml[2 * s]);
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) mstar = fmaxf(mstar, __shfl_xor_sync(0xffffffffu, mstar, off));
            for (int base = 0; base < ns; base += 32) {
                const int cnt = min(32, ns - base);
                const float2 mlj =
                    lane < cnt ? *(const float2*)(ml + 2 * (base + lane)) : make_float2(-INFINITY, 0.f);
                const float w_l = (mlj.x == -INFINITY) ? 0.f : ex2(mlj.x - mstar) * mlj.y;
                den += w_l;
                for (int j = 0; j < cnt; j += 8) {            // eight partial rows in flight
                    uint2 v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        v[u] = j + u < cnt ? *(const uint2*)(ph + (int64_t)(base + j + u) * 128) : make_uint2(0, 0);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const float w = __shfl_sync(0xffffffffu, w_l, (j + u) & 31);   // 0 past cnt
                        const float2 a2 = f16x2_to_f32x2(v[u].x), c2 = f16x2_to_f32x2(v[u].y);
                        acc.x = fmaf(w, a2.x, acc.x);
                        acc.y = fmaf(w, a2.y, acc.y);
                        acc.z = fmaf(w, c2.x, acc.z);
                        acc.w = fmaf(w, c2.y, acc.w);
                    }
                }
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
        const float f = vs / den;
        *(uint2*)(out + row * 128 + lane * 4) =
            make_uint2(pack_bf16x2(acc.x * f, acc.y * f), pack_bf16x2(acc.z * f, acc.w * f));
        return;
    }
    if (ns <= 16) {
        // every load in flight at once: lane j's (max, sum) of partition j and
        // this lane's four dims of every partition; then the arithmetic
        const float2 mlj = lane < ns ? *(const float2*)(ml + 2 * lane) : make_float2(-INFINITY, 0.f);
        float4 v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) v[u] = u < ns ? *(const float4*)(po + (int64_t)u * 128) : make_float4(0.f, 0.f, 0.f, 0.f);
        float mstar = mlj.x;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mstar = fmaxf(mstar, __shfl_xor_sync(0xffffffffu, mstar, off));
        const float w_l = (mlj.x == -INFINITY) ? 0.f : ex2(mlj.x - mstar);
        den = w_l * mlj.y;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const float w = __shfl_sync(0xffffffffu, w_l, u);       // 0 past ns
            acc.x += w * v[u].x;
            acc.y += w * v[u].y;
            acc.z += w * v[u].z;
            acc.w += w * v[u].w;
        }
    } else {
        // partition weights: lane j owns partitions j, j+32, ...
        float mstar = -INFINITY;
        for (int s = lane; s < ns; s += 32) mstar = fmaxf(mstar, ml[2 * s]);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mstar = fmaxf(mstar, __shfl_xor_sync(0xffffffffu, mstar, off));
        for (int base = 0; base < ns; base += 32) {
            const int s_l = base + lane;
            float w_l = 0.f;
            if (s_l < ns) {
                const float ms = ml[2 * s_l];
                w_l = (ms == -INFINITY) ? 0.f : ex2(ms - mstar);
                den += w_l * ml[2 * s_l + 1];
            }
            const int cnt = min(32, ns - base);
            int j = 0;
            for (; j + 8 <= cnt; j += 8) {         // eight partial rows in flight
                float4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = *(const float4*)(po + (int64_t)(base + j + u) * 128);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float w = __shfl_sync(0xffffffffu, w_l, j + u);
                    acc.x += w * v[u].x;
                    acc.y += w * v[u].y;
                    acc.z += w * v[u].z;
                    acc.w += w * v[u].w;
                }
            }
            for (; j < cnt; ++j) {
                const float w = __shfl_sync(0xffffffffu, w_l, j);
                const float4 v = *(const float4*)(po + (int64_t)(base + j) * 128);
                acc.x += w * v.x;
                acc.y += w * v.y;
                acc.z += w * v.z;
                acc.w += w * v.w;
            }
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    const float f = 1.0f / den;
    *(uint2*)(out + row * 128 + lane * 4) =
        make_uint2(pack_bf16x2(acc.x * f, acc.y * f), pack_bf16x2(acc.z * f, acc.w * f));
}

}  // namespace fp8kv

// =====================================================================  host

#include <cudaTypedefs.h>

#include <algorithm>
#include <map>
#include <set>
#include <utility>

#include <mutex>

namespace fp8kv {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    });
    return fn;
}

// 3-D view of a [num_pages][Hkv][PS][128] cache: x = element within the row,
// y = head * PS + slot, z = page.  One box is one (page, head) tile (bf16 rows
// are fetched as two 64-element boxes so each box row is 128 bytes).
static bool make_cache_map(CUtensorMap* m, const void* base, bool fp8, int Hkv, int PS, int num_pages) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t elem = fp8 ? 1 : 2;
    cuuint64_t dims[3] = {128, (cuuint64_t)Hkv * PS, (cuuint64_t)num_pages};
    cuuint64_t strides[2] = {128 * elem, (cuuint64_t)Hkv * PS * 128 * elem};
    cuuint32_t box[3] = {fp8 ? 128u : 64u, (cuuint32_t)PS, 1u};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                    const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor maps by (cache base, dtype, heads, page size, pages): a map is a pure
// function of these, so repeated calls over the same persistent cache reuse
// it instead of encoding it again.  A small direct-mapped table per process.
struct MapKey {
    const void* base;
    int fp8, Hkv, PS, num_pages;
    bool operator==(const MapKey& o) const {
        return base == o.base && fp8 == o.fp8 && Hkv == o.Hkv && PS == o.PS && num_pages == o.num_pages;
    }
};

bool cache_map(CUtensorMap* m, const void* base, bool fp8, int Hkv, int PS, int num_pages) {
    constexpr int kSlots = 512;
    struct Entry {
        MapKey key;
        CUtensorMap map;
        bool valid;
    };
    static Entry table[kSlots];
    static std::mutex mu;
    const MapKey key{base, fp8 ? 1 : 0, Hkv, PS, num_pages};
    const size_t h = ((reinterpret_cast<uintptr_t>(base) >> 8) ^ (size_t)num_pages * 131 ^ (size_t)PS * 7 ^
                      (size_t)Hkv * 3 ^ (size_t)key.fp8) % kSlots;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (table[h].valid && table[h].key == key) {
            *m = table[h].map;
            return true;
        }
    }
    if (!make_cache_map(m, base, fp8, Hkv, PS, num_pages)) return false;
    std::lock_guard<std::mutex> lock(mu);
    table[h].key = key;
    table[h].map = *m;
    table[h].valid = true;
    return true;
}

struct Plan {
    int split_pages, num_splits, split_tokens;
};

static int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// 128-row tiles of the tcgen05 kernel per (sequence, KV head).
static int row_tiles(int M, int Hq, int Hkv) { return ceil_div((int64_t)M * (Hq / Hkv), 128); }

static int check_sizes(int B, int M, int Hq, int Hkv, int D, int PS, int max_seq_len, int window_left,
                       int split_tokens) {
    if (B < 0 || M < 1 || Hq <= 0 || Hkv <= 0 || max_seq_len < 0 || window_left < -1 || split_tokens < 0)
        return FP8KV_ERR_INVALID_ARG;
    if (Hq % Hkv) return FP8KV_ERR_INVALID_ARG;
    if (D != 128 || (PS != 32 && PS != 64) || M > kMaxM) return FP8KV_ERR_UNSUPPORTED;
    // more than 16 rows per sequence or 144 per KV head: the row tiles of the
    // tcgen05 kernel (E4M3 cache, checked with the cache type)
    if ((int64_t)Hkv * row_tiles(M, Hq, Hkv) > 65535) return FP8KV_ERR_UNSUPPORTED;
    if (split_tokens % PS) return FP8KV_ERR_INVALID_ARG;
    if (B > 65535 || Hkv > 65535) return FP8KV_ERR_UNSUPPORTED;
    return FP8KV_OK;
}

// Rows per KV head served by the tcgen05 kernel (on an E4M3 cache): more
// than 16, in tiles of 128.
static bool tc_rows(int M, int Hq, int Hkv) { return (int64_t)M * (Hq / Hkv) > 16; }

// Shapes only the tcgen05 kernel serves: prefill-like row counts.
static bool tc_only(int M, int Hq, int Hkv) { return M > 16 || (int64_t)M * (Hq / Hkv) > 16 * kMaxRowTiles; }

static int make_plan(int B, int M, int Hq, int Hkv, int D, int PS, int max_seq_len, int window_left,
                     int split_tokens, Plan* p) {
    int rc = check_sizes(B, M, Hq, Hkv, D, PS, max_seq_len, window_left, split_tokens);
    if (rc) return rc;
    // pages spanned by the visible keys of the longest sequence
    int pages = ceil_div(max(max_seq_len, 1), PS);
    if (window_left >= 0) pages = min(pages, ceil_div((int64_t)M + window_left, PS) + 1);
    const int RT = tc_rows(M, Hq, Hkv) ? row_tiles(M, Hq, Hkv) : 1;
    int sp;
    if (split_tokens > 0) {
        sp = split_tokens / PS;
    } else {
        // one (decode: a single row tile, one CTA per SM; prefill: several
        // row tiles) or two partitions per SM over all (sequence, head, row
        // tile) units, with at least 1024 keys per partition: per-CTA set-up
        // and the partial write-back make short partitions expensive
        const int64_t units = (int64_t)max(B, 1) * Hkv * RT;
        const int64_t target = (M * (Hq / Hkv) <= 16 || RT > 1 ? 1LL : 2LL) * num_sms();
        const int per = (int)std::max<int64_t>(1, (target + units - 1) / units);
        sp = max(ceil_div(pages, per), 1024 / PS);
        // with many units and long sequences, several partitions per sequence
        // keep the longest ones from holding an SM alone at the end of the
        // launch (sequence lengths are only known on the device): four on
        // the decode kernel, two where the verifier rows of several sequences
        // take their partitions longest first (prefill row tiles are many
        // units already, and every partition writes a partial per row)
        const int min_parts = (tc_rows(M, Hq, Hkv) && B > 1) ? 2 : 4;
        if (RT == 1 && ceil_div(pages, min_parts) >= 1024 / PS) sp = min(sp, ceil_div(pages, min_parts));
        // one sequence of verifier rows (one CTA per SM): at most 8 tiles of
        // 128 keys get a tile per partition (the partitions of a KV head then
        // run as one thread-block cluster and combine on chip); longer ones
        // one wave of partitions over the SMs, whole tiles each
        if (B == 1 && tc_rows(M, Hq, Hkv) && RT == 1) {
            const int tile_pages = max(1, tc_tile_tokens() / PS);
            const int tiles = ceil_div(pages, tile_pages);
            const int wave = max(1, num_sms() / Hkv);
            sp = tiles <= 8 ? tile_pages : tile_pages * ceil_div(tiles, min(tiles, wave));
        }
    }
    if (sp > pages) {
        // one partition: whole 128-key tiles still when the request had them
        const int tp = max(1, tc_tile_tokens() / PS);
        sp = (sp % tp == 0) ? ceil_div(pages, tp) * tp : pages;
    }
    sp = max(1, sp);
    // automatic partitions hold whole 128-key tiles of the tensor-memory kernel
    if (split_tokens == 0) {
        const int tile_pages = tc_tile_tokens() / PS;
        sp = (sp + tile_pages - 1) / tile_pages * tile_pages;
    }
    p->split_pages = sp;
    p->num_splits = ceil_div(pages, sp);
    p->split_tokens = sp * PS;
    return FP8KV_OK;
}

// Workspace: [partial O][partial (m, l)] when a sequence spans several
// partitions (reserved even when the partitions combine on chip).  The
// tcgen05 path writes f16 partial O in the first half of its area and keeps
// its longest-first slot order (B * num_splits ints) in the second half.
static size_t ws_bytes(int B, int M, int Hq, int Hkv, const Plan& p) {
    (void)Hkv;
    if (p.num_splits <= 1) return 0;
    return (size_t)B * M * Hq * p.num_splits * (128 + 2) * sizeof(float);
}

// Opt in to the kernel's dynamic shared memory once per device (so that calls
// made under CUDA-graph capture issue no attribute change).
static int ensure_smem(const void* kern, int bytes) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, int> done;   // largest size opted in so far
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8KV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find({dev, kern});
    if (it != done.end() && it->second >= bytes) return FP8KV_OK;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return FP8KV_ERR_CUDA;
    done[{dev, kern}] = bytes;
    return FP8KV_OK;
}

template <int PS, bool FP8>
static int launch(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& P, cudaStream_t s) {
    using C = Cfg<PS, FP8>;
    const bool decode = P.NT == 1;
    auto kern = decode ? paged_decode_kernel<PS, FP8> : paged_attention_kernel<PS, FP8>;
    const int max_stages = decode ? kDecodeStageBudget / C::kStageBytes : C::kStages;
    if (ensure_smem((const void*)kern, C::smem_bytes(std::max(max_stages, P.KW * P.SG)))) return FP8KV_ERR_CUDA;
    dim3 grid(P.num_splits, P.Hkv, P.B);
    cudaError_t e = launch_pdl(kern, grid, dim3((P.NT * P.KW + 1) * 32), C::smem_bytes(P.KW * P.SG), s, tk, tv, P);
    return e == cudaSuccess ? FP8KV_OK : (cudaGetLastError(), FP8KV_ERR_CUDA);
}

}  // namespace fp8kv

using namespace fp8kv;

extern "C" int fp8kv_paged_attention_plan(int B, int M, int Hq, int Hkv, int D, int page_size,
                                          int max_seq_len, int window_left, int split_tokens,
                                          int* num_splits, int* split_tokens_out) {
    Plan p;
    int rc = make_plan(B, M, Hq, Hkv, D, page_size, max_seq_len, window_left, split_tokens, &p);
    if (rc) return rc;
    if (num_splits) *num_splits = p.num_splits;
    if (split_tokens_out) *split_tokens_out = p.split_tokens;
    return FP8KV_OK;
}

extern "C" size_t fp8kv_paged_attention_workspace_size(int B, int M, int Hq, int Hkv, int D, int page_size,
                                                       int max_seq_len, int window_left, int split_tokens) {
    Plan p;
    if (make_plan(B, M, Hq, Hkv, D, page_size, max_seq_len, window_left, split_tokens, &p)) return (size_t)-1;
    return ws_bytes(B, M, Hq, Hkv, p);
}

static bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// The attention call; with k_new / v_new, the M new tokens of each sequence
// are first written to the cache at positions L - M + m (append).
static int attention_call(const void* k_new, const void* v_new, const void* q, const void* k_cache,
                          const void* v_cache, int cache_dtype, const int32_t* block_table, int max_pages_per_seq,
                          const int32_t* seq_lens, int max_seq_len, int B, int M, int Hq, int Hkv, int D,
                          int page_size, int num_pages, const float* k_scale, const float* v_scale, int scale_stride,
                          float sm_scale, int window_left, int split_tokens, void* workspace, size_t workspace_bytes,
                          void* out, void* stream) {
    if (cache_dtype != FP8KV_CACHE_E4M3 && cache_dtype != FP8KV_CACHE_BF16) return FP8KV_ERR_INVALID_ARG;
    const bool fp8 = cache_dtype == FP8KV_CACHE_E4M3;
    Plan plan;
    int rc = make_plan(B, M, Hq, Hkv, D, page_size, max_seq_len, window_left, split_tokens, &plan);
    if (rc) return rc;
    // more than 16 query rows per KV head on E4M3 pages, partitions of whole
    // 128-key tiles: tcgen05 kernel (128-row MMA tiles); otherwise mma.sync,
    // which serves at most 16 rows per sequence and 144 per KV head
    const bool use_tc = fp8 && tc_rows(M, Hq, Hkv) && (plan.split_tokens % tc_tile_tokens()) == 0;
    if (!use_tc && tc_only(M, Hq, Hkv)) return FP8KV_ERR_UNSUPPORTED;
    if (B == 0) return FP8KV_OK;                                // nothing to do; no pointer is read
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out) return FP8KV_ERR_INVALID_ARG;
    if ((k_new != nullptr) != (v_new != nullptr) || (k_new && (!al16(k_new) || !al16(v_new))))
        return FP8KV_ERR_INVALID_ARG;
    if (fp8 && (!k_scale || !v_scale)) return FP8KV_ERR_INVALID_ARG;
    if (!al16(q) || !al16(k_cache) || !al16(v_cache) || !al16(out)) return FP8KV_ERR_INVALID_ARG;
    if (num_pages <= 0 || max_pages_per_seq <= 0) return FP8KV_ERR_INVALID_ARG;
    if (max_seq_len < M || (int64_t)max_seq_len > (int64_t)max_pages_per_seq * page_size)
        return FP8KV_ERR_INVALID_ARG;
    if (!(sm_scale == sm_scale)) return FP8KV_ERR_INVALID_ARG;
    const size_t need = ws_bytes(B, M, Hq, Hkv, plan);
    if (need && (!workspace || workspace_bytes < need || !al16(workspace))) return FP8KV_ERR_WORKSPACE;

    CUtensorMap tk, tv;
    if (!cache_map(&tk, k_cache, fp8, Hkv, page_size, num_pages) ||
        !cache_map(&tv, v_cache, fp8, Hkv, page_size, num_pages))
        return FP8KV_ERR_CUDA;

    AttnParams P = {};
    P.q = (const uint16_t*)q;
    P.block_table = block_table;
    P.seq_lens = seq_lens;
    P.k_scale = k_scale;
    P.v_scale = v_scale;
    P.scale_stride = scale_stride;
    const size_t rows = (size_t)B * M * Hq;
    P.ws_o = plan.num_splits > 1 ? (float*)workspace : nullptr;
    P.ws_ml = plan.num_splits > 1 ? P.ws_o + rows * plan.num_splits * 128 : nullptr;
    P.out = (uint16_t*)out;
    P.sm_scale = sm_scale;
    P.mpps = max_pages_per_seq;
    P.B = B;
    P.M = M;
    P.Hq = Hq;
    P.Hkv = Hkv;
    P.G = Hq / Hkv;
    P.R = M * P.G;
    P.NT = (P.R + 15) / 16;
    P.KW = P.SG = 1;
    if (P.NT <= kMaxRowTiles) {
        // key groups split a partition's pages when one row tile leaves warps
        // idle; each group keeps at least two stages in flight when it can
        const int stages = page_size == 32 ? (fp8 ? Cfg<32, true>::kStages : Cfg<32, false>::kStages)
                                           : (fp8 ? Cfg<64, true>::kStages : Cfg<64, false>::kStages);
        const int elem_b = fp8 ? 1 : 2;
        const int dstages = kDecodeStageBudget / (2 * page_size * 128 * elem_b);
        int kw = P.NT == 1 ? kDecodeKeyGroups : (P.NT == 2 ? 2 : 1);
        const int avail = P.NT == 1 ? dstages : stages;
        kw = std::max(1, std::min(kw, avail));
        int sg = std::max(1, avail / kw);
        // the epilogue merges the key groups' rows through the stage ring
        const int elem = fp8 ? 1 : 2, stage_bytes = 2 * page_size * 128 * elem;
        const int merge = kw * P.NT * 16 * 132 * 4;
        while (kw * sg * stage_bytes < merge) ++sg;
        P.KW = kw;
        P.SG = sg;
    }
    P.window_left = window_left;
    P.split_pages = plan.split_pages;
    P.num_splits = plan.num_splits;
    P.page_size = page_size;
    P.max_seq_len = max_seq_len;

    cudaStream_t s = (cudaStream_t)stream;
    const int RT = use_tc ? row_tiles(M, Hq, Hkv) : 1;
    // one sequence in at most 8 partitions and one row tile: the partitions
    // of a KV head run as one thread-block cluster and combine in distributed
    // shared memory
    P.cluster = (use_tc && B == 1 && RT == 1 && plan.num_splits > 1 && plan.num_splits <= 8) ? plan.num_splits : 0;
    // several sequences split into partitions of unequal length: longest first
    const bool lpt = use_tc && B > 1 && RT == 1 && plan.num_splits > 1;
    if (lpt)
        P.lpt_order = (const int32_t*)((const uint8_t*)workspace +
                                       (size_t)B * M * Hq * plan.num_splits * 128 * sizeof(uint16_t));
    if (k_new && use_tc && RT == 1) {                               // appended in the kernel
        P.k_new = (const uint16_t*)k_new;
        P.v_new = (const uint16_t*)v_new;
        P.k_cache = (uint8_t*)k_cache;
        P.v_cache = (uint8_t*)v_cache;
        P.num_pages = num_pages;
    } else if (k_new) {
        rc = launch_append(k_new, v_new, seq_lens, block_table, max_pages_per_seq, B, M, Hkv, k_scale, v_scale,
                           scale_stride, (void*)k_cache, (void*)v_cache, num_pages, page_size, fp8, s);
        if (rc) return rc;
    }
    if (lpt) {
        const cudaError_t e =
            launch_pdl(lpt_order_kernel, dim3(1), dim3(512), 0, s, seq_lens, B, M, P.R, P.G, max_pages_per_seq,
                       page_size, window_left, plan.split_pages, plan.num_splits, max_seq_len, (int32_t*)P.lpt_order);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return FP8KV_ERR_CUDA;
        }
    }
    if (use_tc)
        rc = launch_attention_tc(tk, tv, P, s);
    else if (page_size == 32)
        rc = fp8 ? launch<32, true>(tk, tv, P, s) : launch<32, false>(tk, tv, P, s);
    else
        rc = fp8 ? launch<64, true>(tk, tv, P, s) : launch<64, false>(tk, tv, P, s);
    if (rc) return rc;
    if (plan.num_splits > 1 && P.cluster <= 1) {
        const int64_t warps = (int64_t)B * M * Hq;
        cudaError_t e = launch_pdl(use_tc ? attn_reduce_kernel<true> : attn_reduce_kernel<false>,
                                   dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, s, (const float*)P.ws_o,
                                   (const float*)P.ws_ml, seq_lens, B, M, Hq, P.G, use_tc ? 128 : P.R,
                                   max_pages_per_seq, page_size, window_left, plan.split_pages, plan.num_splits,
                                   max_seq_len, k_scale ? v_scale : nullptr, scale_stride, (uint16_t*)out);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return FP8KV_ERR_CUDA;
        }
    }
    char buf[256];
    if (use_tc)
        snprintf(buf, sizeof buf,
                 "attention_tc<ps=%d,e4m3> rows=%d row_tiles=%d tile=128x128 splits=%d split_tokens=%d "
                 "grid=%dx%dx%d threads=%d cluster=%d reduce=%d order=%s",
                 page_size, P.R, RT, plan.num_splits, plan.split_tokens, plan.num_splits, Hkv * RT, B, tc_threads(),
                 P.cluster > 1 ? P.cluster : 1, (plan.num_splits > 1 && P.cluster <= 1) ? 1 : 0,
                 lpt ? "longest_first" : "grid");
    else
        snprintf(buf, sizeof buf,
                 "%s<ps=%d,%s> rows=%d row_tiles=%d key_groups=%d stages_per_group=%d splits=%d "
                 "split_tokens=%d grid=%dx%dx%d threads=%d reduce=%d",
                 P.NT == 1 ? "paged_decode_mma" : "paged_attention_mma", page_size, fp8 ? "e4m3" : "bf16", P.R,
                 P.NT, P.KW, P.SG, plan.num_splits, plan.split_tokens,
                 plan.num_splits, Hkv, B, (P.NT * P.KW + 1) * 32, plan.num_splits > 1 ? 1 : 0);
    set_dispatch(buf);
    return FP8KV_OK;
}

extern "C" int fp8kv_paged_attention(const void* q, const void* k_cache, const void* v_cache, int cache_dtype,
                                     const int32_t* block_table, int max_pages_per_seq, const int32_t* seq_lens,
                                     int max_seq_len, int B, int M, int Hq, int Hkv, int D, int page_size,
                                     int num_pages, const float* k_scale, const float* v_scale, float sm_scale,
                                     int window_left, int split_tokens, void* workspace, size_t workspace_bytes,
                                     void* out, void* stream) {
    return attention_call(nullptr, nullptr, q, k_cache, v_cache, cache_dtype, block_table, max_pages_per_seq,
                          seq_lens, max_seq_len, B, M, Hq, Hkv, D, page_size, num_pages, k_scale, v_scale, 0,
                          sm_scale, window_left, split_tokens, workspace, workspace_bytes, out, stream);
}

extern "C" int fp8kv_paged_attention_per_head(const void* q, const void* k_cache, const void* v_cache,
                                              const int32_t* block_table, int max_pages_per_seq,
                                              const int32_t* seq_lens, int max_seq_len, int B, int M, int Hq,
                                              int Hkv, int D, int page_size, int num_pages, const float* k_scale,
                                              const float* v_scale, float sm_scale, int window_left,
                                              int split_tokens, void* workspace, size_t workspace_bytes, void* out,
                                              void* stream) {
    return attention_call(nullptr, nullptr, q, k_cache, v_cache, FP8KV_CACHE_E4M3, block_table, max_pages_per_seq,
                          seq_lens, max_seq_len, B, M, Hq, Hkv, D, page_size, num_pages, k_scale, v_scale, 1,
                          sm_scale, window_left, split_tokens, workspace, workspace_bytes, out, stream);
}

extern "C" int fp8kv_append_paged_attention(const void* k_new, const void* v_new, const void* q, void* k_cache,
                                            void* v_cache, int cache_dtype, const int32_t* block_table,
                                            int max_pages_per_seq, const int32_t* seq_lens, int max_seq_len, int B,
                                            int M, int Hq, int Hkv, int D, int page_size, int num_pages,
                                            const float* k_scale, const float* v_scale, float sm_scale,
                                            int window_left, int split_tokens, void* workspace,
                                            size_t workspace_bytes, void* out, void* stream) {
    if (B > 0 && (!k_new || !v_new)) return FP8KV_ERR_INVALID_ARG;
    return attention_call(k_new, v_new, q, k_cache, v_cache, cache_dtype, block_table, max_pages_per_seq, seq_lens,
                          max_seq_len, B, M, Hq, Hkv, D, page_size, num_pages, k_scale, v_scale, 0, sm_scale,
                          window_left, split_tokens, workspace, workspace_bytes, out, stream);
}

extern "C" int fp8kv_append_paged_attention_per_head(const void* k_new, const void* v_new, const void* q,
                                                     void* k_cache, void* v_cache, const int32_t* block_table,
                                                     int max_pages_per_seq, const int32_t* seq_lens, int max_seq_len,
                                                     int B, int M, int Hq, int Hkv, int D, int page_size,
                                                     int num_pages, const float* k_scale, const float* v_scale,
                                                     float sm_scale, int window_left, int split_tokens,
                                                     void* workspace, size_t workspace_bytes, void* out,
                                                     void* stream) {
    if (B > 0 && (!k_new || !v_new)) return FP8KV_ERR_INVALID_ARG;
    return attention_call(k_new, v_new, q, k_cache, v_cache, FP8KV_CACHE_E4M3, block_table, max_pages_per_seq,
                          seq_lens, max_seq_len, B, M, Hq, Hkv, D, page_size, num_pages, k_scale, v_scale, 1,
                          sm_scale, window_left, split_tokens, workspace, workspace_bytes, out, stream);
}

// ================================================ allocation-free variant
//
// Some callers cannot allocate device memory at the point where they run
// attention: code inside an allocator-free serving loop, callers with a
// memory pool that is already fully carved up, or host code that only has a
// raw stream and no allocator handle.  For them this entry point uses a
// file-scope device buffer as the split-KV workspace instead of a
// caller-provided one.  The buffer is fixed at load time, so every GPU that
// loads this library holds it until the process exits.

#define FP8KV_NOALLOC_WORKSPACE_BYTES (32u << 20)

static __device__ __align__(256) uint8_t g_noalloc_workspace[FP8KV_NOALLOC_WORKSPACE_BYTES];

// Device address of g_noalloc_workspace, looked up once per device with that
// device current (in host code the symbol is only a host-side stand-in).
static int noalloc_workspace(void** ptr) {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8KV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || !p) return FP8KV_ERR_CUDA;
        addr[dev] = p;
    }
    *ptr = addr[dev];
    return FP8KV_OK;
}

extern "C" int fp8kv_paged_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                             int cache_dtype, const int32_t* block_table, int max_pages_per_seq,
                                             const int32_t* seq_lens, int max_seq_len, int B, int M, int Hq,
                                             int Hkv, int D, int page_size, int num_pages, const float* k_scale,
                                             const float* v_scale, float sm_scale, int window_left,
                                             int split_tokens, void* out, void* stream) {
    const size_t need = fp8kv_paged_attention_workspace_size(B, M, Hq, Hkv, D, page_size, max_seq_len,
                                                             window_left, split_tokens);
    if (need == (size_t)-1 || need > FP8KV_NOALLOC_WORKSPACE_BYTES) {
        // the allocating entry point without a workspace: every argument check
        // runs first (same statuses), then a request that needs workspace
        // partials returns FP8KV_ERR_WORKSPACE; nothing is launched either way
        return fp8kv_paged_attention(q, k_cache, v_cache, cache_dtype, block_table, max_pages_per_seq, seq_lens,
                                     max_seq_len, B, M, Hq, Hkv, D, page_size, num_pages, k_scale, v_scale,
                                     sm_scale, window_left, split_tokens, nullptr, 0, out, stream);
    }
    void* ws = nullptr;
    if (need) {
        const int rc = noalloc_workspace(&ws);
        if (rc) return rc;
    }
    return fp8kv_paged_attention(q, k_cache, v_cache, cache_dtype, block_table, max_pages_per_seq, seq_lens,
                                 max_seq_len, B, M, Hq, Hkv, D, page_size, num_pages, k_scale, v_scale, sm_scale,
                                 window_left, split_tokens, ws, need ? FP8KV_NOALLOC_WORKSPACE_BYTES : 0, out,
                                 stream);
}
