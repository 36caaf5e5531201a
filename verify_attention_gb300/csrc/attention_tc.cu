// attention_tc.cu -- paged verifier attention on the 5th-generation tensor
// cores (tcgen05) for more than 16 query rows per KV head (M x G rows; the
// M = 12 verifier has 108, a prefill chunk of M tokens M x G in 128-row tiles,
// one CTA per tile, each loading the keys its rows see) of "Laguna S 2.1 INT4 --
// calibrated FP8 KV on Intel B70" ("Contract"; "Initial optimization order",
// item 2: exact q1/M12 paged attention) over the E4M3 cache ("Laguna S 2.1
// KV-cache precision decision", property table: "scale/dequantize or use native
// FP8 attention").
//
// Q.K^T runs natively in FP8: the E4M3 K tile is the B operand straight from
// the TMA staging buffer (its 128-byte rows with the 128-byte swizzle are the
// K-major operand layout), and each Q row is split in the kernel into two
// E4M3 terms after a per-row power-of-two scale, q' = q * 2^sh = Q_hi + Q_lo,
// which is exact for every bf16 element within 2^-10 of the row maximum (the
// rest is off by at most 2^-17 of the row maximum); the softmax warps store
// both into tensor memory (A operand) and two accumulating MMAs
// give S = q'.K.  P.V runs in f16: P (softmax weights) is written to tensor
// memory and is the A operand, V is widened E4M3 -> f16 (exact) into a
// swizzled MN-major tile.  Rows past M x G (up to 128) carry Q = 0.
//
// One CTA per (partition, row tile x KV head, sequence), 16 warps:
//   warp 0          TMA producer (128-key tiles: K and V E4M3, 2 or 4 pages);
//                   allocates and frees the tensor memory
//   warp 1          MMA issuer (one thread); completion via tcgen05.commit.
//                   Calls without tokens appended in the kernel issue P.V from
//                   a second thread (warp 15), each thread waiting only for
//                   its own operands: the tile loop is bound by the MMA issue
//                   chain, which one thread serialises with its waits
//   warps 2,3,12-15 V converters (192 threads; 160 when warp 15 issues P.V);
//                   with appended tokens they also encode those, one item
//                   per thread
//   warps 4-11      softmax: warps 4+q and 8+q share TMEM lane quarter q (32
//                   query rows, one per thread) and split the tile's 128 key
//                   columns in halves; the row maximum of a tile is exchanged
//                   through shared memory.  Masks, online softmax in the log2
//                   domain, lazy O rescale (only when a row maximum grows by
//                   more than 2^8), P to TMEM.
// TMEM columns: Q_hi 0-31, Q_lo 32-63, S/P 2 x 128 (64-319), O 320-447.
#include <cudaTypedefs.h>

#include <mutex>
#include <set>
#include <utility>

#include "attention.cuh"
#include "common.cuh"
#include "tcgen05.cuh"

namespace fp8kv {

int status_attention_tc(unsigned int* s, int clear) { return read_status(s, clear); }

namespace tc {

constexpr int NK = 128;                         // keys per tile
constexpr int STAGES = 3;                       // E4M3 staging tiles (K + V)
constexpr int STG_K = NK * 128;                 // 16 KiB
constexpr int STG_BYTES = 2 * STG_K;            // 32 KiB
constexpr int VBUFS = 2;                        // f16 V tiles
constexpr int VBUF_BYTES = NK * 256;            // 32 KiB
constexpr int XCH_BYTES = 3 * 2 * 128 * 4;      // [tile parity 0, parity 1, row sums][half][row]
// Cluster combine: the partials a CTA receives for the rows it owns (row r
// belongs to rank r mod C): C partitions x S slots, S = ceil(rows / C)
// rounded up to even (16-byte blocks of (max, sum)), an f16 row (O / l, 128
// dims) and fp32 (max, sum) each; at most 143 slots for C <= 8.
constexpr int RECV_SLOTS = 144;
constexpr int RECV_BYTES = RECV_SLOTS * (256 + 8);
constexpr int SMEM = STAGES * STG_BYTES + VBUFS * VBUF_BYTES + XCH_BYTES + RECV_BYTES + 1024 + 512;
// epilogue: one staged half row (<= 256 B) per (half, row), padded against
// bank conflicts, in the staging buffers (free once the last tile is consumed)
constexpr int EPI_STRIDE = 272;
static_assert(2 * 128 * EPI_STRIDE <= STAGES * STG_BYTES, "epilogue staging exceeds the stage ring");
constexpr uint32_t TM_QH = 0, TM_QL = 32, TM_S = 64, TM_O = 320, TM_COLS = 512;
constexpr int WARPS = 16, THREADS = WARPS * 32;
// V converters: six warps (2, 3, 12-15), or five (2, 3, 12-14) when warp 15
// issues P.V (DUAL: calls without appended tokens, whose converters also
// encode the new tokens at the start of the launch)
template <bool DUAL> __host__ __device__ constexpr int conv_warps() { return DUAL ? 5 : 6; }

enum {
    B_STG_FULL = 0,
    B_STG_EMPTY = B_STG_FULL + STAGES,
    B_V_FULL = B_STG_EMPTY + STAGES,
    B_V_EMPTY = B_V_FULL + VBUFS,
    B_S_FULL = B_V_EMPTY + VBUFS,
    B_P_FULL = B_S_FULL + 2,
    B_O_DONE = B_P_FULL + 2,
    B_O_FINAL = B_O_DONE + 1,
    B_Q_READY = B_O_FINAL + 1,
    B_MMA_IDLE = B_Q_READY + 1,
    B_PAIR = B_MMA_IDLE + 1,                    // one per TMEM lane quarter: the two softmax warps
    // append: new tokens patched into a staged tile, one barrier for each of
    // the (at most two) tiles that hold them, so that no waiter can fall a
    // whole phase behind
    B_PATCH = B_PAIR + 4,
    B_S_EMPTY = B_PATCH + 2,                    // per S buffer: P.V of the P over it done (DUAL)
    B_RECV = B_S_EMPTY + 2,                     // cluster combine: every partition's partial rows arrived
    B_COUNT = B_RECV + 1
};

// Named barrier 5 of the eight softmax warps that also ANDs `ok` over them.
__device__ __forceinline__ bool softmax_warps_all(bool ok) {
    uint32_t r;
    asm volatile("{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.and.pred q, 5, 256, p; selp.u32 %0, 1, 0, q; }"
                 : "=r"(r)
                 : "r"((uint32_t)ok)
                 : "memory");
    return r != 0;
}

template <bool DUAL>
__device__ __forceinline__ bool is_converter(int warp) { return warp == 2 || warp == 3 || (warp >= 12 && warp < 12 + conv_warps<DUAL>() - 2); }
__device__ __forceinline__ int converter_index(int warp) { return warp < 4 ? warp - 2 : warp - 10; }

// DUAL: Q.K^T (warp 1) and P.V (warp 15) are issued by two threads, each
// waiting only for its own operands; otherwise one thread issues Q.K^T(t)
// then P.V(t - 1).
template <int PS, bool DUAL>
__global__ void __launch_bounds__(THREADS, 1) attention_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                 const __grid_constant__ CUtensorMap tm_v,
                                                                 AttnParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* stg = smem;                                    // STAGES x (K 16 KiB, V 16 KiB)
    uint8_t* vbuf = smem + STAGES * STG_BYTES;              // VBUFS x 32 KiB
    float* xch = (float*)(vbuf + VBUFS * VBUF_BYTES);       // [parity][half][row]
    uint8_t* recv = (uint8_t*)xch + XCH_BYTES;              // [partition][slot] f16 rows
    float* recv_ml = (float*)(recv + RECV_SLOTS * 256);     // [partition][slot] (max, sum)
    uint64_t* bars = (uint64_t*)(recv + RECV_BYTES);
    uint32_t* tmem_slot = (uint32_t*)(bars + B_COUNT);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    constexpr int CONV_WARPS = conv_warps<DUAL>(), CONV_THREADS = CONV_WARPS * 32;

    // blockIdx.y = row tile + RT * KV head: the row tiles of one head are
    // neighbours in launch order and share its pages in L2
    const int RT = (P.R + 127) >> 7;
    const int rt = blockIdx.y % RT;
    int split = blockIdx.x, hk = blockIdx.y / RT, b = blockIdx.z;   // (longest-first: set after the wait)
    const int R0 = rt * 128, RL = min(128, P.R - R0);      // this CTA's rows R0 .. R0 + RL - 1
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_launch_dependents();

    // Set-up that reads no memory an earlier kernel may write: it overlaps
    // the tail of the previous kernel in the stream.
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(B_STG_FULL + s), 1);
            mbar_init(bar(B_STG_EMPTY + s), 1 + CONV_WARPS);   // QK commit + converters
        }
        for (int s = 0; s < VBUFS; ++s) {
            mbar_init(bar(B_V_FULL + s), CONV_WARPS);
            mbar_init(bar(B_V_EMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_S_FULL + s), 1);
            mbar_init(bar(B_P_FULL + s), 8);
        }
        mbar_init(bar(B_O_DONE), 1);
        mbar_init(bar(B_O_FINAL), 1);
        mbar_init(bar(B_Q_READY), 8);
        mbar_init(bar(B_MMA_IDLE), DUAL ? 2 : 1);               // the issuing threads
        mbar_init(bar(B_S_EMPTY), 1);
        mbar_init(bar(B_S_EMPTY + 1), 1);
        mbar_init(bar(B_PATCH), CONV_WARPS);
        mbar_init(bar(B_PATCH + 1), CONV_WARPS);
        for (int q = 0; q < 4; ++q) mbar_init(bar(B_PAIR + q), 2);
        mbar_init(bar(B_RECV), 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        if (lane == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    // cluster: every CTA has started and initialised its barriers before any
    // partial is sent (arrive here, wait before the wait for the previous kernel)
    if (P.cluster > 1) cluster_arrive_relaxed();
    if (warp == 1 && lane == 0 && !P.lpt_order) {
        // L2 prefetch of the block-table entries this partition will read,
        // located from a read of the sequence length made before the wait for
        // the previous kernel: a hint only (the length and the entries used
        // below are read after the wait), it takes the dependent DRAM round
        // trip of the block table off the path to the first page copy
        const int Lg = *(volatile const int*)(P.seq_lens + b);
        if (Lg >= P.M && Lg <= P.max_seq_len) {
            const int hi_g = Lg - P.M + (R0 + RL - 1) / P.G;
            const int lo_g = (P.window_left >= 0) ? max(0, Lg - P.M + R0 / P.G - P.window_left) : 0;
            const int pb = lo_g / PS + split * P.split_pages;
            const int pe = min(pb + P.split_pages, hi_g / PS + 1);
            const int32_t* row = P.block_table + (int64_t)b * P.mpps;
            const uintptr_t a0 = reinterpret_cast<uintptr_t>(row + pb) & ~(uintptr_t)127;
            const uintptr_t a1 = reinterpret_cast<uintptr_t>(row + min(pe, P.mpps));
            for (uintptr_t a = a0; a < a1; a += 128)        // 128-byte lines, usually one
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a) : "memory");
        }
    }

    if (P.cluster > 1) {
        __syncwarp();
        cluster_wait();
    }
    pdl_wait();
    // Converter thread ct's first append item is query m = ct / 16 whenever
    // the partition starts at or before the first new token (the usual case):
    // its K and V rows are loaded now, beside the sequence length, instead of
    // a round trip after it
    uint4 spec_k = make_uint4(0, 0, 0, 0), spec_v = make_uint4(0, 0, 0, 0);
    const int ct_spec = converter_index(warp) * 32 + lane;
    const bool spec = !DUAL && P.k_new != nullptr && !P.lpt_order && is_converter<DUAL>(warp) && ct_spec < P.M * 16;
    if (spec) {
        const int64_t src = (((int64_t)b * P.M + (ct_spec >> 4)) * P.Hkv + hk) * 16 + (ct_spec & 15);
        spec_k = ((const uint4*)P.k_new)[src];
        spec_v = ((const uint4*)P.v_new)[src];
    }
    bool have_work = true;
    if (P.lpt_order) {
        // CTA i: KV head i mod Hkv of the slot of rank i / Hkv, longest first
        const int lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
        const int q = P.lpt_order[lin / P.Hkv];
        hk = lin % P.Hkv;
        if (q < 0) {
            have_work = false;
        } else {
            b = q / P.num_splits;
            split = q % P.num_splits;
        }
    }
    const int L = P.seq_lens[b];
    const bool seq_ok = !(L < P.M || L > P.max_seq_len || (L + PS - 1) / PS > P.mpps);
    bool run = seq_ok && have_work;                         // uniform over the CTA
    if (!seq_ok && !P.lpt_order && threadIdx.x == 0 && split == 0 && blockIdx.y == 0) flag(FP8KV_DEV_BAD_SEQ_LEN);
    // keys visible to any row of the tile: from the first row's window start
    // to the last row's position (row r is query m = r / G at L - M + m)
    const int hi0 = L - P.M + (R0 + RL - 1) / P.G;
    const int lo0 = (P.window_left >= 0) ? max(0, L - P.M + R0 / P.G - P.window_left) : 0;
    const int first_page = lo0 / PS, last_page = hi0 / PS;
    const int nsplit_b = (last_page - first_page + P.split_pages) / P.split_pages;
    if (run && nsplit_b > P.num_splits) {
        if (threadIdx.x == 0 && split == 0) flag(FP8KV_DEV_BAD_SEQ_LEN);
        run = false;
    }
    if (split >= nsplit_b) run = false;
    // cluster combine: S slots per partition (even), and the bytes this CTA
    // receives, S rows + S (max, sum) pairs from each partition (both are
    // recomputed where they are used, rather than held through the tile loop)
    auto cl_slots_of = [&]() { return ((RL + P.cluster - 1) / P.cluster + 1) & ~1; };
    auto cl_combine_of = [&]() { return P.cluster > 1 && seq_ok && nsplit_b > 1 && nsplit_b <= P.num_splits; };
    if (cl_combine_of() && threadIdx.x == 0) mbar_expect_tx(bar(B_RECV), nsplit_b * cl_slots_of() * (256 + 8));
    const int page_begin = first_page + split * P.split_pages;
    const int n_pages = min(P.split_pages, last_page + 1 - page_begin);
    constexpr int PPT = NK / PS;                            // pages per tile
    const int n_tiles = (n_pages + PPT - 1) / PPT;
    const int k_begin = page_begin * PS;
    // append: new tokens at positions [L - M, L) that fall in this partition
    const int app_lo = max(L - P.M, k_begin), app_hi = min(L, k_begin + n_pages * PS);
    // (the two-issuer form serves only calls without appended tokens)
    const bool appends = !DUAL && P.k_new != nullptr && run && app_lo < app_hi;
    // Appended tokens are written to the cache in global memory and, so that
    // no load has to wait for that write, also patched into the staged copy of
    // the tile that holds them (which may have been loaded with the old bytes):
    // tiles app_t0 .. app_t1 of this partition.
    const int app_t0 = appends ? (app_lo - k_begin) / NK : 1 << 30;
    const int app_t1 = appends ? (app_hi - 1 - k_begin) / NK : -1;
    bool ok = true;

    if (!run) {
        // no keys of this sequence fall in this partition (or bad input)
    } else if (warp == 0) {
        // ---------------------------------------------------------- producer
        const uint64_t policy = policy_evict_first();
        const int32_t* bt = P.block_table + (int64_t)b * P.mpps + page_begin;
        int issued_tiles = 0;
        // page ids 32 at a time (whole tiles: PPT divides 32), the next batch
        // loaded while this one is issued; the boxes of a tile (K and V of its
        // PPT pages) go out in one instruction, lane i issuing box i -- one
        // lane issuing them in turn caps the staging rate well below HBM's
        int next = (lane < n_pages) ? bt[lane] : 0;
        for (int base = 0; base < n_pages && ok; base += 32) {
            const int mine = next;
            if (base + 32 < n_pages) next = (base + 32 + lane < n_pages) ? bt[base + 32 + lane] : 0;
            const int cnt = min(32, n_pages - base);
            for (int j0 = 0; j0 < cnt; j0 += PPT) {
                const int t = (base + j0) / PPT, s = t % STAGES, use = t / STAGES;
                const int pages_here = min(PPT, n_pages - t * PPT);
                if (lane == 0) {
                    if (use > 0) ok = mbar_wait(bar(B_STG_EMPTY + s), (use - 1) & 1);
                    if (ok) mbar_expect_tx(bar(B_STG_FULL + s), pages_here * PS * 128 * 2);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                const int pin = lane % PPT;                 // lanes 0..PPT-1: K boxes, PPT..2PPT-1: V boxes
                const int phys = __shfl_sync(0xffffffffu, mine, j0 + pin);
                if (lane < 2 * PPT && pin < pages_here) {
                    const uint32_t dk = smem_u32(stg + s * STG_BYTES + pin * PS * 128);
                    if (lane < PPT)
                        tma_load_3d(dk, &tm_k, 0, hk * PS, phys, bar(B_STG_FULL + s), policy);
                    else
                        tma_load_3d(dk + STG_K, &tm_v, 0, hk * PS, phys, bar(B_STG_FULL + s), policy);
                }
                __syncwarp();
                issued_tiles = t + 1;
            }
        }
        if (lane == 0) {   // never leave with copies into this CTA's shared memory in flight
            for (int t = max(0, issued_tiles - STAGES); t < issued_tiles; ++t)
                mbar_wait(bar(B_STG_FULL + t % STAGES), (t / STAGES) & 1);
        }
    } else if (warp == 1 || (DUAL && warp == 15)) {
        // ------------------------------------------------------ MMA issue
        constexpr uint32_t ID_QK = idesc(128, NK, false);         // kind::f8f6f4, E4M3 x E4M3
        constexpr uint32_t ID_PV = idesc(128, 128, true);         // kind::f16, V MN-major
        // S(t) = q'.K(t) into buffer t & 1
        auto qk = [&](int t) -> bool {
            const int s = t % STAGES, sb = t & 1;
            if (!mbar_wait(bar(B_STG_FULL + s), (t / STAGES) & 1)) return false;
            // DUAL: the buffer holds P(t - 2) until its P.V has read it (one
            // issuing thread orders that by issue order)
            if (DUAL && t >= 2 && !mbar_wait(bar(B_S_EMPTY + sb), ((t >> 1) - 1) & 1)) return false;
            if (t >= app_t0 && t <= app_t1 && !mbar_wait(bar(B_PATCH + (t - app_t0)), 0)) return false;
            fence_after();
            const uint32_t kt = smem_u32(stg + s * STG_BYTES);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t bd = sdesc(kt + ks * 32, 16, 1024);
                mma_f8_ts(tmem + TM_S + sb * 128, tmem + TM_QH + 8 * ks, bd, ID_QK, ks > 0);
                mma_f8_ts(tmem + TM_S + sb * 128, tmem + TM_QL + 8 * ks, bd, ID_QK, 1);
            }
            mma_commit(bar(B_S_FULL + sb));
            mma_commit(bar(B_STG_EMPTY + s));                // K of this stage read
            return true;
        };
        // O += P(u).V(u)
        auto pv = [&](int u) -> bool {
            const int ub = u & 1, vb = u % VBUFS;
            if (!mbar_wait(bar(B_P_FULL + ub), (u >> 1) & 1)) return false;
            if (!mbar_wait(bar(B_V_FULL + vb), (u / VBUFS) & 1)) return false;
            fence_after();
            const uint32_t vf = smem_u32(vbuf + vb * VBUF_BYTES);
#pragma unroll
            for (int kk = 0; kk < NK / 16; ++kk) {
                const uint64_t bd = sdesc(vf + kk * 2048, NK * 128, 1024);
                mma_f16_ts(tmem + TM_O, tmem + TM_S + ub * 128 + 8 * kk, bd, ID_PV, (u > 0 || kk > 0));
            }
            mma_commit(bar(B_O_DONE));
            mma_commit(bar(B_V_EMPTY + vb));
            if (DUAL) mma_commit(bar(B_S_EMPTY + ub));
            if (u == n_tiles - 1) mma_commit(bar(B_O_FINAL));
            return true;
        };
        if (lane == 0) {
            if (warp == 1) {
                ok = mbar_wait(bar(B_Q_READY), 0);
                fence_after();
            }
            if (!DUAL) {
                // Q.K^T(t) then P.V(t - 1): Q.K^T of the next tile overlaps
                // the softmax of this one
                for (int t = 0; t <= n_tiles && ok; ++t) {
                    if (t < n_tiles) ok = qk(t);
                    if (ok && t >= 1) ok = pv(t - 1);
                }
            } else if (warp == 1) {
                for (int t = 0; t < n_tiles && ok; ++t) ok = qk(t);
            } else {
                for (int u = 0; u < n_tiles && ok; ++u) ok = pv(u);
            }
            // nothing the tensor cores still run may outlive the TMEM allocation
            mma_commit(bar(B_MMA_IDLE));
            mbar_wait(bar(B_MMA_IDLE), 0);
        }
        __syncwarp();
    } else if (is_converter<DUAL>(warp)) {
        // ---------------------------------------------------------- V widening
        // 128 keys x 8 chunks of 16 E4M3 values -> two 64-dim blocks of
        // 128 x 128 B f16 (128B-swizzled): the MN-major B operand of P.V.
        // Keys outside every row's range are written as zeros, so stale or NaN
        // bytes there cannot reach the output.
        const int ct = converter_index(warp) * 32 + lane;
        const int n_app = appends ? app_hi - app_lo : 0;
        const float ksc = appends ? P.k_scale[P.scale_stride * hk] : 1.f;
        const float vsc = appends ? P.v_scale[P.scale_stride * hk] : 1.f;
        // the append item `it`: one 8-element chunk of K and of V of a new token
        auto app_item = [&](int it, uint2& kc, uint2& vc, int& pos, int& chunk) {
            pos = app_lo + (it >> 4);
            chunk = it & 15;
            const int m = pos - (L - P.M);
            const int64_t src = (((int64_t)b * P.M + m) * P.Hkv + hk) * 16 + chunk;
            const bool have = spec && it == ct && app_lo == L - P.M;   // loaded before the length
            kc = e4m3_encode8(have ? spec_k : ((const uint4*)P.k_new)[src], ksc);
            vc = e4m3_encode8(have ? spec_v : ((const uint4*)P.v_new)[src], vsc);
        };
        // ----------------------------------------------------- append codes
        // this thread's first item of the new tokens in the cache-insert
        // encoding: the staged tile that holds it is patched with these codes
        // in the loop below, and the cache is written after that loop (the
        // block-table read for the token's page stays off the path to the
        // first Q.K^T; it is issued here and used there)
        uint2 kc0 = make_uint2(0, 0), vc0 = make_uint2(0, 0);
        int pos0 = -1, chunk0 = 0, page0 = -1;
        if (ct < n_app * 16) {
            app_item(ct, kc0, vc0, pos0, chunk0);
            page0 = P.block_table[(int64_t)b * P.mpps + pos0 / PS];
        }
        for (int t = 0; t < n_tiles; ++t) {
            const int s = t % STAGES, vb = t % VBUFS;
            ok = mbar_wait(bar(B_STG_FULL + s), (t / STAGES) & 1);
            if (ok && t >= VBUFS) ok = mbar_wait(bar(B_V_EMPTY + vb), ((t / VBUFS) - 1) & 1);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            const int k0 = k_begin + t * NK;
            const bool patched = t >= app_t0 && t <= app_t1;
            if (patched) {
                // this tile's new rows of K (128-byte swizzled rows of the
                // staging buffer) get the appended tokens' codes, for the
                // Q.K^T of this tile; their V goes straight into the f16 tile
                // below, so the widening waits for no other warp
                uint8_t* kst = stg + s * STG_BYTES;
                for (int it = ct; it < n_app * 16; it += CONV_THREADS) {
                    uint2 kc = kc0, vc = vc0;
                    int pos = pos0, chunk = chunk0;
                    if (it != ct) app_item(it, kc, vc, pos, chunk);
                    const int r = pos - k0;
                    if (r < 0 || r >= NK) continue;
                    *(uint2*)(kst + r * 128 + ((((chunk >> 1) ^ r) & 7) << 4) + (chunk & 1) * 8) = kc;
                }
                fence_proxy_async();                        // for the tensor cores' read of K
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_PATCH + (t - app_t0)));
            }
            // rows [nlo, nhi) of this tile hold appended tokens: the staged V
            // bytes there may be old, so the widening below skips them
            const int nlo = patched ? max(0, app_lo - k0) : 0;
            const int nhi = patched ? min(NK, app_hi - k0) : 0;
            const int pages_here = min(PPT, n_pages - t * PPT);
            const int zlo = max(0, min(NK, lo0 - k0));
            const int zhi = max(0, min(min(NK, pages_here * PS), hi0 + 1 - k0));
            const uint8_t* src = stg + s * STG_BYTES + STG_K;
            uint8_t* dst = vbuf + vb * VBUF_BYTES;
            constexpr int PER = (NK * 8 + CONV_THREADS - 1) / CONV_THREADS;   // chunks per thread
            uint4 code[PER];
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const int i = ct + CONV_THREADS * u;
                const int r = i >> 3, c = i & 7;
                code[u] = (i < NK * 8 && r >= zlo && r < zhi)
                              ? *(const uint4*)(src + r * 128 + (((c ^ r) & 7) << 4))
                              : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const int i = ct + CONV_THREADS * u;
                if (i >= NK * 8) break;
                const int r = i >> 3, c = i & 7;
                if (!DUAL && r >= nlo && r < nhi) continue;
                uint4 lo, hi;
                lo.x = e4m3x2_to_f16x2(code[u].x);
                lo.y = e4m3x2_to_f16x2(code[u].x >> 16);
                lo.z = e4m3x2_to_f16x2(code[u].y);
                lo.w = e4m3x2_to_f16x2(code[u].y >> 16);
                hi.x = e4m3x2_to_f16x2(code[u].z);
                hi.y = e4m3x2_to_f16x2(code[u].z >> 16);
                hi.z = e4m3x2_to_f16x2(code[u].w);
                hi.w = e4m3x2_to_f16x2(code[u].w >> 16);
                uint8_t* blk = dst + (c >> 2) * (NK * 128) + r * 128;
                const int c16 = 2 * (c & 3);
                // alternate the order so each quarter-warp covers all 32 banks
                if (c < 4) {
                    *(uint4*)(blk + (((c16 ^ r) & 7) << 4)) = lo;
                    *(uint4*)(blk + ((((c16 + 1) ^ r) & 7) << 4)) = hi;
                } else {
                    *(uint4*)(blk + ((((c16 + 1) ^ r) & 7) << 4)) = hi;
                    *(uint4*)(blk + (((c16 ^ r) & 7) << 4)) = lo;
                }
            }
            if (patched) {
                // the appended tokens' V, widened from their codes: 8 values
                // (half of a 16-byte f16 unit pair) per item
                for (int it = ct; it < n_app * 16; it += CONV_THREADS) {
                    uint2 kc = kc0, vc = vc0;
                    int pos = pos0, chunk = chunk0;
                    if (it != ct) app_item(it, kc, vc, pos, chunk);
                    const int r = pos - k0;
                    if (r < 0 || r >= NK) continue;
                    const int c = chunk >> 1;
                    uint4 h;
                    h.x = e4m3x2_to_f16x2(vc.x);
                    h.y = e4m3x2_to_f16x2(vc.x >> 16);
                    h.z = e4m3x2_to_f16x2(vc.y);
                    h.w = e4m3x2_to_f16x2(vc.y >> 16);
                    *(uint4*)(dst + (c >> 2) * (NK * 128) + r * 128 + ((((2 * (c & 3) + (chunk & 1)) ^ r) & 7) << 4)) = h;
                }
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(B_STG_EMPTY + s));
                mbar_arrive(bar(B_V_FULL + vb));
            }
        }
        // ---------------------------------------------------- append insert
        // the new tokens of this head into the cache
        for (int it = ct; it < n_app * 16; it += CONV_THREADS) {
            uint2 kc = kc0, vc = vc0;
            int pos = pos0, chunk = chunk0, page = page0;
            if (it != ct) {
                app_item(it, kc, vc, pos, chunk);
                page = P.block_table[(int64_t)b * P.mpps + pos / PS];
            }
            if (page < 0 || page >= P.num_pages) {
                if (chunk == 0) flag(FP8KV_DEV_BAD_SLOT);
                continue;
            }
            const int64_t dst = (((int64_t)page * P.Hkv + hk) * PS + pos % PS) * 128 + chunk * 8;
            *(uint2*)(P.k_cache + dst) = kc;
            *(uint2*)(P.v_cache + dst) = vc;
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int wq = warp & 3, half = (warp - 4) >> 2;
        const int r = wq * 32 + lane;
        const bool active = wq * 32 < RL;                   // quarter holds at least one real row
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        const int rr = R0 + min(r, RL - 1);                 // the row of the (b, hk) block
        const int m = rr / P.G;
        const int p_r = L - P.M + m;
        const int lo_r = (P.window_left >= 0) ? max(0, p_r - P.window_left) : 0;
        const int64_t row_idx = ((int64_t)b * P.M + m) * P.Hq + hk * P.G + rr % P.G;
        const float vs = P.v_scale[P.scale_stride * hk];
        // rows past M*G get Q = 0: their (unused) weights stay finite and their
        // lanes take the same unmasked path as the real rows
        const bool pad = r >= RL;
        float mult;
        {
            // Q row split in place: q' = q * 2^sh with the row maximum |q'| in
            // [128, 256) (from all 128 dims), Q_hi = e4m3(q'), Q_lo =
            // e4m3(q' - Q_hi); this half stores dims 64*half .. +63 of both
            // into tensor memory (the A operand of Q.K^T).  q' is exact in f16
            // (8 significant bits, at most 256) and so is q' - Q_hi.
            const uint4* src = (const uint4*)(P.q + row_idx * 128) + 8 * half;
            uint32_t qh[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint4 w = pad ? make_uint4(0, 0, 0, 0) : src[u];
                qh[4 * u] = w.x;
                qh[4 * u + 1] = w.y;
                qh[4 * u + 2] = w.z;
                qh[4 * u + 3] = w.w;
            }
            // row maximum: this half's 64 dims, then the partner warp's through
            // shared memory (named barrier of the quarter's two warps)
            uint32_t am = 0;
#pragma unroll
            for (int u = 0; u < 32; ++u) am = max_bf16x2(am, qh[u] & 0x7fff7fffu);
            float amax = fmaxf(bf16_lo(am), bf16_hi(am));
            xch[half * 128 + r] = amax;
            asm volatile("bar.sync %0, 64;" ::"r"(1 + wq) : "memory");
            amax = fmaxf(xch[r], xch[128 + r]);
            asm volatile("bar.sync %0, 64;" ::"r"(1 + wq) : "memory");   // xch free for the tile loop
            int e = 7;
            const uint32_t ab = __float_as_uint(amax);
            if (amax > 0.f && ((ab >> 23) & 0xff) != 0xff) {
                const int be = (int)((ab >> 23) & 0xff);
                e = be ? be - 127 : -127;
            }
            const int sh = max(-100, min(100, 7 - e));
            const float scale = ldexpf(1.0f, sh);
            mult = P.k_scale[P.scale_stride * hk] * P.sm_scale * 1.4426950408889634f * ldexpf(1.0f, -sh);
            uint32_t hw[16], lw[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                uint32_t h2[2], l2[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const uint32_t x = qh[2 * k + i];
                    const uint32_t q16 = pack_f16x2(bf16_lo(x) * scale, bf16_hi(x) * scale);
                    h2[i] = f16x2_to_e4m3x2(q16);
                    l2[i] = f16x2_to_e4m3x2(sub_f16x2(q16, e4m3x2_to_f16x2(h2[i])));
                }
                hw[k] = h2[0] | (h2[1] << 16);
                lw[k] = l2[0] | (l2[1] << 16);
            }
            tmem_st_x16(lane_base + TM_QH + 16 * half, hw);
            tmem_st_x16(lane_base + TM_QL + 16 * half, lw);
            tmem_wait_st();
        }
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_Q_READY));

        int pmin = p_r, lomax = lo_r, pmax = p_r, lomin = lo_r;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            pmin = min(pmin, __shfl_xor_sync(0xffffffffu, pmin, off));
            lomax = max(lomax, __shfl_xor_sync(0xffffffffu, lomax, off));
            pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, off));
            lomin = min(lomin, __shfl_xor_sync(0xffffffffu, lomin, off));
        }
        float m_run = -INFINITY, l_run = 0.f;               // l_run: this half's columns only
        for (int t = 0; t < n_tiles; ++t) {
            const int sb = t & 1;
            ok = mbar_wait(bar(B_S_FULL + sb), (t >> 1) & 1);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            fence_after();
            if (active) {
                const uint32_t scol = lane_base + TM_S + sb * 128 + 64 * half;
                const int k0 = k_begin + t * NK + 64 * half;   // first key of this half
                // no row of this warp sees any key of the half (the end of
                // the last tile, the start of a window): its P is zero
                const bool dead = !DUAL && ((k0 > pmax) || (k0 + 63 < lomin));
                uint32_t sv[64];
                float hmax = -INFINITY;
                if (!dead) {
                    tmem_ld_x64(scol, sv);
                    tmem_wait_ld();
                    if (DUAL && ((k0 + 63 > pmin) || (k0 < lomax))) {
#pragma unroll
                        for (int j = 0; j < 64; ++j)
                            if (k0 + j > p_r || k0 + j < lo_r) sv[j] = 0xff800000u;   // -inf
                    } else if ((k0 + 63 > pmin) || (k0 < lomax)) {
                        // this row's visible columns of the half, [jlo, jhi), as
                        // a bit mask: one bit test and select per column
                        const int jlo = max(0, lo_r - k0), jhi = min(64, p_r - k0 + 1);
                        const uint64_t below_hi = jhi <= 0 ? 0ull : (jhi >= 64 ? ~0ull : (1ull << jhi) - 1);
                        const uint64_t below_lo = jlo >= 64 ? ~0ull : (1ull << jlo) - 1;
                        const uint64_t vis = below_hi & ~below_lo;
                        const uint32_t vis_lo = (uint32_t)vis, vis_hi = (uint32_t)(vis >> 32);
#pragma unroll
                        for (int j = 0; j < 64; ++j)
                            sv[j] = (((j < 32 ? vis_lo : vis_hi) >> (j & 31)) & 1u) ? sv[j] : 0xff800000u;   // -inf
                    }
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int j = 0; j < 64; j += 4) {
                        m4[0] = fmaxf(m4[0], __uint_as_float(sv[j]));
                        m4[1] = fmaxf(m4[1], __uint_as_float(sv[j + 1]));
                        m4[2] = fmaxf(m4[2], __uint_as_float(sv[j + 2]));
                        m4[3] = fmaxf(m4[3], __uint_as_float(sv[j + 3]));
                    }
                    hmax = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                }
                xch[(sb * 2 + half) * 128 + r] = hmax;
                // exchange with the partner warp (bounded wait, phase t of the pair barrier)
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_PAIR + wq));
                ok = mbar_wait(bar(B_PAIR + wq), t & 1);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                const float smax = fmaxf(xch[sb * 256 + r], xch[sb * 256 + 128 + r]);
                const float tmax = smax * mult;
                const bool rescale = (m_run != -INFINITY) && (tmax > m_run + 8.0f);
                if (__any_sync(0xffffffffu, rescale)) {
                    // O holds P.V up to tile t-1: wait for it, then rescale this half
                    const bool okw = mbar_wait(bar(B_O_DONE), (t - 1) & 1);
                    if (!__all_sync(0xffffffffu, okw)) { ok = false; break; }
                    fence_after();
                    const float alpha = rescale ? ex2(m_run - tmax) : 1.0f;
#pragma unroll 1
                    for (int c = 0; c < 64; c += 32) {
                        uint32_t ov[32];
                        tmem_ld_x32(lane_base + TM_O + 64 * half + c, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
                        tmem_st_x32(lane_base + TM_O + 64 * half + c, ov);
                    }
                    tmem_wait_st();
                    if (rescale) {
                        l_run *= alpha;
                        m_run = tmax;
                    }
                }
                if (m_run == -INFINITY) m_run = tmax;
                const float neg = (m_run == -INFINITY) ? 0.f : -m_run;
                // P = 2^(s*mult - m) as f16 (masked keys are -inf and give 0);
                // both halves' S reads are complete (pair barrier above)
                float sum0 = 0.f, sum1 = 0.f;
                uint32_t pw[32];
                if (!dead) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float p0 = ex2(fmaf(__uint_as_float(sv[2 * j]), mult, neg));
                        const float p1 = ex2(fmaf(__uint_as_float(sv[2 * j + 1]), mult, neg));
                        sum0 += p0;
                        sum1 += p1;
                        pw[j] = pack_f16x2(p0, p1);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) pw[j] = 0u;
                }
                tmem_st_x32(lane_base + TM_S + sb * 128 + 32 * half, pw);
                l_run += sum0 + sum1;
                tmem_wait_st();
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_P_FULL + sb));
        }
        // ------------------------------------------------------------ epilogue
        if (ok) ok = mbar_wait(bar(B_O_FINAL), 0);
        ok = __all_sync(0xffffffffu, ok);
        if (ok && active) {
            fence_after();
            // row sums of both halves: phase n_tiles of the pair barrier
            xch[(4 + half) * 128 + r] = l_run;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PAIR + wq));
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B_PAIR + wq), n_tiles & 1));
        }
        if (ok && active) {
            const float l_tot = xch[4 * 128 + r] + xch[5 * 128 + r];
            const bool direct = nsplit_b == 1;
            const bool combine = !direct && P.cluster > 1;  // partial stays in shared memory
            const int cl_slots = cl_slots_of();
            // the partition index, read again here rather than held through
            // the tile loop
            const int split_e =
                P.lpt_order ? P.lpt_order[(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z)) / P.Hkv] %
                                  P.num_splits
                            : (int)blockIdx.x;
            // direct: bf16 of O * v_scale / l; partial (cluster or workspace):
            // f16 of O / l in code units (|x| <= 448, 11-bit mantissa) beside
            // its (max, sum), half the bytes of an fp32 partial
            // (a row with no visible key in this partition has l = 0: weight 0, values 0)
            const float f = direct ? vs / l_tot : (l_tot > 0.f ? 1.0f / l_tot : 0.f);
            // This thread's half row (64 dims: bf16 output or fp32 partial)
            // goes through the free staging buffers to one bulk copy: stores
            // straight from the row-per-thread TMEM layout would touch a
            // different row, hence cache line, in every lane.
            uint8_t* row_stage = stg + (half * 128 + r) * EPI_STRIDE;
#pragma unroll 1
            for (int c = 0; c < 64; c += 32) {
                uint32_t ov[32];
                tmem_ld_x32(lane_base + TM_O + 64 * half + c, ov);
                tmem_wait_ld();
                if (direct) {
                    uint4* dst = (uint4*)(row_stage + c * 2);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        dst[v4] = make_uint4(
                            pack_bf16x2(__uint_as_float(ov[8 * v4 + 0]) * f, __uint_as_float(ov[8 * v4 + 1]) * f),
                            pack_bf16x2(__uint_as_float(ov[8 * v4 + 2]) * f, __uint_as_float(ov[8 * v4 + 3]) * f),
                            pack_bf16x2(__uint_as_float(ov[8 * v4 + 4]) * f, __uint_as_float(ov[8 * v4 + 5]) * f),
                            pack_bf16x2(__uint_as_float(ov[8 * v4 + 6]) * f, __uint_as_float(ov[8 * v4 + 7]) * f));
                } else {
                    uint4 w[4];
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        w[v4] = make_uint4(
                            pack_f16x2(__uint_as_float(ov[8 * v4 + 0]) * f, __uint_as_float(ov[8 * v4 + 1]) * f),
                            pack_f16x2(__uint_as_float(ov[8 * v4 + 2]) * f, __uint_as_float(ov[8 * v4 + 3]) * f),
                            pack_f16x2(__uint_as_float(ov[8 * v4 + 4]) * f, __uint_as_float(ov[8 * v4 + 5]) * f),
                            pack_f16x2(__uint_as_float(ov[8 * v4 + 6]) * f, __uint_as_float(ov[8 * v4 + 7]) * f));
                    if (combine) {
                        // staged by owner (rank r mod C), slot r / C: one
                        // contiguous block per owner, sent below; 16-byte
                        // chunk j of row r at chunk j ^ (r & 7), so that a
                        // warp's 32 rows spread over all banks
                        if (r < RL) {
                            uint8_t* row = stg + ((r % P.cluster) * cl_slots + r / P.cluster) * 256;
#pragma unroll
                            for (int v4 = 0; v4 < 4; ++v4)
                                *(uint4*)(row + (((half * 8 + c / 8 + v4) ^ (r & 7)) << 4)) = w[v4];
                        }
                    } else {
                        uint4* dst = (uint4*)(row_stage + c * 2);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) dst[v4] = w[v4];
                    }
                }
            }
            if (r < RL && !combine) {
                fence_proxy_async();        // the staged row, written by this thread, to the bulk copy
                if (direct)
                    bulk_store(P.out + row_idx * 128 + 64 * half, smem_u32(row_stage), 128);
                else
                    bulk_store((uint16_t*)P.ws_o + (row_idx * P.num_splits + split_e) * 128 + 64 * half,
                               smem_u32(row_stage), 128);
                bulk_commit();
                bulk_wait_read();
            }
            if (r < RL && !direct && half == 0) {
                if (combine) {
                    float* cml = (float*)(stg + P.cluster * cl_slots * 256);
                    *(float2*)(cml + ((r % P.cluster) * cl_slots + r / P.cluster) * 2) = make_float2(m_run, l_tot);
                } else {
                    P.ws_ml[(row_idx * P.num_splits + split_e) * 2] = m_run;
                    P.ws_ml[(row_idx * P.num_splits + split_e) * 2 + 1] = l_tot;
                }
            }
        }
        if (cl_combine_of()) {
            const int cl_slots = cl_slots_of();
            // every softmax warp's staged rows, then one thread sends each
            // owner its block of rows and its block of (max, sum), both
            // completing on the owner's receive barrier
            fence_proxy_async();
            if (softmax_warps_all(ok) && warp == 4 && lane == 0) {
                const float* cml = (const float*)(stg + P.cluster * cl_slots * 256);
                for (int j = 0; j < P.cluster; ++j) {
                    const uint32_t rb = dsmem_addr(&bars[B_RECV], j);
                    bulk_copy_to_cluster(dsmem_addr(recv + split * cl_slots * 256, j),
                                         smem_u32(stg + j * cl_slots * 256), cl_slots * 256, rb);
                    bulk_copy_to_cluster(dsmem_addr(recv_ml + split * cl_slots * 2, j),
                                         smem_u32(cml + j * cl_slots * 2), cl_slots * 8, rb);
                }
            }
        }
    }

    if (P.cluster > 1) {
        // ------------------------------------------------- cluster combine
        // The partitions of this (KV head, sequence) are the CTAs of one
        // cluster (rank = partition).  Each has staged its partial rows by
        // owner (row r belongs to rank r mod C) and sent every owner its
        // block with bulk copies that complete on the owner's receive
        // barrier.  Once that barrier completes, a CTA combines the rows it
        // owns from its own shared memory, 16 threads a row, each with 8
        // dims, every thread reading all the partitions' (max, sum) itself:
        // O = v_scale * sum_p w_p O_p / sum_p w_p, w_p = 2^(m_p - m*) l_p.
        // A split cluster barrier (arrive once this CTA has received, wait
        // before exit) keeps each sender's staged blocks in place until
        // every owner has them.
        bool recv_ok = true;
        const bool cl_combine = cl_combine_of();
        const int cl_slots = cl_slots_of();
        if (cl_combine) recv_ok = mbar_wait(bar(B_RECV), 0);
        __syncwarp();
        cluster_arrive_relaxed();
        if (cl_combine && recv_ok) {
            const float vsc = P.v_scale[P.scale_stride * hk];
            const int C = P.cluster, slots = cl_slots;
            for (int i = threadIdx.x; i < slots * 16; i += THREADS) {
                const int k = i >> 4, ch = i & 15;
                const int r = split + C * k;
                if (r >= RL) break;                         // r grows with i
                float mp[8], lp[8];
                float mstar = -INFINITY;
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    mp[p] = -INFINITY;
                    lp[p] = 0.f;
                    if (p < nsplit_b) {
                        const float2 ml = *(const float2*)(recv_ml + (p * slots + k) * 2);
                        mp[p] = ml.x;
                        lp[p] = ml.y;
                        mstar = fmaxf(mstar, ml.x);
                    }
                }
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                float lsum = 0.f;
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    if (p < nsplit_b) {
                        const float w = (mp[p] == -INFINITY) ? 0.f : ex2(mp[p] - mstar) * lp[p];
                        lsum += w;
                        const uint4 o = *(const uint4*)(recv + (p * slots + k) * 256 + ((ch ^ (r & 7)) << 4));
                        const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float2 f2 = f16x2_to_f32x2(ow[j]);
                            acc[2 * j] = fmaf(w, f2.x, acc[2 * j]);
                            acc[2 * j + 1] = fmaf(w, f2.y, acc[2 * j + 1]);
                        }
                    }
                }
                const float inv = vsc / lsum;
                const int m = (R0 + r) / P.G;
                const int64_t orow = ((int64_t)b * P.M + m) * P.Hq + hk * P.G + (R0 + r) % P.G;
                *(uint4*)(P.out + orow * 128 + 8 * ch) =
                    make_uint4(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv),
                               pack_bf16x2(acc[4] * inv, acc[5] * inv), pack_bf16x2(acc[6] * inv, acc[7] * inv));
            }
        }
        __syncwarp();
        cluster_wait();
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

int tc_tile_tokens() { return tc::NK; }
int tc_threads() { return tc::THREADS; }

int launch_attention_tc(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& P, cudaStream_t s) {
    const int RT = (P.R + 127) / 128;
    if (P.R <= 16 || (int64_t)RT * P.Hkv > 65535) return FP8KV_ERR_UNSUPPORTED;
    if (RT > 1 && (P.cluster > 1 || P.k_new)) return FP8KV_ERR_UNSUPPORTED;   // single row tile only
    if ((P.split_pages * P.page_size) % tc::NK) return FP8KV_ERR_UNSUPPORTED;
    static std::mutex mu;
    static std::set<std::pair<int, const void*>> done;
    // two issuing threads when no new tokens are appended in the kernel (the
    // append encodes them in the converter warps, which then need all six)
    const bool dual = P.k_new == nullptr;
    const void* kern = P.page_size == 32 ? (dual ? (const void*)tc::attention_tc_kernel<32, true>
                                                 : (const void*)tc::attention_tc_kernel<32, false>)
                                         : (dual ? (const void*)tc::attention_tc_kernel<64, true>
                                                 : (const void*)tc::attention_tc_kernel<64, false>);
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
    cudaError_t e;
    dim3 grid(P.num_splits, P.Hkv * RT, P.B);
    if (P.cluster > 1 && (P.cluster > 8 || P.cluster != P.num_splits)) return FP8KV_ERR_UNSUPPORTED;
    if (P.lpt_order && (RT > 1 || P.cluster > 1 || (int64_t)P.B * P.num_splits * P.Hkv > INT32_MAX))
        return FP8KV_ERR_UNSUPPORTED;
    auto k = P.page_size == 32 ? (dual ? tc::attention_tc_kernel<32, true> : tc::attention_tc_kernel<32, false>)
                               : (dual ? tc::attention_tc_kernel<64, true> : tc::attention_tc_kernel<64, false>);
    e = launch_pdl_cluster(k, grid, dim3(tc::THREADS), tc::SMEM, s, P.cluster, tk, tv, P);
    return e == cudaSuccess ? FP8KV_OK : (cudaGetLastError(), FP8KV_ERR_CUDA);
}

}  // namespace fp8kv
