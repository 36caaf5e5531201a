// attention_layers.cu -- the verifier step of several layers in one
// persistent launch: the append of each layer's new tokens and its exact
// paged attention over the E4M3 cache, layer after layer, without a kernel
// boundary between layers ("Laguna S 2.1 B70 campaign transfer ledger",
// table "Result progression", rows on graph coverage and persistent
// attention metadata, and section "Graph and topology lessons": the launches
// and metadata work around each attention call set the cycle time; "Laguna S
// 2.1 INT4 -- calibrated FP8 KV on Intel B70", section "Contract": the
// width-12 verifier).
//
// One CTA per SM for the whole step (a cooperative launch, so that every CTA
// is resident and the waits below always end).  Each layer is cut into work
// units (sequence, KV head, key partition of whole 128-key tiles), units u,
// u + grid, u + 2 grid, ... of a layer going to CTA u in that order.  A unit runs the pipeline of the single-layer
// tensor-memory kernel (attention_tc.cu): a TMA producer warp, one MMA
// thread, six V-widening warps, eight softmax warps, with the same Q split,
// masks, online softmax and tile layout.  What differs:
//   * the pipelines run on across units and layers: stage, buffer and barrier
//     phases follow a per-CTA tile count, the tensor memory is allocated once,
//     and the producer runs ahead into the next layer's pages (the cache of
//     the earlier context exists before the step) while the current layer
//     finishes;
//   * layer order is kept: the data a layer's work depends on -- its queries
//     and new tokens, which the previous layer's output would produce in a
//     model -- is read only after every unit of the previous layer has
//     written its output (a counter per layer in the workspace);
//   * partitions of a (sequence, KV head) combine through the workspace:
//     each writes its normalised partial (f16, in E4M3 code units) and its
//     (max, sum); once a counter shows every partition of the group written,
//     each partition's CTA combines a share of the group's rows -- after all
//     of its own units of the layer, so that no CTA waits for a group while
//     holding back a unit another CTA waits for;
//   * appended tokens are written to the cache and patched into the staged
//     tile that holds them, as in the single-layer kernel.
// Every wait is bounded (mbarriers and the global counters: 2 s, then
// FP8KV_DEV_WAIT_TIMEOUT).  The workspace counters must be zero before the
// first call; the last CTA to finish sets them back to zero.
#include <cudaTypedefs.h>
#include <stdio.h>

#include <algorithm>
#include <mutex>
#include <set>
#include <utility>

#include "attention.cuh"
#include "common.cuh"
#include "tcgen05.cuh"

namespace fp8kv {

int status_attention_layers(unsigned int* s, int clear) { return read_status(s, clear); }

namespace pl {

constexpr int NK = 128;                          // keys per tile
constexpr int STAGES = 3;                        // E4M3 staging tiles (K + V)
constexpr int STG_K = NK * 128;                  // 16 KiB
constexpr int STG_BYTES = 2 * STG_K;             // 32 KiB
constexpr int VBUFS = 2;                         // f16 V tiles
constexpr int VBUF_BYTES = NK * 256;             // 32 KiB
constexpr int EPI_STRIDE = 144;                  // one staged half row: 64 x 16 bit + pad
constexpr int EPI_BYTES = 2 * 128 * EPI_STRIDE;
constexpr int XCH_BYTES = 3 * 2 * 128 * 4;
constexpr int SMEM = STAGES * STG_BYTES + VBUFS * VBUF_BYTES + EPI_BYTES + XCH_BYTES + 1024 + 512;
constexpr uint32_t TM_QH = 0, TM_QL = 32, TM_S = 64, TM_O = 320, TM_COLS = 512;
constexpr int WARPS = 16, THREADS = WARPS * 32;
constexpr int CONV_WARPS = 6, CONV_THREADS = CONV_WARPS * 32;
constexpr int SOFT_THREADS = 256;

// Barriers of the patched tiles, used in turn: the converters can be at most
// STAGES tiles ahead of the MMA thread, so with one more barrier than stages
// a barrier cannot complete again before the MMA thread has waited on it.
constexpr int N_PATCH = STAGES + 1;

enum {
    B_STG_FULL = 0,
    B_STG_EMPTY = B_STG_FULL + STAGES,
    B_V_FULL = B_STG_EMPTY + STAGES,
    B_V_EMPTY = B_V_FULL + VBUFS,
    B_S_FULL = B_V_EMPTY + VBUFS,
    B_P_FULL = B_S_FULL + 2,
    B_O_DONE = B_P_FULL + 2,
    B_O_FINAL = B_O_DONE + 1,
    B_O_FREE = B_O_FINAL + 1,                    // the epilogue has read O: the next unit may overwrite it
    B_Q_READY = B_O_FREE + 1,
    B_MMA_IDLE = B_Q_READY + 1,
    B_PAIR = B_MMA_IDLE + 1,                     // one per TMEM lane quarter: the two softmax warps
    // new tokens patched into a staged tile: the CTA's patched tiles take
    // these barriers in turn (N_PATCH of them, above)
    B_PATCH = B_PAIR + 4,
    B_DEP = B_PATCH + N_PATCH,                   // converters: the previous layer is complete (all six warps)
    B_COUNT = B_DEP + 1
};

__device__ __forceinline__ bool is_converter(int warp) { return warp == 2 || warp == 3 || warp >= 12; }
__device__ __forceinline__ int converter_index(int warp) { return warp < 4 ? warp - 2 : warp - 10; }

// Global counters: wait until *c >= target (bounded), release-increment.
__device__ __forceinline__ unsigned ld_acquire(const unsigned* c) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(unsigned* c, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(c), "r"(v) : "memory");
}
__device__ __forceinline__ bool wait_counter(const unsigned* c, unsigned target) {
    if (ld_acquire(c) >= target) return true;
    const uint64_t start = globaltimer();
    unsigned ns = 64;
    while (true) {
        __nanosleep(ns);
        if (ns < 512) ns <<= 1;
        if (ld_acquire(c) >= target) return true;
        if (globaltimer() - start > 2000000000ull) {
            flag(FP8KV_DEV_WAIT_TIMEOUT);
            return false;
        }
    }
}

// One unit of a layer, as every role of the CTA derives it.
struct Unit {
    int b, hk, split, L;
    bool seq_ok, run;                            // run: the partition holds keys
    int lo0, hi0, nsplit_b, page_begin, n_pages, n_tiles, k_begin;
    int app_lo, app_hi, app_t0, app_t1;          // appended positions in this partition and their tiles
};

template <int PS>
__device__ __forceinline__ Unit unit_of(const LayersParams& P, const LayerDesc& D, int u, bool flag_bad) {
    Unit U;
    const int ns = D.num_splits;
    U.split = u % ns;
    const int g = u / ns;
    U.b = g / P.Hkv;
    U.hk = g % P.Hkv;
    U.L = D.seq_lens[U.b];
    const int L = U.L;
    U.seq_ok = !(L < P.M || L > D.max_seq_len || (L + PS - 1) / PS > D.mpps);
    if (!U.seq_ok && flag_bad && U.split == 0 && U.hk == 0) flag(FP8KV_DEV_BAD_SEQ_LEN);
    U.hi0 = L - P.M + (P.R - 1) / P.G;
    U.lo0 = (D.window_left >= 0) ? max(0, L - P.M - D.window_left) : 0;
    const int first_page = U.lo0 / PS, last_page = U.hi0 / PS;
    U.nsplit_b = (last_page - first_page + D.split_pages) / D.split_pages;
    bool run = U.seq_ok && U.nsplit_b <= ns;
    if (U.seq_ok && U.nsplit_b > ns && flag_bad && U.split == 0) flag(FP8KV_DEV_BAD_SEQ_LEN);
    if (U.split >= U.nsplit_b) run = false;
    U.run = run;
    U.page_begin = first_page + U.split * D.split_pages;
    U.n_pages = run ? min(D.split_pages, last_page + 1 - U.page_begin) : 0;
    U.n_tiles = (U.n_pages + NK / PS - 1) / (NK / PS);
    U.k_begin = U.page_begin * PS;
    U.app_lo = max(L - P.M, U.k_begin);
    U.app_hi = min(L, U.k_begin + U.n_pages * PS);
    const bool appends = D.k_new != nullptr && run && U.app_lo < U.app_hi;
    U.app_t0 = appends ? (U.app_lo - U.k_begin) / NK : 1 << 30;
    U.app_t1 = appends ? (U.app_hi - 1 - U.k_begin) / NK : -1;
    if (!appends) U.app_hi = U.app_lo;
    return U;
}

// Barrier of the eight softmax warps (named barrier 6) that also ANDs `ok`
// over them, so that they always leave their loop together.
__device__ __forceinline__ bool soft_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.and.pred q, 6, %2, p; selp.u32 %0, 1, 0, q; }"
        : "=r"(r)
        : "r"((uint32_t)ok), "n"(SOFT_THREADS)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ int units_of(const LayersParams& P, const LayerDesc& D) {
    return P.B * P.Hkv * D.num_splits;
}

template <int PS>
__global__ void __launch_bounds__(THREADS, 1) attention_layers_kernel(const __grid_constant__ LayersParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* stg = smem;                                    // STAGES x (K 16 KiB, V 16 KiB)
    uint8_t* vbuf = smem + STAGES * STG_BYTES;              // VBUFS x 32 KiB
    uint8_t* epi = vbuf + VBUFS * VBUF_BYTES;               // [half][row] staged output rows
    float* xch = (float*)(epi + EPI_BYTES);                 // [parity][half][row]
    uint64_t* bars = (uint64_t*)((uint8_t*)xch + XCH_BYTES);
    uint32_t* tmem_slot = (uint32_t*)(bars + B_COUNT);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int u = blockIdx.x;                               // this CTA's unit in every layer
    constexpr int PPT = NK / PS;                            // pages per tile
    unsigned* grp = P.counters;                                           // [layer][B*Hkv]
    unsigned* done = P.counters + (size_t)P.n_layers * P.B * P.Hkv;      // [layer]
    unsigned* exit_count = done + P.n_layers;

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
        mbar_init(bar(B_O_FREE), 8);
        mbar_init(bar(B_Q_READY), 8);
        mbar_init(bar(B_MMA_IDLE), 1);
        for (int k = 0; k < N_PATCH; ++k) mbar_init(bar(B_PATCH + k), CONV_WARPS);
        mbar_init(bar(B_DEP), CONV_WARPS);                 // every converter warp, the poller last
        for (int q = 0; q < 4; ++q) mbar_init(bar(B_PAIR + q), 2);
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
        // every layer's pages in order, running ahead of the other roles as
        // far as the staging ring allows
        const uint64_t policy = policy_evict_first();
        int tg = 0;                                         // this CTA's tile count
        for (int l = 0; l < P.n_layers && ok; ++l) {
            const LayerDesc& D = P.layer[l];
            if (lane == 0 && u < units_of(P, D)) {
                prefetch_tensormap(&D.tm_k);
                prefetch_tensormap(&D.tm_v);
            }
          for (int uu = u; uu < units_of(P, D) && ok; uu += gridDim.x) {
            const Unit U = unit_of<PS>(P, D, uu, false);
            if (!U.run) continue;
            const int32_t* bt = D.block_table + (int64_t)U.b * D.mpps + U.page_begin;
            int next = (lane < U.n_pages) ? bt[lane] : 0;
            for (int base = 0; base < U.n_pages && ok; base += 32) {
                const int mine = next;
                if (base + 32 < U.n_pages) next = (base + 32 + lane < U.n_pages) ? bt[base + 32 + lane] : 0;
                const int cnt = min(32, U.n_pages - base);
                for (int j0 = 0; j0 < cnt; j0 += PPT, ++tg) {
                    const int t = (base + j0) / PPT, s = tg % STAGES, use = tg / STAGES;
                    const int pages_here = min(PPT, U.n_pages - t * PPT);
                    if (lane == 0) {
                        if (use > 0) ok = mbar_wait(bar(B_STG_EMPTY + s), (use - 1) & 1);
                        if (ok) mbar_expect_tx(bar(B_STG_FULL + s), pages_here * PS * 128 * 2);
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    const int pin = lane % PPT;             // lanes 0..PPT-1: K boxes, PPT..2PPT-1: V boxes
                    const int phys = __shfl_sync(0xffffffffu, mine, j0 + pin);
                    if (lane < 2 * PPT && pin < pages_here) {
                        const uint32_t dk = smem_u32(stg + s * STG_BYTES + pin * PS * 128);
                        if (lane < PPT)
                            tma_load_3d(dk, &D.tm_k, 0, U.hk * PS, phys, bar(B_STG_FULL + s), policy);
                        else
                            tma_load_3d(dk + STG_K, &D.tm_v, 0, U.hk * PS, phys, bar(B_STG_FULL + s), policy);
                    }
                    __syncwarp();
                }
            }
          }
        }
        if (lane == 0) {   // never leave with copies into this CTA's shared memory in flight
            for (int t = max(0, tg - STAGES); t < tg; ++t) mbar_wait(bar(B_STG_FULL + t % STAGES), (t / STAGES) & 1);
        }
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_QK = idesc(128, NK, false);     // kind::f8f6f4, E4M3 x E4M3
            constexpr uint32_t ID_PV = idesc(128, 128, true);     // kind::f16, V MN-major
            int tg = 0, qi = 0, pc = 0;                             // tiles, units, patched tiles
            for (int l = 0; l < P.n_layers && ok; ++l) {
              const LayerDesc& D = P.layer[l];
              for (int uu = u; uu < units_of(P, D) && ok; uu += gridDim.x) {
                const Unit U = unit_of<PS>(P, D, uu, false);
                if (!U.run) continue;
                ok = mbar_wait(bar(B_Q_READY), qi & 1);
                fence_after();
                for (int t = 0; t <= U.n_tiles && ok; ++t) {
                    if (t < U.n_tiles) {
                        const int g = tg + t, s = g % STAGES, sb = g & 1;
                        ok = mbar_wait(bar(B_STG_FULL + s), (g / STAGES) & 1);
                        if (ok && t >= U.app_t0 && t <= U.app_t1)
                            ok = mbar_wait(bar(B_PATCH + (pc + t - U.app_t0) % N_PATCH),
                                           ((pc + t - U.app_t0) / N_PATCH) & 1);
                        if (!ok) break;
                        fence_after();
                        const uint32_t kt = smem_u32(stg + s * STG_BYTES);
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint64_t bd = sdesc(kt + ks * 32, 16, 1024);
                            mma_f8_ts(tmem + TM_S + sb * 128, tmem + TM_QH + 8 * ks, bd, ID_QK, ks > 0);
                            mma_f8_ts(tmem + TM_S + sb * 128, tmem + TM_QL + 8 * ks, bd, ID_QK, 1);
                        }
                        mma_commit(bar(B_S_FULL + sb));
                        mma_commit(bar(B_STG_EMPTY + s));    // K of this stage read
                    }
                    if (t >= 1) {
                        const int g = tg + t - 1, ub = g & 1, vb = g % VBUFS;
                        // the previous unit's epilogue must have read O before the first P.V of this one
                        if (t == 1 && qi > 0) ok = mbar_wait(bar(B_O_FREE), (qi - 1) & 1);
                        if (ok) ok = mbar_wait(bar(B_P_FULL + ub), (g >> 1) & 1);
                        if (ok) ok = mbar_wait(bar(B_V_FULL + vb), (g / VBUFS) & 1);
                        if (!ok) break;
                        fence_after();
                        const uint32_t vf = smem_u32(vbuf + vb * VBUF_BYTES);
#pragma unroll
                        for (int kk = 0; kk < NK / 16; ++kk) {
                            const uint64_t bd = sdesc(vf + kk * 2048, NK * 128, 1024);
                            mma_f16_ts(tmem + TM_O, tmem + TM_S + ub * 128 + 8 * kk, bd, ID_PV, (t > 1 || kk > 0));
                        }
                        mma_commit(bar(B_O_DONE));
                        mma_commit(bar(B_V_EMPTY + vb));
                        if (t == U.n_tiles) mma_commit(bar(B_O_FINAL));
                    }
                }
                tg += U.n_tiles;
                ++qi;
                pc += U.app_t1 >= U.app_t0 ? U.app_t1 - U.app_t0 + 1 : 0;
              }
            }
            // nothing the tensor cores still run may outlive the TMEM allocation
            mma_commit(bar(B_MMA_IDLE));
            mbar_wait(bar(B_MMA_IDLE), 0);
        }
        __syncwarp();
    } else if (is_converter(warp)) {
        // ---------------------------------------------------------- V widening
        const int ct = converter_index(warp) * 32 + lane;
        int tg = 0, di = 0, pc = 0;                         // tiles, dependency waits, patched tiles
        for (int l = 0; l < P.n_layers && ok; ++l) {
          const LayerDesc& D = P.layer[l];
          for (int uu = u; uu < units_of(P, D) && ok; uu += gridDim.x) {
            const Unit U = unit_of<PS>(P, D, uu, false);
            if (!U.run) continue;
            const int n_app = U.app_hi - U.app_lo;
            uint2 kc0 = make_uint2(0, 0), vc0 = make_uint2(0, 0);
            int pos0 = -1, chunk0 = 0;
            float ksc = 1.f, vsc = 1.f;
            auto app_item = [&](int it, uint2& kc, uint2& vc, int& pos, int& chunk) {
                pos = U.app_lo + (it >> 4);
                chunk = it & 15;
                const int m = pos - (U.L - P.M);
                const int64_t src = (((int64_t)U.b * P.M + m) * P.Hkv + U.hk) * 16 + chunk;
                kc = e4m3_encode8(((const uint4*)D.k_new)[src], ksc);
                vc = e4m3_encode8(((const uint4*)D.v_new)[src], vsc);
            };
            for (int t = 0; t < U.n_tiles; ++t) {
                const int g = tg + t, s = g % STAGES, vb = g % VBUFS;
                ok = mbar_wait(bar(B_STG_FULL + s), (g / STAGES) & 1);
                if (ok && g >= VBUFS) ok = mbar_wait(bar(B_V_EMPTY + vb), ((g / VBUFS) - 1) & 1);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                const int k0 = U.k_begin + t * NK;
                if (t == U.app_t0) {
                    // -------------------------------------------- append insert
                    // the new tokens depend on the previous layer: wait until
                    // all of its units have written their output, then write
                    // this head's new tokens to the cache (the cache-insert
                    // encoding), keeping the first item's codes for the patch
                    if (l > 0) {
                        // the first converter warp polls, then releases the
                        // others; every warp arrives, so that none can run a
                        // whole phase ahead to the next unit's wait
                        if (ct == 0) wait_counter(&done[l - 1], (unsigned)units_of(P, P.layer[l - 1]));
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(B_DEP));
                        ok = mbar_wait(bar(B_DEP), di & 1);
                        ++di;
                        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    }
                    ksc = *D.k_scale;
                    vsc = *D.v_scale;
                    for (int it = ct; it < n_app * 16; it += CONV_THREADS) {
                        uint2 kc, vc;
                        int pos, chunk;
                        app_item(it, kc, vc, pos, chunk);
                        if (it == ct) {
                            kc0 = kc;
                            vc0 = vc;
                            pos0 = pos;
                            chunk0 = chunk;
                        }
                        const int page = D.block_table[(int64_t)U.b * D.mpps + pos / PS];
                        if (page < 0 || page >= D.num_pages) {
                            if (chunk == 0) flag(FP8KV_DEV_BAD_SLOT);
                            continue;
                        }
                        const int64_t dst = (((int64_t)page * P.Hkv + U.hk) * PS + pos % PS) * 128 + chunk * 8;
                        *(uint2*)(D.k_cache + dst) = kc;
                        *(uint2*)(D.v_cache + dst) = vc;
                    }
                }
                if (t >= U.app_t0 && t <= U.app_t1) {
                    // patch this tile's new rows (K and V, 128-byte swizzled rows
                    // of the staging buffer) with the appended tokens' codes
                    uint8_t* kst = stg + s * STG_BYTES;
                    for (int it = ct; it < n_app * 16; it += CONV_THREADS) {
                        uint2 kc = kc0, vc = vc0;
                        int pos = pos0, chunk = chunk0;
                        if (it != ct) app_item(it, kc, vc, pos, chunk);
                        const int r = pos - k0;
                        if (r < 0 || r >= NK) continue;
                        const int off = r * 128 + ((((chunk >> 1) ^ r) & 7) << 4) + (chunk & 1) * 8;
                        *(uint2*)(kst + off) = kc;
                        *(uint2*)(kst + STG_K + off) = vc;
                    }
                    fence_proxy_async();                    // for the tensor cores' read of K
                    __syncwarp();
                    const int pk = pc + t - U.app_t0;          // this CTA's patched tile number
                    if (lane == 0) mbar_arrive(bar(B_PATCH + pk % N_PATCH));
                    // every converter warp's rows are in place before V is read
                    ok = mbar_wait(bar(B_PATCH + pk % N_PATCH), (pk / N_PATCH) & 1);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                }
                const int zlo = max(0, min(NK, U.lo0 - k0));
                const int pages_here = min(PPT, U.n_pages - t * PPT);
                const int zhi = max(0, min(min(NK, pages_here * PS), U.hi0 + 1 - k0));
                const uint8_t* src = stg + s * STG_BYTES + STG_K;
                uint8_t* dst = vbuf + vb * VBUF_BYTES;
                constexpr int PER = (NK * 8 + CONV_THREADS - 1) / CONV_THREADS;   // chunks per thread
                uint4 code[PER];
#pragma unroll
                for (int w = 0; w < PER; ++w) {
                    const int i = ct + CONV_THREADS * w;
                    const int r = i >> 3, c = i & 7;
                    code[w] = (i < NK * 8 && r >= zlo && r < zhi)
                                  ? *(const uint4*)(src + r * 128 + (((c ^ r) & 7) << 4))
                                  : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int w = 0; w < PER; ++w) {
                    const int i = ct + CONV_THREADS * w;
                    if (i >= NK * 8) break;
                    const int r = i >> 3, c = i & 7;
                    uint4 lo, hi;
                    lo.x = e4m3x2_to_f16x2(code[w].x);
                    lo.y = e4m3x2_to_f16x2(code[w].x >> 16);
                    lo.z = e4m3x2_to_f16x2(code[w].y);
                    lo.w = e4m3x2_to_f16x2(code[w].y >> 16);
                    hi.x = e4m3x2_to_f16x2(code[w].z);
                    hi.y = e4m3x2_to_f16x2(code[w].z >> 16);
                    hi.z = e4m3x2_to_f16x2(code[w].w);
                    hi.w = e4m3x2_to_f16x2(code[w].w >> 16);
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
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(B_STG_EMPTY + s));
                    mbar_arrive(bar(B_V_FULL + vb));
                }
            }
            tg += U.n_tiles;
            pc += U.app_t1 >= U.app_t0 ? U.app_t1 - U.app_t0 + 1 : 0;
          }
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int wq = warp & 3, half = (warp - 4) >> 2;
        const int r = wq * 32 + lane;                       // TMEM lane = row of the head's tile
        const int RL = P.R;
        const bool active = wq * 32 < RL;                   // quarter holds at least one real row
        const bool pad = r >= RL;
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        const int st = threadIdx.x - 128;                   // 0..255 among the softmax warps
        int tg = 0, qi = 0, pp = 0;                         // tiles, units, pair-barrier phases
        for (int l = 0; l < P.n_layers && ok; ++l) {
            const LayerDesc& D = P.layer[l];
            const int nu = units_of(P, D);
            if (u >= nu) continue;
            // the queries depend on the previous layer: wait until all of its
            // units have written their output
            if (l > 0) {
                // one thread of the CTA polls (many pollers of one counter slow
                // every access to its memory partition); all eight warps go on,
                // or all stop (the pairs meet at named barriers)
                bool w = true;
                if (st == 0) w = wait_counter(&done[l - 1], (unsigned)units_of(P, P.layer[l - 1]));
                ok = soft_all(w);
                if (!ok) break;
            }
            // this CTA's units of the layer: units u, u + grid, ...  Every unit
            // is counted (its group's partial, or its share of the layer's
            // output), also after a failed wait, so that no CTA waits in vain.
            for (int uu = u; uu < nu; uu += gridDim.x) {
            const Unit U = unit_of<PS>(P, D, uu, threadIdx.x == 128);
            const int g_idx = U.b * P.Hkv + U.hk;
            const int rr = min(r, RL - 1);
            const int m = rr / P.G;
            const int p_r = U.L - P.M + m;
            const int lo_r = (D.window_left >= 0) ? max(0, p_r - D.window_left) : 0;
            const int64_t row_idx = ((int64_t)U.b * P.M + m) * P.Hq + U.hk * P.G + rr % P.G;
            if (ok && U.run) {
                float mult;
                {
                    // Q row split (as in the single-layer kernel): q' = q * 2^sh
                    // with the row maximum in [128, 256), Q_hi = e4m3(q'),
                    // Q_lo = e4m3(q' - Q_hi), this half's 64 dims of both
                    const uint4* src = (const uint4*)(D.q + row_idx * 128) + 8 * half;
                    uint32_t qh[32];
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const uint4 x = pad ? make_uint4(0, 0, 0, 0) : src[w];
                        qh[4 * w] = x.x;
                        qh[4 * w + 1] = x.y;
                        qh[4 * w + 2] = x.z;
                        qh[4 * w + 3] = x.w;
                    }
                    uint32_t am = 0;
#pragma unroll
                    for (int w = 0; w < 32; ++w) am = max_bf16x2(am, qh[w] & 0x7fff7fffu);
                    float amax = fmaxf(bf16_lo(am), bf16_hi(am));
                    xch[half * 128 + r] = amax;
                    asm volatile("bar.sync %0, 64;" ::"r"(1 + wq) : "memory");
                    amax = fmaxf(xch[r], xch[128 + r]);
                    asm volatile("bar.sync %0, 64;" ::"r"(1 + wq) : "memory");
                    int e = 7;
                    const uint32_t ab = __float_as_uint(amax);
                    if (amax > 0.f && ((ab >> 23) & 0xff) != 0xff) {
                        const int be = (int)((ab >> 23) & 0xff);
                        e = be ? be - 127 : -127;
                    }
                    const int sh = max(-100, min(100, 7 - e));
                    const float scale = ldexpf(1.0f, sh);
                    mult = (*D.k_scale) * D.sm_scale * 1.4426950408889634f * ldexpf(1.0f, -sh);
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

                int pmin = p_r, lomax = lo_r;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    pmin = min(pmin, __shfl_xor_sync(0xffffffffu, pmin, off));
                    lomax = max(lomax, __shfl_xor_sync(0xffffffffu, lomax, off));
                }
                float m_run = -INFINITY, l_run = 0.f;
                for (int t = 0; t < U.n_tiles; ++t) {
                    const int g = tg + t, sb = g & 1;
                    ok = mbar_wait(bar(B_S_FULL + sb), (g >> 1) & 1);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    fence_after();
                    if (active) {
                        const uint32_t scol = lane_base + TM_S + sb * 128 + 64 * half;
                        const int k0 = U.k_begin + t * NK + 64 * half;
                        uint32_t sv[64];
                        tmem_ld_x64(scol, sv);
                        tmem_wait_ld();
                        if ((k0 + 63 > pmin) || (k0 < lomax)) {
#pragma unroll
                            for (int j = 0; j < 64; ++j)
                                if (k0 + j > p_r || k0 + j < lo_r) sv[j] = 0xff800000u;   // -inf
                        }
                        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                        for (int j = 0; j < 64; j += 4) {
                            m4[0] = fmaxf(m4[0], __uint_as_float(sv[j]));
                            m4[1] = fmaxf(m4[1], __uint_as_float(sv[j + 1]));
                            m4[2] = fmaxf(m4[2], __uint_as_float(sv[j + 2]));
                            m4[3] = fmaxf(m4[3], __uint_as_float(sv[j + 3]));
                        }
                        xch[(sb * 2 + half) * 128 + r] = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(B_PAIR + wq));
                        ok = mbar_wait(bar(B_PAIR + wq), pp & 1);
                        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                        const float smax = fmaxf(xch[sb * 256 + r], xch[sb * 256 + 128 + r]);
                        const float tmax = smax * mult;
                        const bool rescale = (m_run != -INFINITY) && (tmax > m_run + 8.0f);
                        if (__any_sync(0xffffffffu, rescale)) {
                            // O holds P.V up to tile t-1: wait for it, then rescale this half
                            const bool okw = mbar_wait(bar(B_O_DONE), (g - 1) & 1);
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
                        float sum0 = 0.f, sum1 = 0.f;
                        uint32_t pw[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float p0 = ex2(fmaf(__uint_as_float(sv[2 * j]), mult, neg));
                            const float p1 = ex2(fmaf(__uint_as_float(sv[2 * j + 1]), mult, neg));
                            sum0 += p0;
                            sum1 += p1;
                            pw[j] = pack_f16x2(p0, p1);
                        }
                        tmem_st_x32(lane_base + TM_S + sb * 128 + 32 * half, pw);
                        l_run += sum0 + sum1;
                        tmem_wait_st();
                    }
                    ++pp;
                    fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_P_FULL + sb));
                }
                // ------------------------------------------------------ epilogue
                if (ok) ok = mbar_wait(bar(B_O_FINAL), qi & 1);
                ok = __all_sync(0xffffffffu, ok);
                float l_tot = 0.f;
                if (ok && active) {
                    fence_after();
                    xch[(4 + half) * 128 + r] = l_run;      // row sums of both halves
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_PAIR + wq));
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(B_PAIR + wq), pp & 1));
                    l_tot = xch[4 * 128 + r] + xch[5 * 128 + r];
                }
                ++pp;
                // direct: bf16 of O * v_scale / l; partial: f16 of O / l in code
                // units (|x| <= 448) with (max, sum) beside it
                const bool direct = U.nsplit_b == 1;
                const float f = direct ? *D.v_scale / l_tot : (l_tot > 0.f ? 1.0f / l_tot : 0.f);
                uint8_t* row_stage = epi + (half * 128 + r) * EPI_STRIDE;
                if (ok && active) {
#pragma unroll 1
                    for (int c = 0; c < 64; c += 32) {
                        uint32_t ov[32];
                        tmem_ld_x32(lane_base + TM_O + 64 * half + c, ov);
                        tmem_wait_ld();
                        uint4* dst = (uint4*)(row_stage + c * 2);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            const float a0 = __uint_as_float(ov[8 * v4 + 0]) * f, a1 = __uint_as_float(ov[8 * v4 + 1]) * f;
                            const float a2 = __uint_as_float(ov[8 * v4 + 2]) * f, a3 = __uint_as_float(ov[8 * v4 + 3]) * f;
                            const float a4 = __uint_as_float(ov[8 * v4 + 4]) * f, a5 = __uint_as_float(ov[8 * v4 + 5]) * f;
                            const float a6 = __uint_as_float(ov[8 * v4 + 6]) * f, a7 = __uint_as_float(ov[8 * v4 + 7]) * f;
                            dst[v4] = direct ? make_uint4(pack_bf16x2(a0, a1), pack_bf16x2(a2, a3), pack_bf16x2(a4, a5),
                                                          pack_bf16x2(a6, a7))
                                             : make_uint4(pack_f16x2(a0, a1), pack_f16x2(a2, a3), pack_f16x2(a4, a5),
                                                          pack_f16x2(a6, a7));
                        }
                    }
                }
                // O has been read: the next unit's P.V may overwrite it
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_O_FREE));
                if (ok && active && r < RL) {
                    fence_proxy_async();                    // the staged row, to the bulk copy
                    if (direct)
                        bulk_store(D.out + row_idx * 128 + 64 * half, smem_u32(row_stage), 128);
                    else
                        bulk_store(P.part_o + (row_idx * P.max_splits + U.split) * 128 + 64 * half,
                                   smem_u32(row_stage), 128);
                    bulk_commit();
                    if (!direct && half == 0) {
                        P.part_ml[(row_idx * P.max_splits + U.split) * 2] = m_run;
                        P.part_ml[(row_idx * P.max_splits + U.split) * 2 + 1] = l_tot;
                    }
                    // the rows are in global memory before the counter says so
                    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                tg += U.n_tiles;
                ++qi;
            }
            ok = soft_all(ok);
            const bool multi = U.seq_ok && U.nsplit_b > 1 && U.nsplit_b <= D.num_splits;
            if (st == 0) {
                // partial written (the group's counter), or this unit's rows of
                // the output written directly (the layer's counter)
                __threadfence();
                red_release_add(multi ? &grp[(size_t)l * P.B * P.Hkv + g_idx] : &done[l], 1u);
            }
            }
            // ------------------------------------------- combine partitions
            // Only after all of this CTA's units of the layer: a CTA never
            // waits for a group while a unit it has yet to run belongs to
            // another CTA's awaited group.  Each partition's CTA combines a
            // share of its group's rows.
            for (int uu = u; uu < nu; uu += gridDim.x) {
                const Unit U = unit_of<PS>(P, D, uu, false);
                const int g_idx = U.b * P.Hkv + U.hk;
                const bool multi = U.seq_ok && U.nsplit_b > 1 && U.nsplit_b <= D.num_splits;
                if (!multi) continue;
                bool w = ok;
                if (st == 0 && ok) w = wait_counter(&grp[(size_t)l * P.B * P.Hkv + g_idx], (unsigned)D.num_splits);
                ok = soft_all(w && ok);
                if (ok) {
                    // rows split, split + num_splits, ... of the group: one warp per row
                    const float vsc = *D.v_scale;
                    const int sw = warp - 4;                // 0..7
                    for (int rw = U.split + D.num_splits * sw; rw < RL; rw += D.num_splits * 8) {
                        const int mw = rw / P.G;
                        const int64_t orow = ((int64_t)U.b * P.M + mw) * P.Hq + U.hk * P.G + rw % P.G;
                        const uint16_t* po = P.part_o + orow * P.max_splits * 128 + 4 * lane;
                        const float* pml = P.part_ml + orow * P.max_splits * 2;
                        float mp = -INFINITY, lp = 0.f;
                        if (lane < U.nsplit_b) {
                            mp = pml[2 * lane];
                            lp = pml[2 * lane + 1];
                        }
                        uint2 v[16];
#pragma unroll
                        for (int p = 0; p < 16; ++p)
                            v[p] = p < U.nsplit_b ? *(const uint2*)(po + (int64_t)p * 128) : make_uint2(0, 0);
                        float mstar = mp;
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1) mstar = fmaxf(mstar, __shfl_xor_sync(0xffffffffu, mstar, off));
                        const float w8 = (mp == -INFINITY) ? 0.f : ex2(mp - mstar) * lp;
                        float lsum = w8;
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
                        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                        for (int p = 0; p < 16; ++p) {
                            const float wp = __shfl_sync(0xffffffffu, w8, p);   // 0 past nsplit_b
                            const float2 a = f16x2_to_f32x2(v[p].x), c2 = f16x2_to_f32x2(v[p].y);
                            acc.x = fmaf(wp, a.x, acc.x);
                            acc.y = fmaf(wp, a.y, acc.y);
                            acc.z = fmaf(wp, c2.x, acc.z);
                            acc.w = fmaf(wp, c2.y, acc.w);
                        }
                        const float inv = vsc / lsum;
                        *(uint2*)(D.out + orow * 128 + 4 * lane) =
                            make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
                    }
                }
                ok = soft_all(ok);
                // this unit's share of the layer's output is written (counted
                // even after a failed wait, so that no other CTA waits for it in vain)
                if (st == 0) {
                    __threadfence();
                    red_release_add(&done[l], 1u);
                }
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
    if (threadIdx.x == 0) {
        // the last CTA to leave sets the counters back to zero for the next
        // call (every other CTA has finished reading them)
        __threadfence();
        const unsigned prev = atomicAdd(exit_count, 1u);
        if (prev == gridDim.x - 1) {
            __threadfence();
            const size_t n = (size_t)P.n_layers * P.B * P.Hkv + P.n_layers;
            for (size_t i = 0; i < n; ++i) P.counters[i] = 0;
            __threadfence();
            *exit_count = 0;
        }
    }
}

}  // namespace pl

int layers_threads() { return pl::THREADS; }

int launch_attention_layers(const LayersParams& P, int page_size, int grid, cudaStream_t s) {
    static std::mutex mu;
    static std::set<std::pair<int, const void*>> done;
    const void* kern = page_size == 32 ? (const void*)pl::attention_layers_kernel<32>
                                       : (const void*)pl::attention_layers_kernel<64>;
    {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return FP8KV_ERR_CUDA;
        std::lock_guard<std::mutex> lock(mu);
        if (!done.count({dev, kern})) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl::SMEM) != cudaSuccess)
                return FP8KV_ERR_CUDA;
            done.insert({dev, kern});
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(pl::THREADS);
    cfg.dynamicSmemBytes = pl::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;    // every CTA resident: the counter waits end
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = page_size == 32 ? cudaLaunchKernelEx(&cfg, pl::attention_layers_kernel<32>, P)
                                          : cudaLaunchKernelEx(&cfg, pl::attention_layers_kernel<64>, P);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return FP8KV_ERR_CUDA;
    }
    count_launch();
    return FP8KV_OK;
}

// Largest grid of this kernel with every CTA resident (one per SM).
int layers_max_grid() {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    const void* kern = (const void*)pl::attention_layers_kernel<32>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl::SMEM) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pl::attention_layers_kernel<32>, pl::THREADS,
                                                      pl::SMEM) != cudaSuccess)
        return 0;
    return sms * per_sm;
}

}  // namespace fp8kv

// =====================================================================  host

using namespace fp8kv;

namespace {

int ceil_div_i(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// Counters, then the partials (one region: layers run one after another).
size_t counters_bytes(int n_layers, int B, int Hkv) {
    return ((size_t)n_layers * B * Hkv + n_layers + 1) * sizeof(unsigned) + 255 & ~(size_t)255;
}

size_t layers_ws_bytes(int n_layers, int B, int M, int Hq, int Hkv) {
    const size_t rows = (size_t)B * M * Hq;
    return counters_bytes(n_layers, B, Hkv) + rows * kLayersMaxSplits * 128 * sizeof(uint16_t) +
           rows * kLayersMaxSplits * 2 * sizeof(float);
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" size_t fp8kv_paged_attention_layers_workspace_size(int n_layers, int B, int M, int Hq, int Hkv) {
    if (n_layers <= 0 || n_layers > kMaxLayers || B <= 0 || M <= 0 || Hq <= 0 || Hkv <= 0) return (size_t)-1;
    return layers_ws_bytes(n_layers, B, M, Hq, Hkv);
}

extern "C" int fp8kv_paged_attention_layers(const fp8kv_layer* layers, int n_layers, int B, int M, int Hq, int Hkv,
                                            int D, int page_size, int cache_dtype, void* workspace,
                                            size_t workspace_bytes, void* stream) {
    if (!layers || n_layers <= 0 || B < 0 || M < 1 || Hq <= 0 || Hkv <= 0 || Hq % Hkv) return FP8KV_ERR_INVALID_ARG;
    if (cache_dtype != FP8KV_CACHE_E4M3 && cache_dtype != FP8KV_CACHE_BF16) return FP8KV_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    const int64_t R = (int64_t)M * G;
    // one 128-row tile of verifier rows per KV head on an E4M3 cache
    if (cache_dtype != FP8KV_CACHE_E4M3 || D != 128 || (page_size != 32 && page_size != 64) || R <= 16 ||
        R > 128 || n_layers > kMaxLayers)
        return FP8KV_ERR_UNSUPPORTED;
    if (B == 0) return FP8KV_OK;
    for (int l = 0; l < n_layers; ++l) {
        const fp8kv_layer& A = layers[l];
        if (!A.q || !A.k_cache || !A.v_cache || !A.block_table || !A.seq_lens || !A.out || !A.k_scale ||
            !A.v_scale)
            return FP8KV_ERR_INVALID_ARG;
        if ((A.k_new != nullptr) != (A.v_new != nullptr)) return FP8KV_ERR_INVALID_ARG;
        if (!al16(A.q) || !al16(A.k_cache) || !al16(A.v_cache) || !al16(A.out) ||
            (A.k_new && (!al16(A.k_new) || !al16(A.v_new))))
            return FP8KV_ERR_INVALID_ARG;
        if (A.num_pages <= 0 || A.max_pages_per_seq <= 0 || A.window_left < -1) return FP8KV_ERR_INVALID_ARG;
        if (A.max_seq_len < M || (int64_t)A.max_seq_len > (int64_t)A.max_pages_per_seq * page_size)
            return FP8KV_ERR_INVALID_ARG;
        if (!(A.sm_scale == A.sm_scale)) return FP8KV_ERR_INVALID_ARG;
    }
    const size_t need = layers_ws_bytes(n_layers, B, M, Hq, Hkv);
    if (!workspace || workspace_bytes < need || !al16(workspace)) return FP8KV_ERR_WORKSPACE;
    const int grid = layers_max_grid();
    if (grid <= 0) return FP8KV_ERR_CUDA;

    static thread_local LayersParams P;          // 25 KB: kept off the stack
    P.n_layers = n_layers;
    P.B = B;
    P.M = M;
    P.Hq = Hq;
    P.Hkv = Hkv;
    P.G = G;
    P.R = (int)R;
    P.max_splits = kLayersMaxSplits;
    P.counters = (unsigned*)workspace;
    const size_t rows = (size_t)B * M * Hq;
    P.part_o = (uint16_t*)((uint8_t*)workspace + counters_bytes(n_layers, B, Hkv));
    P.part_ml = (float*)(P.part_o + rows * kLayersMaxSplits * 128);
    const int tile_pages = 128 / page_size;
    // partitions per (sequence, KV head): about two units per CTA and layer,
    // and for many sequences at least a quarter of the longest one each
    // (units past the grid run one after another on the CTAs)
    const int64_t groups = (int64_t)B * Hkv;
    const int spread = (int)std::min<int64_t>(kLayersMaxSplits, std::max<int64_t>(1, (2 * grid + groups - 1) / groups));
    const int units_per_group = std::min(kLayersMaxSplits, groups > grid / 2 ? std::max(4, spread) : spread);
    int max_splits_used = 1;
    for (int l = 0; l < n_layers; ++l) {
        const fp8kv_layer& A = layers[l];
        LayerDesc& Dd = P.layer[l];
        if (!cache_map(&Dd.tm_k, A.k_cache, true, Hkv, page_size, A.num_pages) ||
            !cache_map(&Dd.tm_v, A.v_cache, true, Hkv, page_size, A.num_pages))
            return FP8KV_ERR_CUDA;
        // pages spanned by the visible keys of the longest sequence, in
        // partitions of whole 128-key tiles, at most units_per_group of them
        int pages = ceil_div_i(std::max(A.max_seq_len, 1), page_size);
        if (A.window_left >= 0) pages = std::min(pages, ceil_div_i((int64_t)M + A.window_left, page_size) + 1);
        const int tiles = ceil_div_i(pages, tile_pages);
        const int split_tiles = ceil_div_i(tiles, std::min(tiles, units_per_group));
        Dd.split_pages = split_tiles * tile_pages;
        Dd.num_splits = ceil_div_i(pages, Dd.split_pages);
        max_splits_used = std::max(max_splits_used, Dd.num_splits);
        Dd.q = (const uint16_t*)A.q;
        Dd.k_new = (const uint16_t*)A.k_new;
        Dd.v_new = (const uint16_t*)A.v_new;
        Dd.k_cache = (uint8_t*)A.k_cache;
        Dd.v_cache = (uint8_t*)A.v_cache;
        Dd.block_table = A.block_table;
        Dd.seq_lens = A.seq_lens;
        Dd.k_scale = A.k_scale;
        Dd.v_scale = A.v_scale;
        Dd.out = (uint16_t*)A.out;
        Dd.sm_scale = A.sm_scale;
        Dd.mpps = A.max_pages_per_seq;
        Dd.max_seq_len = A.max_seq_len;
        Dd.num_pages = A.num_pages;
        Dd.window_left = A.window_left;
    }
    const int rc = launch_attention_layers(P, page_size, grid, (cudaStream_t)stream);
    if (rc) return rc;
    char buf[256];
    snprintf(buf, sizeof buf,
             "attention_layers<ps=%d,e4m3> layers=%d rows=%d tile=128x128 grid=%d threads=%d max_splits=%d "
             "cooperative=1",
             page_size, n_layers, (int)R, grid, layers_threads(), max_splits_used);
    set_dispatch(buf);
    return FP8KV_OK;
}
