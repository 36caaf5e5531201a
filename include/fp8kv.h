/*
 * fp8kv.h -- C ABI of libfp8kv.so: calibrated-scale E4M3 FP8 paged KV-cache
 * insertion and exact paged decode / speculative-verifier attention on one
 * NVIDIA GB300 (sm_103a).
 *
 * Sources (the "b70-optimization-lab" pages):
 *  - "Laguna S 2.1 INT4 -- calibrated FP8 KV on Intel B70", section "Contract":
 *    target KV is explicit E4M3 FP8 with one calibrated scalar K scale and one V
 *    scale per layer; no runtime scale calculation.  Section "Initial
 *    optimization order": profile the FP8 cache update and exact q1/M12 paged
 *    attention separately; scaled E4M3 insertion at the Q/K norm + RoPE boundary.
 *  - "Laguna S 2.1 KV-cache precision decision", section "What the official
 *    checkpoint requests": kv_cache_scheme = static ("dynamic": false),
 *    symmetric, per-tensor ("strategy": "tensor"), minmax observer; section
 *    "BF16 versus FP8 in concrete terms": 8 KV heads x dim 128, 2048 B per token
 *    per layer in FP8 vs 4096 B in BF16, "quantize, store FP8" on write and
 *    "scale/dequantize" on read; 36 sliding-window-512 and 12 global layers.
 *  - "Laguna FP8 KV -- replicated embedding win, page-32 build, and host
 *    boundary", section "Page-32 attention experiment": page 32 and page 64,
 *    global and sliding attention, and the rule that a fallback path
 *    invalidates a result.
 *  - "Laguna S 2.1 B70 campaign transfer ledger", table "Result progression",
 *    row "Persistent attention metadata": fixed-address metadata refreshed in
 *    place (here: every buffer is caller-owned; the library allocates no
 *    memory).
 *
 * Conventions for every entry point:
 *  - Pointers marked (device) are device pointers owned by the caller; they
 *    must stay valid until the work queued on `stream` has finished.  Host
 *    integers are sizes.  `stream` is a cudaStream_t (NULL = legacy default
 *    stream); all work is queued asynchronously on it, nothing synchronises.
 *  - Arguments are validated on the host before any launch.  A rejected call
 *    returns a status below and launches nothing.  Shapes the kernels do not
 *    implement return FP8KV_ERR_UNSUPPORTED: there is no slower fallback path.
 *  - A failed launch returns FP8KV_ERR_CUDA (cudaGetLastError is consumed).
 *  - Contents that the host cannot see (slot ids, positions, page ids,
 *    sequence lengths) are checked on the device: an offending row is skipped
 *    (never read or written out of bounds) and a bit is set in the device
 *    status word, read with fp8kv_device_status().
 *  - bf16 is the IEEE-like bfloat16 bit layout; every tensor is dense,
 *    row-major, in the order of its dimension list, 16-byte aligned.
 */
#ifndef FP8KV_H
#define FP8KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8KV_OK = 0,
    FP8KV_ERR_INVALID_ARG = 1,  /* null pointer, negative size, misaligned, bad enum */
    FP8KV_ERR_UNSUPPORTED = 2,  /* valid request outside the implemented shapes     */
    FP8KV_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required       */
    FP8KV_ERR_CUDA = 4          /* a CUDA runtime call or a launch failed           */
} fp8kv_status;

typedef enum {
    FP8KV_CACHE_E4M3 = 0,       /* 1 byte per element, E4M3FN codes, scaled          */
    FP8KV_CACHE_BF16 = 1        /* 2 bytes per element, stored as is, scales unused  */
} fp8kv_cache_dtype;

/* Device status bits (fp8kv_device_status). */
#define FP8KV_DEV_BAD_SLOT      0x1u  /* slot_mapping entry >= num_pages*page_size   */
#define FP8KV_DEV_BAD_POSITION  0x2u  /* position outside [0, max_pos)              */
#define FP8KV_DEV_BAD_SEQ_LEN   0x4u  /* seq_len < M or beyond the block-table row  */
#define FP8KV_DEV_WAIT_TIMEOUT  0x8u  /* a bounded pipeline wait gave up            */

/*
 * fp8kv_cache_insert -- write T new tokens into the paged K and V caches.
 *
 * Operation ("KV-cache precision decision", property table row "Cache
 * write/read work": quantize, store FP8; scales per "Contract"): for every
 * token t with slot s = slot_mapping[t] >= 0, head h, element d:
 *     E4M3:  cache[s / page_size][h][s % page_size][d] =
 *                e4m3_rne_satfinite( fp32(x[t][h][d]) / scale )
 *     BF16:  cache[...] = x[t][h][d]  (bits copied, scales ignored, may be NULL)
 * with fp32 IEEE division, round to nearest even, saturation to +-448
 * (infinities included), NaN -> 0x7F with the input's sign, -0 -> 0x80.
 * Slots < 0 are skipped; slots not named are left untouched.  Duplicate
 * non-negative slots race (unspecified which token wins).
 *
 *   k, v          (device) bf16 [T][Hkv][D]
 *   slot_mapping  (device) int64 [T]
 *   k_scale, v_scale (device) one fp32 each, > 0 (E4M3 only)
 *   k_cache, v_cache (device) [num_pages][Hkv][page_size][D] of the cache dtype
 *   D must be 128; page_size 32 or 64; T may be 0 (no launch, FP8KV_OK, no
 *   pointer is read).
 * Device check: slot >= num_pages*page_size -> row skipped, FP8KV_DEV_BAD_SLOT.
 */
int fp8kv_cache_insert(const void* k, const void* v, const int64_t* slot_mapping, int T,
                       int Hkv, int D, const float* k_scale, const float* v_scale,
                       void* k_cache, void* v_cache, int num_pages, int page_size,
                       int cache_dtype, void* stream);

/*
 * fp8kv_cache_insert_per_head -- fp8kv_cache_insert on an E4M3 cache with one
 * scale per KV head: head h of K (V) is encoded with k_scale[h] (v_scale[h]).
 * An extension the pages do not use: their checkpoint asks for one static
 * symmetric scale per tensor ("KV-cache precision decision", "What the
 * official checkpoint requests", strategy "tensor"); a per-head scale keeps
 * the same encoding with a finer calibration grain.
 *
 *   k_scale, v_scale (device) fp32 [Hkv], each > 0
 *   every other argument, check and status as fp8kv_cache_insert with
 *   cache_dtype = FP8KV_CACHE_E4M3.
 */
int fp8kv_cache_insert_per_head(const void* k, const void* v, const int64_t* slot_mapping, int T,
                                int Hkv, int D, const float* k_scale, const float* v_scale,
                                void* k_cache, void* v_cache, int num_pages, int page_size,
                                void* stream);

/*
 * fp8kv_qk_norm_rope_insert -- the Q/K RMSNorm + RoPE boundary fused with the
 * E4M3 insert ("calibrated FP8 KV on Intel B70", "Initial optimization order",
 * item 3; ledger table "Result progression", row "Exact fusion stack").
 *
 * For each token t at position pos = positions[t] and each Q head and K head
 * row x (D = 128), in fp32 with this fixed order (reproduced bit for bit):
 *     part_l  = sum of squares of x[4l..4l+3] accumulated as
 *               fma(x3,x3, fma(x2,x2, fma(x1,x1, x0*x0)))          l = 0..31
 *     ss      = parts added pairwise: l + (l+16), then +8, +4, +2, +1
 *     r       = 1 / sqrt(ss / 128 + eps)                (IEEE sqrt, divide)
 *     y_i     = bf16( bf16(x_i * r) * w_i )
 *     o_k     = bf16( fma(y_k,    c_k, -(y_k+64 * s_k)) )   k = 0..63
 *     o_k+64  = bf16( fma(y_k+64, c_k,   y_k    * s_k ) )
 * with c_k = cos_sin[pos][k], s_k = cos_sin[pos][64 + k].  Q rows go to q_out;
 * rotated K rows and the raw V rows are inserted as in fp8kv_cache_insert
 * (E4M3 cache only).
 *
 *   q (device) bf16 [T][Hq][D]; k, v (device) bf16 [T][Hkv][D]
 *   positions (device) int64 [T]; q_norm_w, k_norm_w (device) bf16 [D]
 *   cos_sin (device) fp32 [max_pos][D]: cos of the 64 frequencies, then sines
 *   q_out (device) bf16 [T][Hq][D] (must not alias q)
 *   other arguments as fp8kv_cache_insert.
 * Device checks: position outside [0, max_pos) -> token skipped entirely
 * (FP8KV_DEV_BAD_POSITION); bad slot -> K/V of that token skipped.
 * T = 0 launches nothing and returns FP8KV_OK without reading any pointer.
 */
int fp8kv_qk_norm_rope_insert(const void* q, const void* k, const void* v,
                              const int64_t* positions, const void* q_norm_w,
                              const void* k_norm_w, float eps, const float* cos_sin,
                              int max_pos, void* q_out, const int64_t* slot_mapping, int T,
                              int Hq, int Hkv, int D, const float* k_scale,
                              const float* v_scale, void* k_cache, void* v_cache,
                              int num_pages, int page_size, void* stream);

/*
 * fp8kv_paged_attention_plan -- the split-KV partition fp8kv_paged_attention
 * will use for these host-visible sizes on the current device.
 *   split_tokens: 0 = choose automatically; otherwise a positive multiple of
 *   page_size.  Returns FP8KV_OK and writes *num_splits (>= 1, the largest
 *   number of partitions any sequence can have) and *split_tokens_out.
 */
int fp8kv_paged_attention_plan(int B, int M, int Hq, int Hkv, int D, int page_size,
                               int max_seq_len, int window_left, int split_tokens,
                               int* num_splits, int* split_tokens_out);

/* Workspace bytes fp8kv_paged_attention needs for the same arguments: room
 * for the split-KV partials (fp32 output, max and sum per query row and
 * partition) when a sequence spans several partitions, counted even when the
 * call combines them on chip.  The size does not depend on the cache dtype.
 * 0 for one partition; (size_t)-1 on bad arguments. */
size_t fp8kv_paged_attention_workspace_size(int B, int M, int Hq, int Hkv, int D,
                                            int page_size, int max_seq_len, int window_left,
                                            int split_tokens);

/*
 * fp8kv_paged_attention -- exact paged attention over the cache for M new
 * query rows per sequence ("calibrated FP8 KV on Intel B70", "Initial
 * optimization order", items 2 and 4; M = 1 is decode, M = 12 the width-12
 * verifier of "Contract").
 *
 * Sequence b has L = seq_lens[b] tokens cached, the last M of them the new
 * rows; row m sits at position p = L - M + m and query head h reads KV head
 * h / (Hq/Hkv).  Key j is visible to row m iff j <= p and, when
 * window_left >= 0, j >= p - window_left (a window of W keys including the
 * row itself is window_left = W - 1).  Logical key j lives in physical page
 * block_table[b][j / page_size] at offset j % page_size.  With
 * Kd = decode(k_code) * k_scale, Vd = decode(v_code) * v_scale (BF16 cache:
 * the stored values, scales unused):
 *     out[b][m][h] = softmax_j( (q . Kd_j) * sm_scale ) . Vd      (rounded to bf16)
 * computed with fp32 accumulation.  Long contexts are cut into partitions of
 * split_tokens keys whose partial (max, sum, unnormalised output) are combined
 * through their log-sum-exp: by a reduce kernel over workspace partials, or,
 * for one sequence (B = 1) of 17 to 128 rows per KV head (one row tile) on an
 * E4M3 cache in at most 8 partitions, on chip by the partitions of a KV head running as one
 * thread-block cluster (fp8kv_last_dispatch reports "cluster=N").
 *
 *   q            (device) bf16 [B][M][Hq][D]
 *   k_cache, v_cache (device) [num_pages][Hkv][page_size][D] (cache_dtype)
 *   block_table  (device) int32 [B][max_pages_per_seq]; entries of pages with
 *                no visible key are never read
 *   seq_lens     (device) int32 [B]; max_seq_len (host) >= every seq_lens[b]
 *   k_scale, v_scale (device) fp32 scalars (E4M3 only)
 *   sm_scale     (host) fp32 logit multiplier, e.g. 1/sqrt(D)
 *   window_left  (host) -1 for a global layer, else >= 0
 *   split_tokens (host) 0 = automatic, else a multiple of page_size
 *   workspace    (device) >= fp8kv_paged_attention_workspace_size(...) bytes,
 *                may be NULL when that size is 0; contents need no
 *                initialisation and are scratch after the call
 *   out          (device) bf16 [B][M][Hq][D]
 * Supported: D = 128, page_size 32 or 64, Hq % Hkv == 0, and either
 * 1 <= M <= 16 with M * (Hq/Hkv) <= 144 rows per KV head (any cache type), or
 * up to M = 16384 query rows per sequence on an E4M3 cache with partitions of
 * whole 128-key tiles (split_tokens 0 or a multiple of 128): a prefill chunk
 * at the end of the context, causal within the chunk, on the tcgen05 kernel
 * in 128-row tiles (Hkv * ceil(M * Hq/Hkv / 128) <= 65535); other shapes
 * return FP8KV_ERR_UNSUPPORTED.  B = 0 launches nothing and returns FP8KV_OK
 * without reading any pointer.
 * Device checks: seq_len < M, seq_len > max_seq_len or more pages than
 * max_pages_per_seq -> that sequence's output is left untouched
 * (FP8KV_DEV_BAD_SEQ_LEN); page ids outside [0, num_pages) read zeros.
 */
int fp8kv_paged_attention(const void* q, const void* k_cache, const void* v_cache,
                          int cache_dtype, const int32_t* block_table, int max_pages_per_seq,
                          const int32_t* seq_lens, int max_seq_len, int B, int M, int Hq,
                          int Hkv, int D, int page_size, int num_pages, const float* k_scale,
                          const float* v_scale, float sm_scale, int window_left,
                          int split_tokens, void* workspace, size_t workspace_bytes, void* out,
                          void* stream);

/*
 * fp8kv_append_paged_attention -- one verifier step of a layer: the M new
 * tokens of every sequence are written to the cache, then attention runs
 * ("calibrated FP8 KV on Intel B70", "Contract": the insert at the new rows'
 * positions followed by the exact paged attention over the cache).
 *
 * Token m of sequence b (k_new, v_new: bf16 [B][M][Hkv][D], device) goes to
 * position p = seq_lens[b] - M + m, i.e. slot
 * block_table[b][p / page_size] * page_size + p % page_size, with the
 * fp8kv_cache_insert encoding; then fp8kv_paged_attention runs with the same
 * arguments.  Cache bytes and output are identical to fp8kv_cache_insert
 * with those slots followed by fp8kv_paged_attention.  On the tensor-memory
 * path with one 128-row tile per KV head the CTA whose partition holds a new
 * position writes it before loading that page (no separate insert launch);
 * otherwise (a prefill chunk in several row tiles, or the mma.sync kernels)
 * an append kernel runs first.  k_new and v_new must be 16-byte aligned; B = 0 is a no-op.
 * Device check: a block-table entry outside [0, num_pages) at a new
 * position -> that token is not written (FP8KV_DEV_BAD_SLOT).
 */
int fp8kv_append_paged_attention(const void* k_new, const void* v_new, const void* q, void* k_cache,
                                 void* v_cache, int cache_dtype, const int32_t* block_table,
                                 int max_pages_per_seq, const int32_t* seq_lens, int max_seq_len, int B,
                                 int M, int Hq, int Hkv, int D, int page_size, int num_pages,
                                 const float* k_scale, const float* v_scale, float sm_scale,
                                 int window_left, int split_tokens, void* workspace,
                                 size_t workspace_bytes, void* out, void* stream);

/*
 * fp8kv_paged_attention_per_head, fp8kv_append_paged_attention_per_head --
 * fp8kv_paged_attention and fp8kv_append_paged_attention on an E4M3 cache
 * written with per-head scales (fp8kv_cache_insert_per_head): KV head hk is
 * dequantized with k_scale[hk], v_scale[hk] (device fp32 [Hkv]), and the
 * append encodes head hk's new tokens with them:
 *     Kd = decode(k_code) * k_scale[hk],  Vd = decode(v_code) * v_scale[hk]
 * Every other argument, kernel choice, check and status as the per-tensor
 * entry points with cache_dtype = FP8KV_CACHE_E4M3 (the same workspace size).
 */
int fp8kv_paged_attention_per_head(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_table, int max_pages_per_seq,
                                   const int32_t* seq_lens, int max_seq_len, int B, int M, int Hq,
                                   int Hkv, int D, int page_size, int num_pages, const float* k_scale,
                                   const float* v_scale, float sm_scale, int window_left,
                                   int split_tokens, void* workspace, size_t workspace_bytes, void* out,
                                   void* stream);

int fp8kv_append_paged_attention_per_head(const void* k_new, const void* v_new, const void* q,
                                          void* k_cache, void* v_cache, const int32_t* block_table,
                                          int max_pages_per_seq, const int32_t* seq_lens, int max_seq_len,
                                          int B, int M, int Hq, int Hkv, int D, int page_size,
                                          int num_pages, const float* k_scale, const float* v_scale,
                                          float sm_scale, int window_left, int split_tokens,
                                          void* workspace, size_t workspace_bytes, void* out,
                                          void* stream);

/*
 * fp8kv_paged_attention_layers -- the verifier step of several layers in one
 * launch: for each layer in order, fp8kv_append_paged_attention (or, with
 * k_new = v_new = NULL, fp8kv_paged_attention) with the same results
 * ("Laguna S 2.1 B70 campaign transfer ledger", table "Result progression",
 * rows on graph coverage and persistent attention metadata; "Laguna S 2.1
 * INT4 -- calibrated FP8 KV on Intel B70", section "Contract": the width-12
 * verifier over the FP8 cache).
 *
 * One persistent, cooperative launch with one CTA per SM.  Layer order is
 * kept: a layer's queries and new tokens are read only after every output row
 * of the previous layer has been written, as if the previous layer's output
 * produced them.  The pages of the earlier context are loaded ahead, across
 * layer boundaries.  Partitions of a sequence's keys combine through the
 * workspace (normalised f16 partials in E4M3 code units and fp32 (max, sum),
 * as the cluster combine of fp8kv_paged_attention), so results equal those of
 * the per-layer calls within the attention tolerance, not bit for bit.
 *
 *   layers     (host) n_layers descriptors (1 .. 64), each naming one layer's
 *              tensors with the meaning, layout and dtype they have in
 *              fp8kv_append_paged_attention: q, k_new, v_new (device, bf16,
 *              k_new/v_new may both be NULL), k_cache, v_cache (device, E4M3),
 *              block_table, seq_lens (device, int32), k_scale, v_scale
 *              (device fp32), out (device bf16), and host sizes
 *              max_pages_per_seq, max_seq_len, num_pages, window_left,
 *              sm_scale.  Layers may share or have their own tensors.
 *   B, M, Hq, Hkv, D, page_size, cache_dtype: as fp8kv_paged_attention, the
 *              same for every layer.
 *   workspace  (device) >= fp8kv_paged_attention_layers_workspace_size bytes,
 *              16-byte aligned.  Its first bytes hold the launch's
 *              synchronisation counters: they must be zero before the first
 *              call on a workspace (cudaMemset once) and every call leaves
 *              them zero.  Calls sharing a workspace must not overlap on the
 *              GPU.
 * Supported: E4M3 cache, D = 128, page_size 32 or 64, 16 < M*Hq/Hkv <= 128
 * (one 128-row tile of verifier rows per KV head), any B (with more work
 * units than SMs, a CTA runs several units of a layer one after another);
 * other shapes return FP8KV_ERR_UNSUPPORTED.  Per-layer arguments are
 * validated as in fp8kv_paged_attention before anything is launched.
 * Device checks as fp8kv_paged_attention; a wait that runs out (2 s) sets
 * FP8KV_DEV_WAIT_TIMEOUT and the launch still ends.
 */
typedef struct {
    const void* q;
    const void* k_new;
    const void* v_new;
    void* k_cache;
    void* v_cache;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const float* k_scale;
    const float* v_scale;
    void* out;
    int max_pages_per_seq;
    int max_seq_len;
    int num_pages;
    int window_left;
    float sm_scale;
} fp8kv_layer;

/* Workspace bytes of fp8kv_paged_attention_layers; (size_t)-1 on bad arguments. */
size_t fp8kv_paged_attention_layers_workspace_size(int n_layers, int B, int M, int Hq, int Hkv);

int fp8kv_paged_attention_layers(const fp8kv_layer* layers, int n_layers, int B, int M, int Hq, int Hkv,
                                 int D, int page_size, int cache_dtype, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * fp8kv_paged_attention_noalloc -- fp8kv_paged_attention without a
 * caller-provided workspace.  (The pages have no counterpart: this is an
 * integration convenience, not part of the method.)
 *
 * For callers that cannot allocate device memory where they run attention
 * (an allocator-free serving loop, a fully carved-up memory pool, host code
 * holding only a raw stream): the split-KV partials go to a buffer that is a
 * file-scope __device__ array of FP8KV_NOALLOC_WORKSPACE_BYTES (32 MiB) inside
 * the library.  Every GPU that loads the library holds that buffer until the
 * process exits.  The call allocates nothing (no cudaMalloc, no allocating
 * library routine).
 *
 * Arguments and results are those of fp8kv_paged_attention without
 * workspace / workspace_bytes; out must hold B*M*Hq*D bf16 values (the C
 * entry point cannot check its size).  Every argument is validated first,
 * with the statuses of fp8kv_paged_attention; then a request whose workspace
 * size (fp8kv_paged_attention_workspace_size) exceeds 32 MiB returns
 * FP8KV_ERR_WORKSPACE (a larger split_tokens needs less; otherwise use the
 * allocating entry point).  The first call on a device looks up the buffer's
 * device address (cudaGetSymbolAddress, with that device current) and keeps
 * it for the life of the process; make that first call before any stream
 * capture.  A cudaDeviceReset while the library is loaded is not supported
 * (the kept address, like the kernels' shared-memory opt-ins, would be
 * stale).  Every call shares the one buffer, which keeps
 * the last call's contents (no part of it needs to start at zero): calls
 * that overlap on the GPU -- on different streams, or from several threads --
 * race and must be serialised by the caller.
 */
int fp8kv_paged_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                  int cache_dtype, const int32_t* block_table,
                                  int max_pages_per_seq, const int32_t* seq_lens, int max_seq_len,
                                  int B, int M, int Hq, int Hkv, int D, int page_size,
                                  int num_pages, const float* k_scale, const float* v_scale,
                                  float sm_scale, int window_left, int split_tokens, void* out,
                                  void* stream);

/*
 * fp8kv_e4m3_encode_bits -- encode the fp32 bit patterns first .. first+n-1
 * with the same device routine the insert kernels use (for exhaustive checks
 * of the encoder).  out (device) uint8 [n].
 */
int fp8kv_e4m3_encode_bits(uint32_t first, size_t n, uint8_t* out, void* stream);

/*
 * fp8kv_selftest_bounded_wait -- exercise the device-side failure path of a
 * pipeline wait: one warp waits on a barrier that by construction gets no
 * arrival; after limit_us microseconds (1 .. 2000000) the wait gives up, sets
 * FP8KV_DEV_WAIT_TIMEOUT in the device status word and the kernel returns, so
 * the context stays usable.  Every barrier wait of the attention kernels takes
 * the same path after 2 s.  ("Laguna S 2.1 B70 campaign transfer ledger",
 * section "Harness, recovery, and evidence lessons": a stage that does not
 * finish is classified from a bounded wait and a recorded marker, never left
 * to hang.)  Returns FP8KV_OK when launched; read the bit with
 * fp8kv_device_status().
 */
int fp8kv_selftest_bounded_wait(unsigned int limit_us, void* stream);

/* Text of a status code (static storage). */
const char* fp8kv_status_string(int status);

/* Kernel variant and partition count chosen by the last fp8kv_paged_attention
 * call on this host thread, as text (truncated to n-1 bytes).  Returns the
 * full length. */
int fp8kv_last_dispatch(char* buf, size_t n);

/* Number of kernel launches this library has made in this process (all
 * threads, all devices), e.g. the launches one step captures into a graph. */
unsigned long long fp8kv_launch_count(void);

/* Read (and with clear != 0, reset) the device status word of the current
 * device.  Synchronises the device.  Returns FP8KV_OK or FP8KV_ERR_CUDA. */
int fp8kv_device_status(unsigned int* status, int clear);

#ifdef __cplusplus
}
#endif

#endif /* FP8KV_H */
