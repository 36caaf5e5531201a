// attention.cuh -- parameters shared by the paged-attention kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8kv {

struct AttnParams {
    const uint16_t* q;          // bf16 [B][M][Hq][128]
    const int32_t* block_table; // [B][mpps]
    const int32_t* seq_lens;    // [B]
    const float* k_scale;       // [1] per tensor, or [Hkv] per KV head (scale_stride 1)
    const float* v_scale;
    int scale_stride;           // 0: one scale per tensor; 1: scale of KV head hk at [hk]
    float* ws_o;                // [B*M*Hq][num_splits][128]
    float* ws_ml;               // [B*M*Hq][num_splits][2]
    uint16_t* out;              // bf16 [B][M][Hq][128]
    float sm_scale;
    int mpps, B, M, Hq, Hkv, G, R, NT, KW, SG;   // SG: stages per key group
    int window_left, split_pages, num_splits, page_size, max_seq_len;
    // > 1 (tcgen05 path, one sequence): the num_splits partitions of a (KV
    // head, sequence) form one thread-block cluster and combine their
    // partial results through distributed shared memory, without workspace
    // partials or the reduce kernel
    int cluster;
    // tcgen05 path, several sequences in several partitions, one row tile:
    // the (sequence, partition) slots q = b * num_splits + s longest first
    // (lpt_order_kernel; -1 past the last slot that holds keys); CTA i (in
    // launch order) takes slot lpt_order[i / Hkv] and KV head i % Hkv, so
    // that the last CTAs to start are the shortest.  Null: grid order.
    const int32_t* lpt_order;
    // append (tcgen05 path): the M new tokens of each sequence, bf16
    // [B][M][Hkv][128], are encoded into the cache at positions L - M + m by
    // the CTA whose partition holds them before it loads those pages; null
    // for a plain call
    const uint16_t* k_new;
    const uint16_t* v_new;
    uint8_t* k_cache;
    uint8_t* v_cache;
    int num_pages;
};

// ------------------------------------------------ persistent multi-layer step
// (attention_layers.cu): one launch runs the append + attention of several
// layers, layer after layer.
constexpr int kMaxLayers = 64;          // layers per launch (kernel parameter space)
constexpr int kLayersMaxSplits = 16;    // partitions per (sequence, KV head)

struct LayerDesc {                      // 64-byte aligned by its tensor maps
    CUtensorMap tm_k, tm_v;             // 3-D maps of the layer's caches
    const uint16_t* q;                  // bf16 [B][M][Hq][128]
    const uint16_t* k_new;              // bf16 [B][M][Hkv][128], or null (no append)
    const uint16_t* v_new;
    uint8_t* k_cache;                   // E4M3 [num_pages][Hkv][page_size][128]
    uint8_t* v_cache;
    const int32_t* block_table;         // [B][mpps]
    const int32_t* seq_lens;            // [B]
    const float* k_scale;
    const float* v_scale;
    uint16_t* out;                      // bf16 [B][M][Hq][128]
    float sm_scale;
    int mpps, max_seq_len, num_pages, window_left, split_pages, num_splits;
};

struct LayersParams {
    int n_layers, B, M, Hq, Hkv, G, R, max_splits;
    unsigned* counters;                 // [n_layers][B*Hkv] groups, [n_layers] layers, exit
    uint16_t* part_o;                   // f16 [B*M*Hq][max_splits][128]: partial O / l
    float* part_ml;                     // [B*M*Hq][max_splits][2]: (max, sum)
    LayerDesc layer[kMaxLayers];
};

int launch_attention_layers(const LayersParams& P, int page_size, int grid, cudaStream_t s);
int layers_max_grid();                  // CTAs of the persistent kernel resident at once
int status_attention_layers(unsigned int* s, int clear);

// The cached 3-D tensor map of a [num_pages][Hkv][PS][128] cache (attention.cu).
bool cache_map(CUtensorMap* m, const void* base, bool fp8, int Hkv, int PS, int num_pages);

// Append kernel (insert.cu): the same encoding for the other attention paths.
int launch_append(const void* k, const void* v, const int32_t* seq_lens, const int32_t* block_table, int mpps, int B,
                  int M, int Hkv, const float* k_scale, const float* v_scale, int scale_stride, void* k_cache,
                  void* v_cache,
                  int num_pages, int page_size, bool fp8, cudaStream_t s);

// Host launcher of the tcgen05 kernel (attention_tc.cu).  Returns
// FP8KV_ERR_UNSUPPORTED when the shape is not one it implements.
int launch_attention_tc(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& P, cudaStream_t s);
int status_attention_tc(unsigned int* s, int clear);
int tc_tile_tokens();   // keys per tile of the tcgen05 kernel
int tc_threads();       // threads per CTA of the tcgen05 kernel

}  // namespace fp8kv
