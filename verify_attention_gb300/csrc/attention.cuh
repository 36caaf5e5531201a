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
    const float* k_scale;
    const float* v_scale;
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
};

// Host launcher of the tcgen05 kernel (attention_tc.cu).  Returns
// FP8KV_ERR_UNSUPPORTED when the shape is not one it implements.
int launch_attention_tc(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& P, cudaStream_t s);
int status_attention_tc(unsigned int* s, int clear);
int tc_tile_tokens();   // keys per tile of the tcgen05 kernel
int tc_threads();       // threads per CTA of the tcgen05 kernel

}  // namespace fp8kv
