// Host-side launch interfaces shared by the C ABI and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

constexpr int kHeadDim = 128;        // head size the attention kernels implement
constexpr int kConsumerWarps = 4;    // warps that compute on staged K/V tiles
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;  // + one TMA producer warp
constexpr int kAutoPartition = 512;  // tokens per partition in automatic split mode

struct DecodeArgs {
    const void* q;              // [S][Hq][128]
    void* out;                  // [S][Hq][128]
    const int32_t* block_tables;  // [S][max_blocks_per_seq]
    const int32_t* seq_lens;    // [S]
    float* ws_acc;              // [S][Hq][max_partitions][128]   (split mode)
    float* ws_m;                // [S][Hq][max_partitions]  running max, log2 units
    float* ws_l;                // [S][Hq][max_partitions]  running sum
    int32_t* err;               // nullable
    int32_t max_blocks_per_seq;
    int32_t num_seqs;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t group;              // num_q_heads / num_kv_heads
    int32_t num_blocks;
    int32_t partition_size;     // tokens per partition (multiple of block size)
    int32_t max_partitions;     // ceil(max_seq_len / partition_size), >= 1
    int32_t max_seq_len;
    float scale_log2;           // softmax scale * log2(e)
};

// Launch the split (or single-pass, when max_partitions == 1) decode
// kernel and, in split mode, the merge kernel.
cudaError_t launch_paged_decode(const CUtensorMap& k_map, const CUtensorMap& v_map,
                                const DecodeArgs& args, pkv_dtype dtype, int block_size,
                                cudaStream_t stream);

cudaError_t launch_kv_write(const void* k, const void* v, const int64_t* slot_mapping,
                            int32_t num_tokens, void* k_cache, void* v_cache,
                            const pkv_cache_desc& c, int32_t* err, cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const pkv_cache_desc& c,
                               const int64_t* pairs, int32_t num_pairs, int32_t* err,
                               cudaStream_t stream);

}  // namespace pkv
