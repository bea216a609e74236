// Host-side launch interfaces shared by the C ABI and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "pkv.h"

namespace pkv {

constexpr int kHeadDim = 128;        // head size the attention kernels implement
constexpr int kConsumerWarps = 4;    // warps that compute on staged K/V tiles
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;  // + one TMA producer warp
constexpr int kAutoPartition = 512;  // tokens per partition in automatic split mode

// Bytes of one stored scalar of a pool, and 16-byte vectors per (token, head) row.
inline int elem_bytes(pkv_dtype d) { return d == PKV_FP8_E4M3 ? 1 : 2; }
inline int32_t row_vectors(const pkv_cache_desc& c) { return c.head_dim * elem_bytes(c.dtype) / 16; }

// Launch `kernel` on `stream` with programmatic stream serialisation allowed
// (the kernel waits for its prerequisites itself, see pkv_device.cuh).
template <typename... KernelArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KernelArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raise kKernel's dynamic shared-memory limit to at least `bytes` on the
// current device; the limit reached is remembered per (kernel, device), so
// later calls skip the driver.
template <auto kKernel>
cudaError_t ensure_smem_limit(size_t bytes) {
    constexpr int kMaxDevices = 64;
    static std::atomic<size_t> configured[kMaxDevices];
    int device = 0;
    cudaError_t err = cudaGetDevice(&device);
    if (err != cudaSuccess) return err;
    if (device >= 0 && device < kMaxDevices &&
        configured[device].load(std::memory_order_relaxed) >= bytes)
        return cudaSuccess;
    err = cudaFuncSetAttribute(kKernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(bytes));
    if (err == cudaSuccess && device >= 0 && device < kMaxDevices) {
        size_t cur = configured[device].load(std::memory_order_relaxed);
        while (cur < bytes && !configured[device].compare_exchange_weak(cur, bytes)) {
        }
    }
    return err;
}

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
    float scale_log2;           // softmax scale * log2(e) (* k_scale for 8-bit pools)
    int32_t num_warps;          // stream mode: warps in the grid
    float v_scale;              // 8-bit pools: value scale (1 otherwise)
};

#ifndef PKV_STREAM_WARPS
#define PKV_STREAM_WARPS 7
#endif
#ifndef PKV_STREAM_STAGES
#define PKV_STREAM_STAGES 2
#endif
#ifndef PKV_STREAM_WARPS_FP8
#define PKV_STREAM_WARPS_FP8 8
#endif
#ifndef PKV_STREAM_WARPS_FP8_COLS
#define PKV_STREAM_WARPS_FP8_COLS 8
#endif
#ifndef PKV_STREAM_TILES_PER_WARP
#define PKV_STREAM_TILES_PER_WARP 4
#endif
#ifndef PKV_STREAM_STAGES_FP8
#define PKV_STREAM_STAGES_FP8 2
#endif
#ifndef PKV_TILE_TOKENS_FP8
#define PKV_TILE_TOKENS_FP8 32
#endif
#ifndef PKV_FP8_SPLIT_P
#define PKV_FP8_SPLIT_P 0
#endif
constexpr int kStreamWarps = PKV_STREAM_WARPS;    // warps per CTA of the streaming kernel
constexpr int kStreamStages = PKV_STREAM_STAGES;  // 8 KiB stages per warp
// Over 8-bit pools: warps per CTA, tokens per streamed tile, stages per warp
// (tile tokens x 256 bytes each), and whether P is split into two binary16
// parts (binary16 P already carries 11 bits).
constexpr int kStreamWarpsFp8 = PKV_STREAM_WARPS_FP8;          // groups of 9..16 heads
constexpr int kStreamWarpsFp8Cols = PKV_STREAM_WARPS_FP8_COLS;  // groups of up to 8 heads
constexpr int kTileTokensFp8 = PKV_TILE_TOKENS_FP8;
constexpr int kStreamStagesFp8 = PKV_STREAM_STAGES_FP8;
constexpr bool kFp8SplitP = PKV_FP8_SPLIT_P != 0;
constexpr int kStreamMaxWarps =
    (kStreamWarps > kStreamWarpsFp8 ? kStreamWarps : kStreamWarpsFp8) > kStreamWarpsFp8Cols
        ? (kStreamWarps > kStreamWarpsFp8 ? kStreamWarps : kStreamWarpsFp8)
        : kStreamWarpsFp8Cols;
// target tiles per warp when the grid need not fill every SM
constexpr int kStreamTilesPerWarp = PKV_STREAM_TILES_PER_WARP;
constexpr int kStreamMaxCtas = 160;     // cap of its grid (one CTA per SM)
constexpr int kStreamMaxSeqs = 4096;    // sequences whose prefix fits shared memory
constexpr int kTileTokens = 16;         // tokens per streamed tile (16-bit pools)

// Streaming mode: every warp of a persistent grid takes an equal share of
// all 16-token tiles in (sequence, KV head, tile) order; shares that cut a
// (sequence, head) segment leave partial statistics for the merge kernel.
bool stream_supported(int num_seqs, int group, int block_size);
size_t stream_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads_or_0);
cudaError_t launch_paged_decode_stream(const CUtensorMap& k_map16, const CUtensorMap& v_map16,
                                       DecodeArgs args, pkv_dtype dtype, int block_size,
                                       cudaStream_t stream);
// The same over 8-bit (E4M3) pools; q_dtype is the type of q and out, the
// maps view the pools as bytes (one 128-byte box per 16 token rows).
cudaError_t launch_paged_decode_stream_fp8(const CUtensorMap& k_map8, const CUtensorMap& v_map8,
                                           DecodeArgs args, pkv_dtype q_dtype, int block_size,
                                           cudaStream_t stream);

// Launch the split (or single-pass, when max_partitions == 1) decode
// kernel and, in split mode, the merge kernel.
cudaError_t launch_paged_decode(const CUtensorMap& k_map, const CUtensorMap& v_map,
                                const DecodeArgs& args, pkv_dtype dtype, int block_size,
                                cudaStream_t stream);

struct PrefillArgs {
    const void* q;                // [total query tokens][Hq][128]
    void* out;                    // [total query tokens][Hq][128]
    const int32_t* cu_q;          // [S + 1] query-token offsets
    const int32_t* block_tables;  // [S][max_blocks_per_seq]
    const int32_t* seq_lens;      // [S] cached tokens, queries included
    int32_t* err;                 // nullable
    int32_t max_blocks_per_seq;
    int32_t num_seqs;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t group;
    int32_t num_blocks;
    int32_t max_seq_len;
    int32_t max_q_len;
    float scale_log2;
};

cudaError_t launch_paged_prefill(const CUtensorMap& k_map16, const CUtensorMap& v_map16,
                                 const PrefillArgs& args, pkv_dtype dtype, int block_size,
                                 cudaStream_t stream);

// The tcgen05 prefill kernel (groups dividing 128); its pool maps use boxes
// of prefill_tc_box_rows(block_size) token rows.
bool prefill_tc_supported(int group);
int prefill_tc_box_rows(int block_size);
cudaError_t launch_paged_prefill_tc(const CUtensorMap& k_map, const CUtensorMap& v_map,
                                    const PrefillArgs& args, pkv_dtype dtype, int block_size,
                                    cudaStream_t stream);

cudaError_t launch_kv_write(const void* k, const void* v, const int64_t* slot_mapping,
                            int32_t num_tokens, void* k_cache, void* v_cache,
                            const pkv_cache_desc& c, int32_t* err, cudaStream_t stream);

cudaError_t launch_kv_write_fp8(const void* k, const void* v, pkv_dtype kv_dtype,
                                const int64_t* slot_mapping, int32_t num_tokens, void* k_cache,
                                void* v_cache, const pkv_cache_desc& c, float k_scale,
                                float v_scale, int32_t* err, cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const pkv_cache_desc& c,
                               const int64_t* pairs, int32_t num_pairs, int32_t* err,
                               cudaStream_t stream);

constexpr int kMaxLayers = PKV_MAX_LAYERS;

// 16 KiB chunks per block of one pool (the grid's y extent for block copies).
int64_t block_copy_chunks(const pkv_cache_desc& c);

cudaError_t launch_transfer_blocks(const void* src_k, const void* src_v, int32_t src_blocks,
                                   void* dst_k, void* dst_v, int32_t dst_blocks,
                                   const pkv_cache_desc& c, const int64_t* pairs,
                                   int32_t num_pairs, int32_t* err, cudaStream_t stream);

cudaError_t launch_copy_blocks_layers(void* const* k_caches, void* const* v_caches,
                                      int32_t num_layers, const pkv_cache_desc& c,
                                      const int64_t* pairs, int32_t num_pairs, int32_t* err,
                                      cudaStream_t stream);

cudaError_t launch_kv_write_layers(const void* const* k, const void* const* v,
                                   const int64_t* slot_mapping, int32_t num_tokens,
                                   void* const* k_caches, void* const* v_caches, int32_t num_layers,
                                   const pkv_cache_desc& c, int32_t* err, cudaStream_t stream);

}  // namespace pkv
