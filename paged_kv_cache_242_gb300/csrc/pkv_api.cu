// The C ABI of libpkv.so (declared in include/pkv.h): host-side argument
// validation, TMA descriptor encoding and kernel dispatch.  Nothing here
// allocates device memory or keeps state beyond a cached driver entry point.
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cudaTypedefs.h>

#include "pkv_internal.h"

namespace {

using pkv::kAutoPartition;
using pkv::kHeadDim;

bool aligned(const void* p, uintptr_t bytes) {
    return (reinterpret_cast<uintptr_t>(p) & (bytes - 1)) == 0;
}

bool valid_dtype(pkv_dtype d) { return d == PKV_FP16 || d == PKV_BF16 || d == PKV_FP8_E4M3; }
bool valid_16bit(pkv_dtype d) { return d == PKV_FP16 || d == PKV_BF16; }

// Geometry checks shared by every call (any pool format).
pkv_status check_cache(const pkv_cache_desc& c) {
    if (c.num_blocks <= 0 || c.num_kv_heads <= 0 || c.block_size <= 0 || c.head_dim <= 0 ||
        !valid_dtype(c.dtype))
        return PKV_ERR_INVALID_ARG;
    if ((c.head_dim * pkv::elem_bytes(c.dtype)) % 16 != 0) return PKV_ERR_UNSUPPORTED;  // 16-byte rows
    return PKV_OK;
}

// The calls whose q / k / v / out share the pools' 16-bit type.
pkv_status check_cache_16bit(const pkv_cache_desc& c) {
    pkv_status st = check_cache(c);
    if (st != PKV_OK) return st;
    return valid_16bit(c.dtype) ? PKV_OK : PKV_ERR_INVALID_ARG;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A 4-D view of one pool, {head_dim, block_size, num_kv_heads, num_blocks}
// (innermost first), tiled in boxes of {128 bytes, box_rows, 1, 1} with the
// 128-byte swizzle: one box is one half (64 columns) of box_rows token rows
// of a (block, head) tile of a 16-bit pool, or a whole row of 128 codes of
// an 8-bit pool (box_rows = block_size, or 16 for streamed tiles).
bool encode_pool(CUtensorMap* map, const void* base, const pkv_cache_desc& c, int box_rows) {
    auto encode = tensor_map_encoder();
    if (encode == nullptr) return false;
    const int eb = pkv::elem_bytes(c.dtype);
    const cuuint64_t row = static_cast<cuuint64_t>(c.head_dim) * eb;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(c.head_dim), static_cast<cuuint64_t>(c.block_size),
                          static_cast<cuuint64_t>(c.num_kv_heads),
                          static_cast<cuuint64_t>(c.num_blocks)};
    cuuint64_t strides[3] = {row, row * c.block_size, row * c.block_size * c.num_kv_heads};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / eb), static_cast<cuuint32_t>(box_rows), 1, 1};
    cuuint32_t elem[4] = {1, 1, 1, 1};
    const CUtensorMapDataType type =
        c.dtype == PKV_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
        : c.dtype == PKV_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                              : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = encode(map, type, 4, const_cast<void*>(base), dims, strides, box, elem,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Effective partition size: >= max_seq_len means one pass per sequence.
int32_t effective_partition(int32_t max_seq_len, int32_t block_size, int32_t partition_size) {
    if (max_seq_len < 0 || block_size <= 0 || partition_size < 0) return -1;
    const int64_t single = round_up(max_seq_len > 0 ? max_seq_len : 1, block_size);
    int64_t part;
    if (partition_size == 0) {
        part = max_seq_len > kAutoPartition ? kAutoPartition : single;
        if (part % block_size != 0) part = round_up(part, block_size);
    } else {
        if (partition_size % block_size != 0) return -1;
        part = partition_size;
    }
    if (part >= single) part = single;
    return static_cast<int32_t>(part);
}

int32_t partitions_for(int32_t max_seq_len, int32_t part) {
    const int32_t n = max_seq_len > 0 ? max_seq_len : 1;
    return static_cast<int32_t>((static_cast<int64_t>(n) + part - 1) / part);
}

size_t workspace_for(int32_t num_seqs, int32_t num_q_heads, int32_t max_partitions) {
    if (max_partitions <= 1) return 0;
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * max_partitions;
    return rows * (kHeadDim + 2) * sizeof(float);
}

}  // namespace

extern "C" {

int32_t pkv_abi_version(void) { return 101; }

const char* pkv_status_string(pkv_status status) {
    switch (status) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        case PKV_ERR_WORKSPACE_TOO_SMALL: return "PKV_ERR_WORKSPACE_TOO_SMALL";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    }
    return "PKV_UNKNOWN_STATUS";
}

pkv_status pkv_kv_write(const void* k, const void* v, const int64_t* slot_mapping,
                        int32_t num_tokens, void* k_cache, void* v_cache, pkv_cache_desc c,
                        int32_t* err_flag, void* stream) {
    pkv_status st = check_cache_16bit(c);
    if (st != PKV_OK) return st;
    if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8))
        return PKV_ERR_INVALID_ARG;
    cudaError_t e = pkv::launch_kv_write(k, v, slot_mapping, num_tokens, k_cache, v_cache, c,
                                         err_flag, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int32_t pkv_decode_partition_size(int32_t max_seq_len, int32_t block_size, int32_t partition_size) {
    return effective_partition(max_seq_len, block_size, partition_size);
}

size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                  int32_t max_seq_len, int32_t block_size,
                                  int32_t partition_size) {
    (void)head_dim;
    if (num_seqs <= 0 || num_q_heads <= 0) return 0;
    const int32_t part = effective_partition(max_seq_len, block_size, partition_size);
    if (part <= 0) return 0;
    size_t need = workspace_for(num_seqs, num_q_heads, partitions_for(max_seq_len, part));
    // automatic mode streams when the shape allows it (the group size is not
    // known here, so size for the larger of the two layouts)
    if (partition_size == 0 && pkv::stream_supported(num_seqs, 1, block_size)) {
        const size_t stream = pkv::stream_workspace_bytes(num_seqs, num_q_heads, 0);
        if (stream > need) need = stream;
    }
    return need;
}

pkv_status pkv_paged_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* seq_lens, int32_t max_seq_len,
                                      int32_t num_seqs, int32_t num_q_heads, pkv_cache_desc c,
                                      float scale, int32_t partition_size, void* workspace,
                                      size_t workspace_bytes, void* out, int32_t* err_flag,
                                      void* stream) {
    pkv_status st = check_cache_16bit(c);
    if (st != PKV_OK) return st;
    if (num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0 ||
        partition_size < 0 || !std::isfinite(scale))
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % c.num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks_per_seq) * c.block_size)
        return PKV_ERR_INVALID_ARG;
    if (partition_size > 0 && partition_size % c.block_size != 0) return PKV_ERR_INVALID_ARG;
    const bool block_ok = c.block_size == 8 || c.block_size == 16 || c.block_size == 32 ||
                          c.block_size == 64 || c.block_size == 128;
    if (c.head_dim != kHeadDim || !block_ok || num_q_heads / c.num_kv_heads > 64 ||
        num_seqs > 65535 || c.num_kv_heads > 65535)
        return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !out) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 4) || !aligned(out, 4) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PKV_ERR_INVALID_ARG;

    const int32_t group = num_q_heads / c.num_kv_heads;
    const bool streaming =
        partition_size == 0 && pkv::stream_supported(num_seqs, group, c.block_size);
    // the partition kernel stages whole blocks of 16 or 32 rows
    if (!streaming && c.block_size != 16 && c.block_size != 32) return PKV_ERR_UNSUPPORTED;
    const int32_t part = effective_partition(max_seq_len, c.block_size, partition_size);
    const int32_t max_parts = partitions_for(max_seq_len, part);
    const size_t need = streaming ? pkv::stream_workspace_bytes(num_seqs, num_q_heads, c.num_kv_heads)
                                  : workspace_for(num_seqs, num_q_heads, max_parts);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need))
        return PKV_ERR_WORKSPACE_TOO_SMALL;
    if (need > 0 && !aligned(workspace, 16)) return PKV_ERR_INVALID_ARG;

    CUtensorMap k_map, v_map;
    const int box_rows =
        streaming ? (c.block_size < pkv::kTileTokens ? c.block_size : pkv::kTileTokens)
                  : c.block_size;
    if (!encode_pool(&k_map, k_cache, c, box_rows) || !encode_pool(&v_map, v_cache, c, box_rows))
        return PKV_ERR_CUDA;

    pkv::DecodeArgs a{};
    a.q = q;
    a.out = out;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    if (streaming) {
        a.ws_acc = static_cast<float*>(workspace);  // laid out by the stream launcher
    } else if (need > 0) {
        const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * max_parts;
        float* ws = static_cast<float*>(workspace);
        a.ws_acc = ws;
        a.ws_m = ws + rows * kHeadDim;
        a.ws_l = a.ws_m + rows;
    }
    a.err = err_flag;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = c.num_kv_heads;
    a.group = group;
    a.num_blocks = c.num_blocks;
    a.partition_size = part;
    a.max_partitions = max_parts;
    a.max_seq_len = max_seq_len;
    a.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
    a.v_scale = 1.f;
    cudaError_t e =
        streaming ? pkv::launch_paged_decode_stream(k_map, v_map, a, c.dtype, c.block_size,
                                                    static_cast<cudaStream_t>(stream))
                  : pkv::launch_paged_decode(k_map, v_map, a, c.dtype, c.block_size,
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, pkv_cache_desc c,
                           const int64_t* src_dst_pairs, int32_t num_pairs, int32_t* err_flag,
                           void* stream) {
    pkv_status st = check_cache(c);
    if (st != PKV_OK) return st;
    if (num_pairs < 0) return PKV_ERR_INVALID_ARG;
    if (num_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !src_dst_pairs) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(src_dst_pairs, 8))
        return PKV_ERR_INVALID_ARG;
    const int64_t vecs = static_cast<int64_t>(c.num_kv_heads) * c.block_size * pkv::row_vectors(c);
    if ((vecs + 1023) / 1024 > 65535) return PKV_ERR_UNSUPPORTED;
    cudaError_t e = pkv::launch_copy_blocks(k_cache, v_cache, c, src_dst_pairs, num_pairs,
                                            err_flag, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_paged_prefill_attention(const void* q, const int32_t* cu_seqlens_q,
                                       int32_t max_q_len, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, int32_t max_seq_len,
                                       int32_t num_seqs, int32_t num_q_heads, pkv_cache_desc c,
                                       float scale, void* out, int32_t* err_flag, void* stream) {
    pkv_status st = check_cache_16bit(c);
    if (st != PKV_OK) return st;
    if (num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0 ||
        max_q_len < 0 || !std::isfinite(scale))
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % c.num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks_per_seq) * c.block_size)
        return PKV_ERR_INVALID_ARG;
    const bool block_ok = c.block_size == 8 || c.block_size == 16 || c.block_size == 32 ||
                          c.block_size == 64 || c.block_size == 128;
    if (c.head_dim != kHeadDim || !block_ok || num_q_heads / c.num_kv_heads > 64 ||
        num_seqs > 65535 || c.num_kv_heads > 65535)
        return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0 || max_q_len == 0) return PKV_OK;
    if (!q || !cu_seqlens_q || !k_cache || !v_cache || !block_tables || !seq_lens || !out)
        return PKV_ERR_INVALID_ARG;
    // q and out rows move as 16-byte vectors
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4) || !aligned(cu_seqlens_q, 4))
        return PKV_ERR_INVALID_ARG;
    const int64_t row_tiles =
        (static_cast<int64_t>(max_q_len) * (num_q_heads / c.num_kv_heads) + 15) / 16;
    if (row_tiles > 0x7fffffff) return PKV_ERR_UNSUPPORTED;
    const bool tensor_cores = pkv::prefill_tc_supported(num_q_heads / c.num_kv_heads);
    CUtensorMap k_map, v_map;
    const int box_rows =
        tensor_cores ? pkv::prefill_tc_box_rows(c.block_size)
                     : (c.block_size < pkv::kTileTokens ? c.block_size : pkv::kTileTokens);
    if (!encode_pool(&k_map, k_cache, c, box_rows) || !encode_pool(&v_map, v_cache, c, box_rows))
        return PKV_ERR_CUDA;
    pkv::PrefillArgs a{};
    a.q = q;
    a.out = out;
    a.cu_q = cu_seqlens_q;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.err = err_flag;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = c.num_kv_heads;
    a.group = num_q_heads / c.num_kv_heads;
    a.num_blocks = c.num_blocks;
    a.max_seq_len = max_seq_len;
    a.max_q_len = max_q_len;
    a.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
    cudaError_t e =
        tensor_cores
            ? pkv::launch_paged_prefill_tc(k_map, v_map, a, c.dtype, c.block_size,
                                           static_cast<cudaStream_t>(stream))
            : pkv::launch_paged_prefill(k_map, v_map, a, c.dtype, c.block_size,
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_kv_write_fp8(const void* k, const void* v, pkv_dtype kv_dtype,
                            const int64_t* slot_mapping, int32_t num_tokens, void* k_cache,
                            void* v_cache, pkv_cache_desc c, float k_scale, float v_scale,
                            int32_t* err_flag, void* stream) {
    pkv_status st = check_cache(c);
    if (st != PKV_OK) return st;
    if (c.dtype != PKV_FP8_E4M3 || !valid_16bit(kv_dtype) || num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (!std::isfinite(k_scale) || !std::isfinite(v_scale) || !(k_scale > 0.f) || !(v_scale > 0.f))
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8))
        return PKV_ERR_INVALID_ARG;
    cudaError_t e = pkv::launch_kv_write_fp8(k, v, kv_dtype, slot_mapping, num_tokens, k_cache,
                                             v_cache, c, k_scale, v_scale, err_flag,
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_paged_decode_attention_fp8(const void* q, pkv_dtype q_dtype, const void* k_cache,
                                          const void* v_cache, const int32_t* block_tables,
                                          int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                          int32_t max_seq_len, int32_t num_seqs,
                                          int32_t num_q_heads, pkv_cache_desc c, float scale,
                                          float k_scale, float v_scale, void* workspace,
                                          size_t workspace_bytes, void* out, int32_t* err_flag,
                                          void* stream) {
    pkv_status st = check_cache(c);
    if (st != PKV_OK) return st;
    if (c.dtype != PKV_FP8_E4M3 || !valid_16bit(q_dtype)) return PKV_ERR_INVALID_ARG;
    if (num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0 ||
        !std::isfinite(scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale) ||
        !(k_scale > 0.f) || !(v_scale > 0.f))
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % c.num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks_per_seq) * c.block_size)
        return PKV_ERR_INVALID_ARG;
    const float scale_log2 = scale * k_scale * 1.4426950408889634f;  // log2(e)
    if (!std::isfinite(scale_log2)) return PKV_ERR_INVALID_ARG;
    const int32_t group = num_q_heads / c.num_kv_heads;
    if (c.head_dim != kHeadDim || c.num_kv_heads > 65535 ||
        !pkv::stream_supported(num_seqs > 0 ? num_seqs : 1, group, c.block_size))
        return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !out) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 8) || !aligned(out, 8) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PKV_ERR_INVALID_ARG;
    const size_t need = pkv::stream_workspace_bytes(num_seqs, num_q_heads, c.num_kv_heads);
    if (workspace == nullptr || workspace_bytes < need) return PKV_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 16)) return PKV_ERR_INVALID_ARG;

    CUtensorMap k_map, v_map;
    const int box_rows = c.block_size < pkv::kTileTokensFp8 ? c.block_size : pkv::kTileTokensFp8;
    if (!encode_pool(&k_map, k_cache, c, box_rows) || !encode_pool(&v_map, v_cache, c, box_rows))
        return PKV_ERR_CUDA;
    pkv::DecodeArgs a{};
    a.q = q;
    a.out = out;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.ws_acc = static_cast<float*>(workspace);  // laid out by the stream launcher
    a.err = err_flag;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = c.num_kv_heads;
    a.group = group;
    a.num_blocks = c.num_blocks;
    a.partition_size = 0;
    a.max_partitions = 1;
    a.max_seq_len = max_seq_len;
    a.scale_log2 = scale_log2;
    a.v_scale = v_scale;
    cudaError_t e = pkv::launch_paged_decode_stream_fp8(k_map, v_map, a, q_dtype, c.block_size,
                                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Address a kernel can use for a pool: device or managed memory as is,
// page-locked host memory through its device mapping; null otherwise.
static const void* device_address(const void* p) {
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();  // do not leave the query's error for the next launch check
        return nullptr;
    }
    switch (attr.type) {
        case cudaMemoryTypeDevice:
        case cudaMemoryTypeManaged:
            return p;
        case cudaMemoryTypeHost:
            return attr.devicePointer;
        default:
            return nullptr;
    }
}

pkv_status pkv_swap_blocks(const void* src_k, const void* src_v, int32_t src_num_blocks,
                           void* dst_k, void* dst_v, int32_t dst_num_blocks, pkv_cache_desc c,
                           const int64_t* src_dst_pairs, int32_t num_pairs, int32_t* err_flag,
                           void* stream) {
    pkv_cache_desc geometry = c;
    geometry.num_blocks = 1;  // not used: the two pools carry their own sizes
    pkv_status st = check_cache(geometry);
    if (st != PKV_OK) return st;
    if (num_pairs < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (num_pairs == 0) return PKV_OK;
    if (!src_k || !src_v || !dst_k || !dst_v || !src_dst_pairs || !aligned(src_dst_pairs, 8))
        return PKV_ERR_INVALID_ARG;
    if (pkv::block_copy_chunks(geometry) > 65535) return PKV_ERR_UNSUPPORTED;
    const void* sk = device_address(src_k);
    const void* sv = device_address(src_v);
    void* dk = const_cast<void*>(device_address(dst_k));
    void* dv = const_cast<void*>(device_address(dst_v));
    if (!sk || !sv || !dk || !dv) return PKV_ERR_INVALID_ARG;
    if (!aligned(sk, 16) || !aligned(sv, 16) || !aligned(dk, 16) || !aligned(dv, 16))
        return PKV_ERR_INVALID_ARG;
    cudaError_t e = pkv::launch_transfer_blocks(sk, sv, src_num_blocks, dk, dv, dst_num_blocks,
                                                geometry, src_dst_pairs, num_pairs, err_flag,
                                                static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_kv_write_layers(const void* const* k, const void* const* v,
                               const int64_t* slot_mapping, int32_t num_tokens,
                               void* const* k_caches, void* const* v_caches, int32_t num_layers,
                               pkv_cache_desc c, int32_t* err_flag, void* stream) {
    pkv_status st = check_cache_16bit(c);
    if (st != PKV_OK) return st;
    if (num_tokens < 0 || num_layers < 1 || num_layers > PKV_MAX_LAYERS) return PKV_ERR_INVALID_ARG;
    if (!k || !v || !k_caches || !v_caches) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!slot_mapping || !aligned(slot_mapping, 8)) return PKV_ERR_INVALID_ARG;
    for (int l = 0; l < num_layers; ++l) {
        if (!k[l] || !v[l] || !k_caches[l] || !v_caches[l]) return PKV_ERR_INVALID_ARG;
        if (!aligned(k[l], 16) || !aligned(v[l], 16) || !aligned(k_caches[l], 16) ||
            !aligned(v_caches[l], 16))
            return PKV_ERR_INVALID_ARG;
    }
    cudaError_t e = pkv::launch_kv_write_layers(k, v, slot_mapping, num_tokens, k_caches, v_caches,
                                                num_layers, c, err_flag,
                                                static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_copy_blocks_layers(void* const* k_caches, void* const* v_caches,
                                  int32_t num_layers, pkv_cache_desc c,
                                  const int64_t* src_dst_pairs, int32_t num_pairs,
                                  int32_t* err_flag, void* stream) {
    pkv_status st = check_cache(c);
    if (st != PKV_OK) return st;
    if (num_pairs < 0 || num_layers < 1 || num_layers > PKV_MAX_LAYERS) return PKV_ERR_INVALID_ARG;
    if (!k_caches || !v_caches) return PKV_ERR_INVALID_ARG;
    if (num_pairs == 0) return PKV_OK;
    if (!src_dst_pairs || !aligned(src_dst_pairs, 8)) return PKV_ERR_INVALID_ARG;
    for (int l = 0; l < num_layers; ++l) {
        if (!k_caches[l] || !v_caches[l] || !aligned(k_caches[l], 16) || !aligned(v_caches[l], 16))
            return PKV_ERR_INVALID_ARG;
    }
    if (pkv::block_copy_chunks(c) > 65535) return PKV_ERR_UNSUPPORTED;
    cudaError_t e = pkv::launch_copy_blocks_layers(k_caches, v_caches, num_layers, c,
                                                   src_dst_pairs, num_pairs, err_flag,
                                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // extern "C"
