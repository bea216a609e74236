// Streaming paged decode attention over 16-bit pools (the kernel template
// is in decode_stream.cuh), and the host-side shape and workspace rules shared
// with the 8-bit instantiation.
#include "decode_stream.cuh"

namespace pkv {

bool stream_supported(int num_seqs, int group, int block_size) {
    return num_seqs >= 1 && num_seqs <= kStreamMaxSeqs && group >= 1 && group <= 16 &&
           (block_size == 8 || block_size == 16 || block_size == 32 || block_size == 64 ||
            block_size == 128) &&
           stream_smem_bytes<false, kStreamWarps>(num_seqs) <= 232448 &&
           stream_smem_bytes<true, kStreamWarpsFp8>(num_seqs) <= 232448 &&
           stream_smem_bytes<true, kStreamWarpsFp8Cols>(num_seqs) <= 232448;
}

// Rows of partial statistics: one per (partial id, query head of the group);
// partial ids are (warp + segment) < warps + S * H_kv.  Without H_kv the
// group is bounded by min(16, H_q).
size_t stream_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads_or_0) {
    const size_t warps = static_cast<size_t>(kStreamMaxCtas) * kStreamMaxWarps;
    size_t rows;
    if (num_kv_heads_or_0 > 0) {
        const size_t g = static_cast<size_t>(num_q_heads / num_kv_heads_or_0);
        rows = (warps + static_cast<size_t>(num_seqs) * num_kv_heads_or_0) * g;
    } else {
        const size_t gmax = static_cast<size_t>(num_q_heads < 16 ? num_q_heads : 16);
        rows = warps * gmax + static_cast<size_t>(num_seqs) * num_q_heads;
    }
    const size_t floats = rows * (kHeadDim + 2);
    return floats * sizeof(float);
}

cudaError_t launch_paged_decode_stream(const CUtensorMap& k_map16, const CUtensorMap& v_map16,
                                       DecodeArgs a, pkv_dtype dtype, int block_size,
                                       cudaStream_t stream) {
    return launch_stream<Rows16Policy>(k_map16, v_map16, a, dtype, block_size, stream);
}

}  // namespace pkv
