// Streaming paged decode attention over 8-bit (E4M3) pools: the kernel of
// decode_stream.cuh with the transposed policy for groups of up to 8 query
// heads and the row policy for larger groups (decode_policy.cuh).
#include "decode_stream.cuh"

namespace pkv {

cudaError_t launch_paged_decode_stream_fp8(const CUtensorMap& k_map8, const CUtensorMap& v_map8,
                                           DecodeArgs a, pkv_dtype q_dtype, int block_size,
                                           cudaStream_t stream) {
    // groups of up to 8 query heads fit the transposed form's 8 MMA columns
    return a.group <= 8
               ? launch_stream<E4m3ColsPolicy>(k_map8, v_map8, a, q_dtype, block_size, stream)
               : launch_stream<E4m3RowsPolicy>(k_map8, v_map8, a, q_dtype, block_size, stream);
}

}  // namespace pkv
