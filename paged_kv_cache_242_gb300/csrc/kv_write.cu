// kv_write: scatter new keys / values into their cache slots through the
// slot mapping (slot = physical block * block_size + offset).  Decode
// writes each sequence's next token into the spare slot of its last block
// (vLLM PagedAttention & continuous batching, "PagedAttention", the
// seven-token example).
//
// One thread moves one 16-byte vector of a (token, KV head) row of K and
// the matching vector of V; rows are head_dim * 2 bytes, contiguous on both
// sides, so loads and stores are fully coalesced.  The kernel is bound by
// launch latency at decode sizes (tens to hundreds of KiB per call).
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256) kv_write_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v,
    const int64_t* __restrict__ slot_mapping, int32_t num_tokens, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, int32_t num_kv_heads, int32_t block_size, int32_t chunks,
    int64_t num_slots, int32_t* err) {
    const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * chunks;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += stride) {
        const int64_t row = idx / chunks;  // token * num_kv_heads + head
        const int32_t c = static_cast<int32_t>(idx - row * chunks);
        const int64_t t = row / num_kv_heads;
        const int32_t h = static_cast<int32_t>(row - t * num_kv_heads);
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;  // padding token
        if (slot >= num_slots) {
            if (h == 0 && c == 0) report(err, PKV_DEVERR_BAD_SLOT);
            continue;
        }
        const int64_t block = slot / block_size;
        const int64_t offset = slot - block * block_size;
        const int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * chunks + c;
        const uint4 kv = __ldg(k + idx);
        const uint4 vv = __ldg(v + idx);
        k_cache[dst] = kv;
        v_cache[dst] = vv;
    }
}

}  // namespace

cudaError_t launch_kv_write(const void* k, const void* v, const int64_t* slot_mapping,
                            int32_t num_tokens, void* k_cache, void* v_cache,
                            const pkv_cache_desc& c, int32_t* err, cudaStream_t stream) {
    const int32_t chunks = c.head_dim / 8;  // 16-byte vectors per row
    const int64_t total = static_cast<int64_t>(num_tokens) * c.num_kv_heads * chunks;
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    const int grid = static_cast<int>(blocks < 152 * 16 ? blocks : 152 * 16);
    kv_write_kernel<<<grid, threads, 0, stream>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping, num_tokens,
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), c.num_kv_heads, c.block_size,
        chunks, static_cast<int64_t>(c.num_blocks) * c.block_size, err);
    return cudaGetLastError();
}

}  // namespace pkv
