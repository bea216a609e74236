// copy_blocks: bitwise copy of whole physical blocks (every KV head and
// every slot of both caches) for copy-on-write of a shared block ("vLLM
// PagedAttention & continuous batching", sharing with reference counts and
// copy-on-write: allocate a new block and copy that one block).
//
// A block is num_kv_heads * block_size * head_dim contiguous scalars in each
// pool.  Grid: x = pair, y = 16 KiB chunk of the block; each thread moves
// four 16-byte vectors of K and four of V.  HBM-bound (read + write of the
// block), but rare: it runs only when a shared partial block is written.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;
constexpr int kVecsPerCta = kCopyThreads * kCopyUnroll;

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, const int64_t* __restrict__ pairs,
    int64_t vecs_per_block, int32_t num_blocks, int32_t* err) {
    pdl_wait_prerequisites();
    pdl_allow_dependents();
    const int64_t pair = blockIdx.x;
    const int64_t src = __ldg(pairs + 2 * pair);
    const int64_t dst = __ldg(pairs + 2 * pair + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (blockIdx.y == 0 && threadIdx.x == 0) report(err, PKV_DEVERR_BAD_PAIR);
        return;
    }
    const int64_t base = static_cast<int64_t>(blockIdx.y) * kVecsPerCta + threadIdx.x;
    const uint4* ks = k_cache + src * vecs_per_block;
    const uint4* vs = v_cache + src * vecs_per_block;
    uint4* kd = k_cache + dst * vecs_per_block;
    uint4* vd = v_cache + dst * vecs_per_block;
    uint4 kr[kCopyUnroll], vr[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t i = base + u * kCopyThreads;
        if (i < vecs_per_block) {
            kr[u] = ks[i];
            vr[u] = vs[i];
        }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t i = base + u * kCopyThreads;
        if (i < vecs_per_block) {
            kd[i] = kr[u];
            vd[i] = vr[u];
        }
    }
}

}  // namespace

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const pkv_cache_desc& c,
                               const int64_t* pairs, int32_t num_pairs, int32_t* err,
                               cudaStream_t stream) {
    if (num_pairs == 0) return cudaSuccess;
    const int64_t vecs_per_block =
        static_cast<int64_t>(c.num_kv_heads) * c.block_size * row_vectors(c);
    const int64_t chunks = (vecs_per_block + kVecsPerCta - 1) / kVecsPerCta;
    dim3 grid(static_cast<unsigned>(num_pairs), static_cast<unsigned>(chunks));
    return launch_pdl(copy_blocks_kernel, grid, dim3(kCopyThreads), 0, stream,
                      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), pairs,
                      vecs_per_block, c.num_blocks, err);
}

}  // namespace pkv
