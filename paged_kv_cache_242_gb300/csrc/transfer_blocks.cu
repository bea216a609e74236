// Block transfers beyond a single pool:
//
//  * transfer_blocks_kernel: whole-block copies from one pair of pools to
//    another, the swap path of preemption ("vLLM PagedAttention & continuous
//    batching", "Preemption when blocks run out": Swap copies the evicted
//    blocks to CPU memory managed by a second block allocator and back when
//    the sequence resumes).  Either pool may be page-locked host memory: on
//    GB300 the kernel reads and writes it directly over the CPU-GPU link, so
//    a swap of many small blocks is one launch, not one transfer per block.
//  * copy_blocks_layers_kernel / kv_write_layers_kernel: copy-on-write copies
//    and slot writes applied to every layer's caches in one launch (a model
//    keeps one pair of pools per layer, all sharing the block tables).
//
// Work split: one CTA per (pair or token group, 16 KiB chunk, layer); each
// thread moves 16-byte vectors.  All three are bound by memory bandwidth
// (HBM, or the CPU-GPU link for host pools).
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;
constexpr int kVecsPerCta = kThreads * kUnroll;

// Copy vectors [base, base + kVecsPerCta) of one block (strided by threads).
__device__ __forceinline__ void copy_chunk(const uint4* __restrict__ ks, const uint4* __restrict__ vs,
                                           uint4* __restrict__ kd, uint4* __restrict__ vd,
                                           int64_t base, int64_t vecs_per_block) {
    uint4 kr[kUnroll], vr[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = base + u * kThreads;
        if (i < vecs_per_block) {
            kr[u] = ks[i];
            vr[u] = vs[i];
        }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = base + u * kThreads;
        if (i < vecs_per_block) {
            kd[i] = kr[u];
            vd[i] = vr[u];
        }
    }
}

__global__ void __launch_bounds__(kThreads) transfer_blocks_kernel(
    const uint4* __restrict__ src_k, const uint4* __restrict__ src_v, int32_t src_blocks,
    uint4* __restrict__ dst_k, uint4* __restrict__ dst_v, int32_t dst_blocks,
    const int64_t* __restrict__ pairs, int64_t vecs_per_block, int32_t* err) {
    pdl_wait_prerequisites();
    pdl_allow_dependents();
    const int64_t pair = blockIdx.x;
    const int64_t src = __ldg(pairs + 2 * pair);
    const int64_t dst = __ldg(pairs + 2 * pair + 1);
    if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
        if (blockIdx.y == 0 && threadIdx.x == 0) report(err, PKV_DEVERR_BAD_PAIR);
        return;
    }
    copy_chunk(src_k + src * vecs_per_block, src_v + src * vecs_per_block,
               dst_k + dst * vecs_per_block, dst_v + dst * vecs_per_block,
               static_cast<int64_t>(blockIdx.y) * kVecsPerCta + threadIdx.x, vecs_per_block);
}

struct LayerCaches {
    uint4* k[kMaxLayers];
    uint4* v[kMaxLayers];
};

__global__ void __launch_bounds__(kThreads) copy_blocks_layers_kernel(
    const __grid_constant__ LayerCaches caches, const int64_t* __restrict__ pairs,
    int64_t vecs_per_block, int32_t num_blocks, int32_t* err) {
    pdl_wait_prerequisites();
    pdl_allow_dependents();
    const int64_t pair = blockIdx.x;
    const int layer = blockIdx.z;
    const int64_t src = __ldg(pairs + 2 * pair);
    const int64_t dst = __ldg(pairs + 2 * pair + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (blockIdx.y == 0 && layer == 0 && threadIdx.x == 0) report(err, PKV_DEVERR_BAD_PAIR);
        return;
    }
    uint4* k = caches.k[layer];
    uint4* v = caches.v[layer];
    copy_chunk(k + src * vecs_per_block, v + src * vecs_per_block, k + dst * vecs_per_block,
               v + dst * vecs_per_block, static_cast<int64_t>(blockIdx.y) * kVecsPerCta + threadIdx.x,
               vecs_per_block);
}

struct LayerTokens {
    const uint4* k[kMaxLayers];
    const uint4* v[kMaxLayers];
};

// One thread per 16-byte vector of a (token, KV head) row, per layer (grid z).
__global__ void __launch_bounds__(kThreads) kv_write_layers_kernel(
    const __grid_constant__ LayerTokens tokens, const __grid_constant__ LayerCaches caches,
    const int64_t* __restrict__ slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
    int32_t block_size, int32_t chunks, int64_t num_slots, int32_t* err) {
    pdl_wait_prerequisites();
    pdl_allow_dependents();
    const int layer = blockIdx.z;
    const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * chunks;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const uint4* k = tokens.k[layer];
    const uint4* v = tokens.v[layer];
    uint4* kc = caches.k[layer];
    uint4* vc = caches.v[layer];
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += stride) {
        const int64_t row = idx / chunks;
        const int32_t c = static_cast<int32_t>(idx - row * chunks);
        const int64_t t = row / num_kv_heads;
        const int32_t h = static_cast<int32_t>(row - t * num_kv_heads);
        const uint4 kv = __ldg(k + idx);
        const uint4 vv = __ldg(v + idx);
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (h == 0 && c == 0 && layer == 0) report(err, PKV_DEVERR_BAD_SLOT);
            continue;
        }
        const int64_t block = slot / block_size;
        const int64_t offset = slot - block * block_size;
        const int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * chunks + c;
        kc[dst] = kv;
        vc[dst] = vv;
    }
}

int64_t chunks_of(const pkv_cache_desc& c) {
    const int64_t vecs = static_cast<int64_t>(c.num_kv_heads) * c.block_size * row_vectors(c);
    return (vecs + kVecsPerCta - 1) / kVecsPerCta;
}

}  // namespace

int64_t block_copy_chunks(const pkv_cache_desc& c) { return chunks_of(c); }

cudaError_t launch_transfer_blocks(const void* src_k, const void* src_v, int32_t src_blocks,
                                   void* dst_k, void* dst_v, int32_t dst_blocks,
                                   const pkv_cache_desc& c, const int64_t* pairs,
                                   int32_t num_pairs, int32_t* err, cudaStream_t stream) {
    if (num_pairs == 0) return cudaSuccess;
    const int64_t vecs = static_cast<int64_t>(c.num_kv_heads) * c.block_size * row_vectors(c);
    return launch_pdl(transfer_blocks_kernel,
                      dim3(static_cast<unsigned>(num_pairs), static_cast<unsigned>(chunks_of(c))),
                      dim3(kThreads), 0, stream, static_cast<const uint4*>(src_k),
                      static_cast<const uint4*>(src_v), src_blocks, static_cast<uint4*>(dst_k),
                      static_cast<uint4*>(dst_v), dst_blocks, pairs, vecs, err);
}

cudaError_t launch_copy_blocks_layers(void* const* k_caches, void* const* v_caches,
                                      int32_t num_layers, const pkv_cache_desc& c,
                                      const int64_t* pairs, int32_t num_pairs, int32_t* err,
                                      cudaStream_t stream) {
    if (num_pairs == 0 || num_layers == 0) return cudaSuccess;
    LayerCaches caches{};
    for (int l = 0; l < num_layers; ++l) {
        caches.k[l] = static_cast<uint4*>(k_caches[l]);
        caches.v[l] = static_cast<uint4*>(v_caches[l]);
    }
    const int64_t vecs = static_cast<int64_t>(c.num_kv_heads) * c.block_size * row_vectors(c);
    return launch_pdl(copy_blocks_layers_kernel,
                      dim3(static_cast<unsigned>(num_pairs), static_cast<unsigned>(chunks_of(c)),
                           static_cast<unsigned>(num_layers)),
                      dim3(kThreads), 0, stream, caches, pairs, vecs, c.num_blocks, err);
}

cudaError_t launch_kv_write_layers(const void* const* k, const void* const* v,
                                   const int64_t* slot_mapping, int32_t num_tokens,
                                   void* const* k_caches, void* const* v_caches, int32_t num_layers,
                                   const pkv_cache_desc& c, int32_t* err, cudaStream_t stream) {
    if (num_tokens == 0 || num_layers == 0) return cudaSuccess;
    LayerTokens tokens{};
    LayerCaches caches{};
    for (int l = 0; l < num_layers; ++l) {
        tokens.k[l] = static_cast<const uint4*>(k[l]);
        tokens.v[l] = static_cast<const uint4*>(v[l]);
        caches.k[l] = static_cast<uint4*>(k_caches[l]);
        caches.v[l] = static_cast<uint4*>(v_caches[l]);
    }
    const int32_t chunks = c.head_dim / 8;
    const int64_t total = static_cast<int64_t>(num_tokens) * c.num_kv_heads * chunks;
    const int64_t blocks = (total + kThreads - 1) / kThreads;
    const unsigned grid = static_cast<unsigned>(blocks < 152 * 4 ? blocks : 152 * 4);
    return launch_pdl(kv_write_layers_kernel, dim3(grid, 1, static_cast<unsigned>(num_layers)),
                      dim3(kThreads), 0, stream, tokens, caches, slot_mapping, num_tokens,
                      c.num_kv_heads, c.block_size, chunks,
                      static_cast<int64_t>(c.num_blocks) * c.block_size, err);
}

}  // namespace pkv
