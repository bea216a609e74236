// kv_write: scatter new keys / values into their cache slots through the
// slot mapping (slot = physical block * block_size + offset).  Decode
// writes each sequence's next token into the spare slot of its last block
// (vLLM PagedAttention & continuous batching, "PagedAttention", the
// seven-token example).
//
// One thread moves one 16-byte vector of a (token, KV head) row of K and
// the matching vector of V; rows are head_dim * 2 bytes, contiguous on both
// sides, so loads and stores are fully coalesced.  The kernel is bound by
// launch latency at decode sizes (tens to hundreds of KiB per call); index
// arithmetic stays in 32 bits unless the pool or the batch needs more.
//
// The 8-bit variant stores each scalar of a row as the E4M3 code of
// x / scale (binary32 quotient, saturating round-to-nearest-even), the
// reading of a lower-precision key-value cache ("Serving Language Models
// Within a Memory Budget", section 4) that the header describes.
#include <cuda_fp8.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

template <typename I>
__global__ void __launch_bounds__(256) kv_write_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v,
    const int64_t* __restrict__ slot_mapping, int32_t num_tokens, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, int32_t num_kv_heads, int32_t block_size, int32_t chunks,
    int64_t num_slots, int32_t* err) {
    pdl_wait_prerequisites();
    pdl_allow_dependents();
    const I total = static_cast<I>(num_tokens) * num_kv_heads * chunks;
    const I stride = static_cast<I>(gridDim.x) * blockDim.x;
    for (I idx = static_cast<I>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const I row = idx / chunks;  // token * num_kv_heads + head
        const int32_t c = static_cast<int32_t>(idx - row * chunks);
        const I t = row / num_kv_heads;
        const int32_t h = static_cast<int32_t>(row - t * num_kv_heads);
        const uint4 kv = __ldg(k + idx);
        const uint4 vv = __ldg(v + idx);
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;  // padding token
        if (slot >= num_slots) {
            if (h == 0 && c == 0) report(err, PKV_DEVERR_BAD_SLOT);
            continue;
        }
        const I block = static_cast<I>(slot) / block_size;
        const I offset = static_cast<I>(slot) - block * block_size;
        const int64_t dst =
            ((static_cast<int64_t>(block) * num_kv_heads + h) * block_size + offset) * chunks + c;
        k_cache[dst] = kv;
        v_cache[dst] = vv;
    }
}

// ---- 8-bit pools -------------------------------------------------------------
// Two 16-bit scalars of a word, widened exactly to binary32.
template <typename T>
__device__ __forceinline__ float2 widen2(uint32_t w);
template <>
__device__ __forceinline__ float2 widen2<__nv_bfloat16>(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <>
__device__ __forceinline__ float2 widen2<__half>(uint32_t w) {
    __half2_raw raw;
    raw.x = static_cast<unsigned short>(w & 0xffffu);
    raw.y = static_cast<unsigned short>(w >> 16);
    return __half22float2(__half2(raw));
}

// E4M3 codes of x / scale for the 8 scalars of a 16-byte vector: binary32
// quotient (round to nearest), then the saturating round-to-nearest-even
// conversion; scalar j lands in byte j.
template <typename T>
__device__ __forceinline__ uint2 quantize8(uint4 x, float scale) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t pair[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = widen2<T>(w[i]);
        const float2 qf = make_float2(__fdiv_rn(f.x, scale), __fdiv_rn(f.y, scale));
        pair[i] = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(qf, __NV_SATFINITE, __NV_E4M3));
    }
    return make_uint2(pair[0] | (pair[1] << 16), pair[2] | (pair[3] << 16));
}

template <typename T>
__global__ void __launch_bounds__(256) kv_write_fp8_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v,
    const int64_t* __restrict__ slot_mapping, int32_t num_tokens, uint2* __restrict__ k_cache,
    uint2* __restrict__ v_cache, int32_t num_kv_heads, int32_t block_size, int32_t chunks,
    int64_t num_slots, float k_scale, float v_scale, int32_t* err) {
    pdl_wait_prerequisites();
    pdl_allow_dependents();
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
        const uint4 kv = __ldg(k + idx);
        const uint4 vv = __ldg(v + idx);
        const int64_t block = slot / block_size;
        const int64_t offset = slot - block * block_size;
        const int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * chunks + c;
        k_cache[dst] = quantize8<T>(kv, k_scale);
        v_cache[dst] = quantize8<T>(vv, v_scale);
    }
}

}  // namespace

cudaError_t launch_kv_write_fp8(const void* k, const void* v, pkv_dtype kv_dtype,
                                const int64_t* slot_mapping, int32_t num_tokens, void* k_cache,
                                void* v_cache, const pkv_cache_desc& c, float k_scale,
                                float v_scale, int32_t* err, cudaStream_t stream) {
    const int32_t chunks = c.head_dim / 8;  // 16-byte input vectors (8-byte outputs) per row
    const int64_t total = static_cast<int64_t>(num_tokens) * c.num_kv_heads * chunks;
    if (total == 0) return cudaSuccess;
    const int64_t num_slots = static_cast<int64_t>(c.num_blocks) * c.block_size;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    const int grid = static_cast<int>(blocks < 152 * 16 ? blocks : 152 * 16);
    auto kernel = kv_dtype == PKV_BF16 ? kv_write_fp8_kernel<__nv_bfloat16> : kv_write_fp8_kernel<__half>;
    return launch_pdl(kernel, dim3(grid), dim3(threads), 0, stream, static_cast<const uint4*>(k),
                      static_cast<const uint4*>(v), slot_mapping, num_tokens,
                      static_cast<uint2*>(k_cache), static_cast<uint2*>(v_cache), c.num_kv_heads,
                      c.block_size, chunks, num_slots, k_scale, v_scale, err);
}

cudaError_t launch_kv_write(const void* k, const void* v, const int64_t* slot_mapping,
                            int32_t num_tokens, void* k_cache, void* v_cache,
                            const pkv_cache_desc& c, int32_t* err, cudaStream_t stream) {
    const int32_t chunks = c.head_dim / 8;  // 16-byte vectors per row
    const int64_t total = static_cast<int64_t>(num_tokens) * c.num_kv_heads * chunks;
    if (total == 0) return cudaSuccess;
    const int64_t num_slots = static_cast<int64_t>(c.num_blocks) * c.block_size;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    const int grid = static_cast<int>(blocks < 152 * 16 ? blocks : 152 * 16);
    const bool narrow = total < (int64_t{1} << 31) && num_slots < (int64_t{1} << 31);
    const uint4* kp = static_cast<const uint4*>(k);
    const uint4* vp = static_cast<const uint4*>(v);
    uint4* kc = static_cast<uint4*>(k_cache);
    uint4* vc = static_cast<uint4*>(v_cache);
    if (narrow)
        return launch_pdl(kv_write_kernel<int32_t>, dim3(grid), dim3(threads), 0, stream, kp, vp,
                          slot_mapping, num_tokens, kc, vc, c.num_kv_heads, c.block_size, chunks,
                          num_slots, err);
    return launch_pdl(kv_write_kernel<int64_t>, dim3(grid), dim3(threads), 0, stream, kp, vp,
                      slot_mapping, num_tokens, kc, vc, c.num_kv_heads, c.block_size, chunks,
                      num_slots, err);
}

}  // namespace pkv
