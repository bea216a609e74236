// Paged prefill attention for sm_103a: many query tokens per sequence,
// causal, over keys and values that sit in the paged cache.
//
// What it computes ("vLLM PagedAttention & continuous batching", "Prompt
// phase, decode phase": prefill runs the known prompt as matrix-matrix
// work and writes K and V): sequence s holds n = seq_lens[s] tokens in its
// blocks; its last q_len = cu_q[s+1] - cu_q[s] tokens are this call's
// queries, query i at position ctx + i (ctx = n - q_len: an earlier prompt
// chunk or a shared prefix already cached).  Query i attends to positions
// 0 .. ctx + i with softmax(scale * q K^T) V, accumulated key tile by key
// tile with the running max / running sum of Eq. (4) of "Serving Language
// Models Within a Memory Budget".
//
// Work decomposition.  One CTA per (128-row tile, KV head, sequence), where
// a row is one (query token, query head of the KV head's group) pair, so
// the group shares every K/V tile.  Row tiles run longest-first (the last
// rows see the most keys).  Warp 8 is a TMA producer: it streams 64-key
// tiles of K and V (16-row boxes of the 4-D pool view, 128-byte swizzle,
// two 8-row boxes per 16 keys at block size 8) into a three-stage ring
// guarded by full / empty mbarriers.  Warps 0-7 own 16 rows each and
// consume every tile: S = Q K^T with mma.sync m16n8k16 (Q fragments held in
// registers), per-row causal mask, fp32 online softmax in the log2 domain,
// O += P V with P split into high and low 16-bit parts.  Each row's output
// is O / l, rounded to the storage type.
//
// The contraction is dense here: 128 rows x 64 keys x 128 per tile and
// direction, ~128 flops per K/V byte read at 4 query heads per KV head.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

#ifndef PKV_PREFILL_WARPS
#define PKV_PREFILL_WARPS 8
#endif
constexpr int kWarps = PKV_PREFILL_WARPS;      // consumer warps, 16 rows each
constexpr int kThreads = (kWarps + 1) * 32;    // + the TMA producer warp
constexpr int kRows = kWarps * 16;             // rows per CTA
constexpr int kKeys = 64;                      // keys per stage
constexpr int kSub = kKeys / kTileTokens;      // 16-key sub-tiles per stage
constexpr int kHalfBytes = kTileTokens * 128;  // one 64-column box of 16 rows: 2 KiB
constexpr int kSubBytes = 2 * kHalfBytes;      // [16 x 128] sub-tile: 4 KiB
constexpr int kTileBytes = kSub * kSubBytes;   // K (or V) of a stage: 16 KiB
constexpr int kStageBytes = 2 * kTileBytes;    // 32 KiB
constexpr int kStages = 3;
constexpr int kRingBytes = kStages * kStageBytes;

struct alignas(8) PrefillControl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int32_t valid[kStages];
};

// One stage: rows a / b of this thread may see keys up to lim0 / lim1.
template <typename T>
__device__ __forceinline__ void attend_tile_causal(uint32_t k_base, uint32_t v_base, int key0,
                                                   int n, int lim0, int lim1,
                                                   const uint32_t (&qa)[8][4], float (&o)[16][4],
                                                   float& m0, float& m1, float& l0, float& l1,
                                                   float scale_log2, int lane) {
    constexpr int NT = kKeys / 8;  // n-tiles of 8 keys
    const int mi = lane >> 3;
    const int r = lane & 7;
    const int quad = lane & 3;

    float sc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int j = 0; j < kSub; ++j) {
        const uint32_t kt = k_base + j * kSubBytes;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int token = (mi >> 1) * 8 + r;
            const int chunk = (ks & 3) * 2 + (mi & 1);
            const uint32_t addr = kt + (ks >> 2) * kHalfBytes + token * 128 + ((chunk ^ r) << 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(addr, b0, b1, b2, b3);
            Mma<T>::run(sc[2 * j], qa[ks], b0, b1);
            Mma<T>::run(sc[2 * j + 1], qa[ks], b2, b3);
        }
    }

    float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int key = key0 + nt * 8 + quad * 2 + (e & 1);
            const int lim = (e < 2) ? lim0 : lim1;
            const float x = sc[nt][e] * scale_log2;
            sc[nt][e] = key <= lim ? x : -INFINITY;  // select: discards NaN of unloaded rows
        }
        bm0 = fmaxf(bm0, fmaxf(sc[nt][0], sc[nt][1]));
        bm1 = fmaxf(bm1, fmaxf(sc[nt][2], sc[nt][3]));
    }
    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 1));
    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 2));
    bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 1));
    bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 2));
    const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
    const float base0 = mn0 == -INFINITY ? 0.f : mn0;
    const float base1 = mn1 == -INFINITY ? 0.f : mn1;
    const float alpha0 = ex2(m0 - base0), alpha1 = ex2(m1 - base1);
    m0 = mn0;
    m1 = mn1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        sc[nt][0] = ex2(sc[nt][0] - base0);
        sc[nt][1] = ex2(sc[nt][1] - base0);
        sc[nt][2] = ex2(sc[nt][2] - base1);
        sc[nt][3] = ex2(sc[nt][3] - base1);
        ps0 += sc[nt][0] + sc[nt][1];
        ps1 += sc[nt][2] + sc[nt][3];
    }
    l0 = l0 * alpha0 + ps0;
    l1 = l1 * alpha1 + ps1;
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
        o[nd][0] *= alpha0;
        o[nd][1] *= alpha0;
        o[nd][2] *= alpha1;
        o[nd][3] *= alpha1;
    }

#pragma unroll
    for (int kk = 0; kk < kSub; ++kk) {
        const int nvalid = n - (key0 + kk * kTileTokens);  // keys of this sub-tile in the cache
        if (nvalid <= 0) continue;                          // nothing loaded: weights are all 0
        uint32_t pa[4], pl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int nt = 2 * kk + (e >> 1);
            const int c = (e & 1) * 2;
            pa[e] = Mma<T>::pack(sc[nt][c], sc[nt][c + 1]);
            const float2 hi = Mma<T>::unpack(pa[e]);
            pl[e] = Mma<T>::pack(sc[nt][c] - hi.x, sc[nt][c + 1] - hi.y);
        }
        const uint32_t vt = v_base + kk * kSubBytes;
        const bool partial = nvalid < kTileTokens;
#pragma unroll
        for (int np = 0; np < 8; ++np) {
            const int token = (mi & 1) * 8 + r;
            const int d8 = 2 * np + (mi >> 1);
            const uint32_t addr = vt + (d8 >> 3) * kHalfBytes + token * 128 + (((d8 & 7) ^ r) << 4);
            uint32_t v0, v1, v2, v3;
            ldsm_x4_trans(addr, v0, v1, v2, v3);
            if (partial) {  // rows past the sequence end hold stale bytes: zero them
                const int t0 = quad * 2;
                const uint32_t keep0 =
                    ((t0 < nvalid) ? 0x0000ffffu : 0u) | ((t0 + 1 < nvalid) ? 0xffff0000u : 0u);
                const uint32_t keep1 =
                    ((t0 + 8 < nvalid) ? 0x0000ffffu : 0u) | ((t0 + 9 < nvalid) ? 0xffff0000u : 0u);
                v0 &= keep0;
                v2 &= keep0;
                v1 &= keep1;
                v3 &= keep1;
            }
            Mma<T>::run(o[2 * np], pa, v0, v1);
            Mma<T>::run(o[2 * np + 1], pa, v2, v3);
            Mma<T>::run(o[2 * np], pl, v0, v1);
            Mma<T>::run(o[2 * np + 1], pl, v2, v3);
        }
    }
}

template <typename T, int BS>
__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap k_map,
                         const __grid_constant__ CUtensorMap v_map, const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    PrefillControl* ctl = reinterpret_cast<PrefillControl*>(ring + kRingBytes);

    const int h = blockIdx.y;
    const int s = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = a.group;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_addr(&ctl->full[i]), 1);
            mbar_init(smem_addr(&ctl->empty[i]), kWarps);
        }
        fence_barrier_init();
        prefetch_tensormap(&k_map);
        prefetch_tensormap(&v_map);
    }
    pdl_wait_prerequisites();
    pdl_allow_dependents();

    const int q0 = __ldg(a.cu_q + s);
    const int q_len = __ldg(a.cu_q + s + 1) - q0;
    const int n = __ldg(a.seq_lens + s);
    const bool report_here = blockIdx.x == 0 && h == 0 && threadIdx.x == 0;
    if (n < 0 || n > a.max_seq_len || q_len < 0 || q_len > a.max_q_len || q_len > n) {
        if (report_here) report(a.err, PKV_DEVERR_BAD_SEQ_LEN);
        return;  // uniform over the CTA
    }
    const int ctx = n - q_len;
    const int rows_total = q_len * g;
    const int row_tiles = (rows_total + kRows - 1) / kRows;
    if (static_cast<int>(blockIdx.x) >= row_tiles) return;
    const int row_tile = row_tiles - 1 - static_cast<int>(blockIdx.x);  // longest first
    const int R0 = row_tile * kRows;
    const int last_row = min(R0 + kRows, rows_total) - 1;
    const int kv_len = ctx + last_row / g + 1;  // keys the CTA's last row sees
    const int n_tiles = (kv_len + kKeys - 1) / kKeys;
    __syncthreads();  // barrier initialisation visible to every warp

    if (warp == kWarps) {
        // ======================== TMA producer warp ===========================
        constexpr int kBlocksPerSub = BS < kTileTokens ? kTileTokens / BS : 1;
        constexpr int kBoxRows = BS < kTileTokens ? BS : kTileTokens;
        const int nblocks = (n + BS - 1) / BS;
        const int32_t* table = a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq;
        int win_base = -(1 << 30), win_id = -1;
        for (int kt = 0; kt < n_tiles; ++kt) {
            const int st = kt % kStages;
            const int use = kt / kStages;
            // the block ids of this tile (at most 8), through a 32-entry window
            const int first_blk = (kt * kKeys) / BS;
            const int last_blk = min((kt * kKeys + kKeys - 1) / BS, nblocks - 1);
            if (first_blk < win_base || last_blk >= win_base + 32) {
                win_base = first_blk;
                const int e = win_base + lane;
                win_id = e < nblocks ? __ldg(table + e) : -1;
            }
            bool ok = true;
            uint32_t bytes = 0;
            int ids[kSub * kBlocksPerSub];
#pragma unroll
            for (int j = 0; j < kSub; ++j) {
#pragma unroll
                for (int b = 0; b < kBlocksPerSub; ++b) {
                    const int key = kt * kKeys + j * kTileTokens + b * kBoxRows;
                    const int src = min(max(key / BS - win_base, 0), 31);
                    const int id = __shfl_sync(0xffffffffu, win_id, src);
                    ids[j * kBlocksPerSub + b] = id;
                    if (key < n) {  // blocks past the sequence end are not read
                        ok = ok && id >= 0 && id < a.num_blocks;
                        bytes += kBoxRows * 128 * 4;
                    }
                }
            }
            int timed_out = 0;
            if (lane == 0 && use > 0 && !mbar_wait(smem_addr(&ctl->empty[st]), (use - 1) & 1))
                timed_out = 1;
            if (__shfl_sync(0xffffffffu, timed_out, 0)) {  // the whole warp stops together
                if (lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
                break;
            }
            if (lane == 0) {
                const uint32_t full = smem_addr(&ctl->full[st]);
                ctl->valid[st] = ok ? 1 : 0;
                if (ok) {
                    const uint32_t kb = smem_addr(ring + st * kStageBytes);
                    const uint32_t vb = kb + kTileBytes;
                    mbar_arrive_expect_tx(full, bytes);
#pragma unroll
                    for (int j = 0; j < kSub; ++j) {
#pragma unroll
                        for (int b = 0; b < kBlocksPerSub; ++b) {
                            const int key = kt * kKeys + j * kTileTokens + b * kBoxRows;
                            if (key >= n) continue;
                            const int id = ids[j * kBlocksPerSub + b];
                            const int row = key % BS;  // 0 unless BS > 16
                            const uint32_t off = j * kSubBytes + b * kBoxRows * 128;
                            tma_load_4d(kb + off, &k_map, full, 0, row, h, id);
                            tma_load_4d(kb + off + kHalfBytes, &k_map, full, 64, row, h, id);
                            tma_load_4d(vb + off, &v_map, full, 0, row, h, id);
                            tma_load_4d(vb + off + kHalfBytes, &v_map, full, 64, row, h, id);
                        }
                    }
                } else {
                    report(a.err, PKV_DEVERR_BAD_BLOCK_ID);
                    mbar_arrive(full);
                }
            }
            __syncwarp();
        }
        if (lane == 0) {  // leave only once this CTA's copies have landed (bounded)
            const int first = n_tiles > kStages ? n_tiles - kStages : 0;
            for (int kt = first; kt < n_tiles; ++kt)
                mbar_wait(smem_addr(&ctl->full[kt % kStages]), (kt / kStages) & 1);
        }
        return;
    }

    // =========================== consumer warps ================================
    const int row_a = R0 + warp * 16 + (lane >> 2);  // this thread's two rows
    const int row_b = row_a + 8;
    const bool live_a = row_a < rows_total, live_b = row_b < rows_total;
    const int lim_a = live_a ? ctx + row_a / g : -1;
    const int lim_b = live_b ? ctx + row_b / g : -1;
    const T* q = static_cast<const T*>(a.q);
    const size_t qa_off = live_a ? (static_cast<size_t>(q0 + row_a / g) * a.num_q_heads +
                                    static_cast<size_t>(h) * g + row_a % g) * kHeadDim : 0;
    const size_t qb_off = live_b ? (static_cast<size_t>(q0 + row_b / g) * a.num_q_heads +
                                    static_cast<size_t>(h) * g + row_b % g) * kHeadDim : 0;
    const int quad = lane & 3;
    uint32_t qa[8][4];
    {
        const uint32_t* qra = reinterpret_cast<const uint32_t*>(q + qa_off);
        const uint32_t* qrb = reinterpret_cast<const uint32_t*>(q + qb_off);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int w = ks * 8 + quad;
            qa[ks][0] = live_a ? __ldg(qra + w) : 0u;
            qa[ks][1] = live_b ? __ldg(qrb + w) : 0u;
            qa[ks][2] = live_a ? __ldg(qra + w + 4) : 0u;
            qa[ks][3] = live_b ? __ldg(qrb + w + 4) : 0u;
        }
    }
    float o[16][4];
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int kt = 0; kt < n_tiles; ++kt) {
        const int st = kt % kStages;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->full[st]), (kt / kStages) & 1))) {
            if (lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
            break;  // the whole warp stops together
        }
        if (ctl->valid[st]) {
            const uint32_t kb = smem_addr(ring + st * kStageBytes);
            attend_tile_causal<T>(kb, kb + kTileBytes, kt * kKeys, n, lim_a, lim_b, qa, o, m0, m1,
                                  l0, l1, a.scale_log2, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&ctl->empty[st]));
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
    const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    T* out = static_cast<T*>(a.out);
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
        const int col = nd * 8 + quad * 2;
        if (live_a)
            *reinterpret_cast<uint32_t*>(out + qa_off + col) =
                Mma<T>::pack(o[nd][0] * inv0, o[nd][1] * inv0);
        if (live_b)
            *reinterpret_cast<uint32_t*>(out + qb_off + col) =
                Mma<T>::pack(o[nd][2] * inv1, o[nd][3] * inv1);
    }
}

template <typename T, int BS>
cudaError_t launch_prefill_typed(const CUtensorMap& k_map, const CUtensorMap& v_map,
                                 const PrefillArgs& a, cudaStream_t stream) {
    const size_t smem = 1024 + kRingBytes + sizeof(PrefillControl);
    cudaError_t err = ensure_smem_limit<paged_prefill_kernel<T, BS>>(smem);
    if (err != cudaSuccess) return err;
    const int64_t row_tiles = (static_cast<int64_t>(a.max_q_len) * a.group + kRows - 1) / kRows;
    dim3 grid(static_cast<unsigned>(row_tiles > 0 ? row_tiles : 1),
              static_cast<unsigned>(a.num_kv_heads), static_cast<unsigned>(a.num_seqs));
    return launch_pdl(paged_prefill_kernel<T, BS>, grid, dim3(kThreads), smem, stream, k_map,
                      v_map, a);
}

template <typename T>
cudaError_t launch_prefill_dtype(const CUtensorMap& k_map, const CUtensorMap& v_map,
                                 const PrefillArgs& a, int block_size, cudaStream_t stream) {
    switch (block_size) {
        case 8: return launch_prefill_typed<T, 8>(k_map, v_map, a, stream);
        case 16: return launch_prefill_typed<T, 16>(k_map, v_map, a, stream);
        case 32: return launch_prefill_typed<T, 32>(k_map, v_map, a, stream);
        case 64: return launch_prefill_typed<T, 64>(k_map, v_map, a, stream);
        default: return launch_prefill_typed<T, 128>(k_map, v_map, a, stream);
    }
}

}  // namespace

cudaError_t launch_paged_prefill(const CUtensorMap& k_map16, const CUtensorMap& v_map16,
                                 const PrefillArgs& args, pkv_dtype dtype, int block_size,
                                 cudaStream_t stream) {
    return dtype == PKV_BF16
               ? launch_prefill_dtype<__nv_bfloat16>(k_map16, v_map16, args, block_size, stream)
               : launch_prefill_dtype<__half>(k_map16, v_map16, args, block_size, stream);
}

}  // namespace pkv
