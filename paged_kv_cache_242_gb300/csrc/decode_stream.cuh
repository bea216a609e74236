// The streaming paged decode kernel as a template over the per-warp
// attention policy (decode_policy.cuh), with its merge kernel and launch
// helpers.  decode_stream.cu instantiates it for 16-bit pools and
// decode_stream_fp8.cu for 8-bit pools.
//
// Streaming paged decode attention: a persistent grid with one CTA of
// kStreamWarps (7) warps per SM (8 over 8-bit pools), each warp an
// independent TMA pipeline.
//
// What it computes is the same as the partition kernel (decode_attention.cu):
// for every sequence and query head, softmax(scale * q K^T) V over the
// sequence's paged keys and values, block by block with the running max /
// running sum of Eq. (4) of "Serving Language Models Within a Memory Budget"
// (vLLM PagedAttention & continuous batching, "PagedAttention": the kernel
// scores the query against one block, then the next, and combines them).
//
// Work split.  All (sequence, KV head) segments are cut into 16-token tiles
// (a whole block at block size 16, a slice of one block at 32 / 64 / 128,
// two blocks at 8; 32-token tiles over 8-bit pools) and laid end to end in
// (sequence, head, tile) order.  Warp w of the grid takes the contiguous
// range [w * per, (w + 1) * per) of that order, per = ceil(tiles / warps), so
// every warp streams the same number of bytes and the grid finishes together
// whatever the mix of lengths.  A warp that covers a whole segment writes the
// final output; a warp whose range cuts a segment writes that segment's
// partial (max, sum, weighted sum) statistics, which the merge kernel
// combines by the same Eq. (4) rule.
//
// Pipeline.  Each warp owns kStreamStages (2) 8 KiB shared-memory stages
// (K and V of one tile, two 64-column boxes each, 128-byte swizzle); over
// 8-bit (E4M3) pools, kStreamStagesFp8 (4) stages of 4 KiB (one 128-byte
// box per tile) and the per-tile math of attend_tile_e4m3.  Lane 0
// issues the TMA loads of tile k + stages as soon as the warp has finished
// tile k, so 16-bit pools keep 14 tiles per SM in flight or being consumed.  (Sweeps of warps x
// stages on GB300 put the optimum at 7-8 warps x 2 stages: more requests in
// flight only queue at the saturated HBM.)  Block-table entries are fetched
// 32 at a time by the whole warp.  The per-tile math is the policy's
// (decode_policy.cuh): mma.sync Q K^T, fp32 online softmax in the log2
// domain, mma.sync P V.
//
// The prologue of every CTA scans the sequence lengths into a prefix of tile
// counts held in shared memory (up to 4096 sequences).
#pragma once

#include "decode_policy.cuh"

namespace pkv {
namespace {

// Shared-memory layout of one warp's ring.  16-bit pools: a stage holds the
// K and V tiles of 16 rows as two 64-column boxes each (8 KiB).  8-bit pools
// (E4M3 codes): one 128-byte box per tile (4 KiB), twice the stages.
template <bool kFp8, int kWarpsPerCta>
struct StreamLayout {
    static constexpr int kWarps = kWarpsPerCta;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kStages = kFp8 ? kStreamStagesFp8 : kStreamStages;
    static constexpr int kTileTokens = kFp8 ? kTileTokensFp8 : pkv::kTileTokens;
    static constexpr int kTileBytes = kTileTokens * kHeadDim * (kFp8 ? 1 : 2);  // K or V
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kRingBytes = kWarps * kStages * kStageBytes;
};
constexpr int kHalf = kTileTokens * 128;  // one 64-column box of 16 rows of a 16-bit pool

template <int kWarps, int kStages>
struct alignas(8) StreamControl {
    uint64_t full[kWarps][kStages];
    int32_t valid[kWarps][kStages];
    int32_t warp_total[kWarps];
};

// Position of one tile in the (sequence, head, tile) order.
struct Cursor {
    int s;   // sequence
    int h;   // KV head
    int i;   // tile within the segment
    int nt;  // tiles in the segment
};

__device__ __forceinline__ void cursor_advance(Cursor& c, const int32_t* prefix, int num_seqs,
                                               int num_kv_heads) {
    if (++c.i < c.nt) return;
    c.i = 0;
    if (++c.h < num_kv_heads) return;
    c.h = 0;
    do {
        ++c.s;
    } while (c.s < num_seqs && prefix[c.s + 1] == prefix[c.s]);
    c.nt = c.s < num_seqs ? prefix[c.s + 1] - prefix[c.s] : 1;
}

// Locate global tile index t (0 <= t < total tiles).
__device__ __forceinline__ Cursor cursor_at(int64_t t, const int32_t* prefix, int num_seqs,
                                            int num_kv_heads) {
    // largest s with num_kv_heads * prefix[s] <= t
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<int64_t>(prefix[mid]) * num_kv_heads <= t) lo = mid;
        else hi = mid - 1;
    }
    Cursor c;
    c.s = lo;
    c.nt = prefix[lo + 1] - prefix[lo];
    const int64_t rem = t - static_cast<int64_t>(prefix[lo]) * num_kv_heads;
    c.h = static_cast<int>(rem / c.nt);
    c.i = static_cast<int>(rem - static_cast<int64_t>(c.h) * c.nt);
    return c;
}

template <typename Policy, int BS>
__global__ void __launch_bounds__(Policy::kWarps * 32, 1)
    paged_decode_stream_kernel(const __grid_constant__ CUtensorMap k_map,
                               const __grid_constant__ CUtensorMap v_map, const DecodeArgs a) {
    using T = typename Policy::Scalar;
    constexpr bool kFp8 = Policy::kFp8;
    using L = StreamLayout<kFp8, Policy::kWarps>;
    constexpr int kWarps = L::kWarps;
    constexpr int kThreads = L::kThreads;
    constexpr int kStages = L::kStages;
    constexpr int kStageBytes = L::kStageBytes;
    constexpr int kTT = L::kTileTokens;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    auto* ctl = reinterpret_cast<StreamControl<kWarps, kStages>*>(ring + L::kRingBytes);
    int32_t* prefix = reinterpret_cast<int32_t*>(ctl + 1);  // [S + 1]
    int32_t* lens = prefix + a.num_seqs + 1;                // [S]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = a.num_seqs;
    const int H = a.num_kv_heads;
    if (threadIdx.x == 0) {
        prefetch_tensormap(&k_map);
        prefetch_tensormap(&v_map);
    }
    pdl_wait_prerequisites();
    pdl_allow_dependents();

    // ---- prologue: tile-count prefix over the sequences ---------------------
    {
        const int per_thread = (S + kThreads - 1) / kThreads;  // <= 19 (S <= 4096)
        const int base = threadIdx.x * per_thread;
        int sum = 0;
        for (int k = 0; k < per_thread; ++k) {
            const int idx = base + k;
            if (idx < S) {
                const int n = clamped_len(a, idx, blockIdx.x == 0);
                lens[idx] = n;
                sum += (n + kTT - 1) / kTT;
            }
        }
        // block-wide exclusive scan of the per-thread sums
        int incl = sum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        if (lane == 31) ctl->warp_total[warp] = incl;
        if (threadIdx.x == 0) {
            for (int w = 0; w < kWarps; ++w) {
                for (int st = 0; st < kStages; ++st) mbar_init(smem_addr(&ctl->full[w][st]), 1);
            }
            fence_barrier_init();
        }
        __syncthreads();
        int offset = 0;
        for (int w = 0; w < warp; ++w) offset += ctl->warp_total[w];
        int run = offset + incl - sum;  // exclusive prefix of this thread's first element
        for (int k = 0; k < per_thread; ++k) {
            const int idx = base + k;
            if (idx < S) {
                prefix[idx] = run;
                run += (lens[idx] + kTT - 1) / kTT;
            }
        }
        if (threadIdx.x == kThreads - 1) {
            int total = 0;
            for (int w = 0; w < kWarps; ++w) total += ctl->warp_total[w];
            prefix[S] = total;
        }
        __syncthreads();
    }

    // ---- this warp's share of the tiles --------------------------------------
    const int64_t total_tiles = static_cast<int64_t>(prefix[S]) * H;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
    const int64_t per = total_tiles > 0 ? (total_tiles + a.num_warps - 1) / a.num_warps : 1;
    const int64_t t0 = gw * per;
    const int64_t t1 = min(t0 + per, total_tiles);
    if (t0 >= t1) return;
    const int count = static_cast<int>(t1 - t0);

    uint8_t* my_ring = ring + warp * kStages * kStageBytes;
    const int g = a.group;

    // ---- issue side: cursor, block-table window ------------------------------
    Cursor iss = cursor_at(t0, prefix, S, H);
    int win_s = -1, win_base = 0, win_id = -1;
    int issued = 0;
    // A tile is 16 token rows: rows of one block when BS >= 16, two whole
    // blocks of 8 rows each when BS == 8 (the 128-byte swizzle repeats every
    // 8 rows, so two 8-row boxes land exactly as one 16-row box would).
    constexpr int kBlocksPerTile = BS < kTT ? kTT / BS : 1;
    constexpr int kBoxRows = BS < kTT ? BS : kTT;
    auto issue = [&](int k) {
        issued = k + 1;
        const int st = k % kStages;
        const int blk = (iss.i * kTT) / BS;  // first block of the tile
        const int nblocks = (lens[iss.s] + BS - 1) / BS;
        if (iss.s != win_s || blk < win_base || blk + kBlocksPerTile > win_base + 32) {
            win_s = iss.s;
            win_base = blk;
            const int e = win_base + lane;
            win_id = e < nblocks ? __ldg(a.block_tables + static_cast<size_t>(iss.s) *
                                                               a.max_blocks_per_seq + e)
                                 : -1;
        }
        int ids[kBlocksPerTile];
#pragma unroll
        for (int b = 0; b < kBlocksPerTile; ++b)
            ids[b] = __shfl_sync(0xffffffffu, win_id, blk + b - win_base);
        if (lane == 0) {
            bool ok = true;
            int present = 0;
#pragma unroll
            for (int b = 0; b < kBlocksPerTile; ++b) {
                if (blk + b < nblocks) {  // blocks past the sequence end are not read
                    ok = ok && ids[b] >= 0 && ids[b] < a.num_blocks;
                    ++present;
                }
            }
            const uint32_t full = smem_addr(&ctl->full[warp][st]);
            ctl->valid[warp][st] = ok ? 1 : 0;
            if (ok) {
                const uint32_t kt = smem_addr(my_ring + st * kStageBytes);
                const uint32_t vt = kt + L::kTileBytes;
                const int row = (iss.i * kTT) % BS;  // 0 when BS <= kTT
                fence_proxy_async_shared();  // earlier generic reads of this stage
                mbar_arrive_expect_tx(full, present * kBoxRows * 128 * (kFp8 ? 2 : 4));
#pragma unroll
                for (int b = 0; b < kBlocksPerTile; ++b) {
                    if (blk + b < nblocks) {
                        const uint32_t off = b * kBoxRows * 128;
                        tma_load_4d(kt + off, &k_map, full, 0, row, iss.h, ids[b]);
                        tma_load_4d(vt + off, &v_map, full, 0, row, iss.h, ids[b]);
                        if constexpr (!kFp8) {  // second 64-column half of 16-bit rows
                            tma_load_4d(kt + kHalf + off, &k_map, full, 64, row, iss.h, ids[b]);
                            tma_load_4d(vt + kHalf + off, &v_map, full, 64, row, iss.h, ids[b]);
                        }
                    }
                }
            } else {
                report(a.err, PKV_DEVERR_BAD_BLOCK_ID);
                mbar_arrive(full);
            }
        }
        cursor_advance(iss, prefix, S, H);
    };

    const int prologue = count < kStages ? count : kStages;
    for (int k = 0; k < prologue; ++k) issue(k);

    // ---- consume side ----------------------------------------------------------
    Cursor cur = cursor_at(t0, prefix, S, H);
    bool seg_from_start = cur.i == 0;
    Policy pol;
    auto reset = [&]() {
        const T* q_rows = static_cast<const T*>(a.q) +
                          (static_cast<size_t>(cur.s) * a.num_q_heads + static_cast<size_t>(cur.h) * g) *
                              kHeadDim;
        pol.reset(a, q_rows, g, lane);
    };
    // Write the finished segment `seg` (its whole range, or this warp's part).
    auto flush = [&](const Cursor& seg, bool whole) {
        const size_t qrow = static_cast<size_t>(seg.s) * a.num_q_heads + static_cast<size_t>(seg.h) * g;
        const size_t rbase = static_cast<size_t>(gw + static_cast<int64_t>(seg.s) * H + seg.h) * g;
        pol.flush(a, qrow, rbase, whole, g, lane);
    };

    reset();
    bool aborted = false;
    for (int k = 0; k < count; ++k) {
        const int st = k % kStages;
        if (k > 0 && cur.i == 0) {  // a new segment starts with this tile
            seg_from_start = true;
            reset();
        }
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->full[warp][st]), (k / kStages) & 1))) {
            if (lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
            aborted = true;  // the whole warp stops together
            break;
        }
        if (ctl->valid[warp][st]) {
            const uint32_t kt = smem_addr(my_ring + st * kStageBytes);
            const int nvalid = min(kTT, lens[cur.s] - cur.i * kTT);
            pol.template attend<kTT>(kt, kt + L::kTileBytes, nvalid, lane);
        }
        __syncwarp();
        if (k + kStages < count) issue(k + kStages);
        const bool seg_ends = cur.i == cur.nt - 1 || k == count - 1;
        if (seg_ends) flush(cur, seg_from_start && cur.i == cur.nt - 1);
        cursor_advance(cur, prefix, S, H);
    }
    if (aborted && lane == 0) {
        // do not leave while this warp's copies are still landing (bounded)
        for (int st = 0; st < kStages && st < issued; ++st) {
            const int last = ((issued - 1 - st) / kStages) * kStages + st;  // last use of st
            mbar_wait(smem_addr(&ctl->full[warp][st]), (last / kStages) & 1);
        }
    }
}

// Merge of the partial statistics of segments cut by warp ranges (Eq. 4):
// out = sum_w 2^(m_w - M) acc_w / sum_w 2^(m_w - M) l_w, M = max_w m_w.
// One warp per (segment, query head of the group), four output columns per
// lane.  Launched with programmatic dependent launch, its CTAs start while the
// streaming kernel runs: each warp first derives its segment's position (the
// tile prefix of its sequence and the total) from the sequence lengths, which
// are inputs complete before the streaming kernel started, then waits for the
// streaming kernel.  After that the (m, l, acc) of up to eight pieces are
// loaded together and folded in with the running max / sum, so a segment of
// up to eight pieces costs one dependent memory round trip.
//
// Narrow form: kMergeWarps warps per CTA, one per (segment, query head).
// Wide form, for grids with many warps per segment (long sequences, few
// segments): one CTA of kMergeWideWarps warps per (segment,
// query head); the warps take the batches of eight pieces in turn and their
// (max, sum, acc) are combined through shared memory with the same rule.
constexpr int kMergeWarps = 4;
constexpr int kMergeWideWarps = 8;
#ifndef PKV_MERGE_WIDE_PIECES
#define PKV_MERGE_WIDE_PIECES 8
#endif
constexpr int kMergeWidePieces = PKV_MERGE_WIDE_PIECES;  // expected pieces per segment
constexpr int kMergeBatch = 8;

#ifndef PKV_MERGE_NARROW_CTAS
#define PKV_MERGE_NARROW_CTAS 1
#endif
#ifndef PKV_MERGE_WIDE_CTAS
#define PKV_MERGE_WIDE_CTAS 3
#endif
// CTAs per SM the register budget allows (merge CTAs start as streaming CTAs
// leave their SMs, so a merge grid that fits in one wave drains quickest)
constexpr int kMergeNarrowCtas = PKV_MERGE_NARROW_CTAS;
constexpr int kMergeWideCtas = PKV_MERGE_WIDE_CTAS;

template <typename T, int kTT, bool kWide>
__global__ void __launch_bounds__((kWide ? kMergeWideWarps : kMergeWarps) * 32,
                                  kWide ? kMergeWideCtas : kMergeNarrowCtas)
    merge_stream_kernel(const DecodeArgs a) {
    const int g = a.group;
    const int H = a.num_kv_heads;
    const int S = a.num_seqs;
    const int warp = threadIdx.x >> 5;
    constexpr int kWpi = kWide ? kMergeWideWarps : 1;  // warps per item
    const int sub = kWide ? warp : 0;                  // this warp's place among them
    // every early exit below depends on the item alone: uniform over a wide CTA
    const int64_t item = kWide ? static_cast<int64_t>(blockIdx.x)
                               : static_cast<int64_t>(blockIdx.x) * kMergeWarps + warp;
    if (item >= static_cast<int64_t>(S) * H * g) return;
    const int lane = threadIdx.x & 31;
    const int r = static_cast<int>(item % g);
    const int64_t j = item / g;  // segment = s * H + h
    const int s = static_cast<int>(j / H);
    const int h = static_cast<int>(j - static_cast<int64_t>(s) * H);
    // tiles before sequence s, of sequence s, and in all (the streaming kernel's prefix)
    int before = 0, mine = 0, total = 0;
    for (int base = 0; base < S; base += 32) {
        const int idx = base + lane;
        const int t = idx < S ? (clamped_len(a, idx, false) + kTT - 1) / kTT : 0;
        total += t;
        before += idx < s ? t : 0;
        mine += idx == s ? t : 0;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        total += __shfl_xor_sync(0xffffffffu, total, off);
        before += __shfl_xor_sync(0xffffffffu, before, off);
        mine += __shfl_xor_sync(0xffffffffu, mine, off);
    }
    pdl_wait_prerequisites();
    pdl_allow_dependents();
    const int p_s = before;
    const int nt = mine;
    const int64_t total_tiles = static_cast<int64_t>(total) * H;
    // 32-bit stores: out is only 4-byte aligned
    uint32_t* ocol = reinterpret_cast<uint32_t*>(
        static_cast<T*>(a.out) +
        (static_cast<size_t>(s) * a.num_q_heads + static_cast<size_t>(h) * g + r) * kHeadDim +
        lane * 4);
    if (nt == 0) {  // empty sequence: zero output
        if (sub == 0) {
            ocol[0] = 0u;
            ocol[1] = 0u;
        }
        return;
    }
    const int64_t per = (total_tiles + a.num_warps - 1) / a.num_warps;
    const int64_t first = static_cast<int64_t>(p_s) * H + static_cast<int64_t>(h) * nt;
    const int64_t w0 = first / per;
    const int64_t w1 = (first + nt - 1) / per;
    if (w0 == w1) return;  // one warp covered the segment and wrote the output
    const int np = static_cast<int>(w1 - w0 + 1);
    const size_t row0 = static_cast<size_t>(w0 + j) * g + r;  // piece p is row row0 + p * g

    float big = -INFINITY, den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = sub * kMergeBatch; base < np; base += kWpi * kMergeBatch) {
        float m[kMergeBatch], l[kMergeBatch];
        float4 v[kMergeBatch];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
            const size_t row = row0 + static_cast<size_t>(base + u) * g;
            const bool live = base + u < np;
            m[u] = live ? a.ws_m[row] : -INFINITY;
            l[u] = live ? a.ws_l[row] : 0.f;
            v[u] = live ? *reinterpret_cast<const float4*>(a.ws_acc + row * kHeadDim + lane * 4)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
            const float nb = fmaxf(big, m[u]);
            if (nb == -INFINITY) continue;
            const float sa = ex2(big - nb);  // 0 while big = -inf
            const float sb = ex2(m[u] - nb);
            den = den * sa + l[u] * sb;
            acc.x = acc.x * sa + v[u].x * sb;
            acc.y = acc.y * sa + v[u].y * sb;
            acc.z = acc.z * sa + v[u].z * sb;
            acc.w = acc.w * sa + v[u].w * sb;
            big = nb;
        }
    }
    if constexpr (kWide) {
        // dynamic shared memory: acc [warps][32] float4, then max and sum [warps]
        extern __shared__ float4 merge_smem[];
        float4(*s_acc)[32] = reinterpret_cast<float4(*)[32]>(merge_smem);
        float* s_big = reinterpret_cast<float*>(merge_smem + kMergeWideWarps * 32);
        float* s_den = s_big + kMergeWideWarps;
        if (lane == 0) {
            s_big[warp] = big;
            s_den[warp] = den;
        }
        s_acc[warp][lane] = acc;
        __syncthreads();
        if (warp != 0) return;
        big = -INFINITY;
#pragma unroll
        for (int w = 0; w < kMergeWideWarps; ++w) big = fmaxf(big, s_big[w]);
        den = 0.f;
        acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kMergeWideWarps; ++w) {
            if (s_big[w] == -INFINITY) continue;  // no pieces, or none with a token
            const float sc = ex2(s_big[w] - big);
            const float4 v = s_acc[w][lane];
            den += s_den[w] * sc;
            acc.x += v.x * sc;
            acc.y += v.y * sc;
            acc.z += v.z * sc;
            acc.w += v.w * sc;
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    ocol[0] = Mma<T>::pack(acc.x * inv, acc.y * inv);
    ocol[1] = Mma<T>::pack(acc.z * inv, acc.w * inv);
}

template <bool kFp8, int kWarps>
constexpr size_t stream_smem_bytes(int num_seqs) {
    using L = StreamLayout<kFp8, kWarps>;
    return 1024 + L::kRingBytes + sizeof(StreamControl<L::kWarps, L::kStages>) +
           (2 * static_cast<size_t>(num_seqs) + 1) * sizeof(int32_t);
}

template <typename Policy, int BS>
cudaError_t launch_stream_typed(const CUtensorMap& k_map, const CUtensorMap& v_map,
                                const DecodeArgs& a, int ctas, int sms, cudaStream_t stream) {
    using T = typename Policy::Scalar;
    constexpr bool kFp8 = Policy::kFp8;
    const size_t smem = stream_smem_bytes<kFp8, Policy::kWarps>(a.num_seqs);
    auto kernel = paged_decode_stream_kernel<Policy, BS>;
    cudaError_t err = ensure_smem_limit<paged_decode_stream_kernel<Policy, BS>>(smem);
    if (err != cudaSuccess) return err;
    err = launch_pdl(kernel, dim3(ctas), dim3(Policy::kWarps * 32), smem, stream, k_map, v_map, a);
    if (err != cudaSuccess) return err;
    const int64_t items = static_cast<int64_t>(a.num_seqs) * a.num_kv_heads * a.group;
    constexpr int kTT = StreamLayout<kFp8, Policy::kWarps>::kTileTokens;
    // The wide form for about kMergeWidePieces or more pieces per segment,
    // when its grid fits in one wave.
    if (a.num_warps >= kMergeWidePieces * static_cast<int64_t>(a.num_seqs) * a.num_kv_heads &&
        items <= static_cast<int64_t>(kMergeWideCtas) * sms) {
        constexpr size_t kWideSmem = kMergeWideWarps * (32 * sizeof(float4) + 2 * sizeof(float));
        return launch_pdl(merge_stream_kernel<T, kTT, true>, dim3(static_cast<unsigned>(items)),
                          dim3(kMergeWideWarps * 32), kWideSmem, stream, a);
    }
    const int64_t blocks = (items + kMergeWarps - 1) / kMergeWarps;
    return launch_pdl(merge_stream_kernel<T, kTT, false>, dim3(static_cast<unsigned>(blocks)),
                      dim3(kMergeWarps * 32), 0, stream, a);
}

template <typename Policy>
cudaError_t launch_stream_block(const CUtensorMap& k_map, const CUtensorMap& v_map,
                                const DecodeArgs& a, int block_size, int ctas, int sms,
                                cudaStream_t stream) {
    switch (block_size) {
        case 8: return launch_stream_typed<Policy, 8>(k_map, v_map, a, ctas, sms, stream);
        case 16: return launch_stream_typed<Policy, 16>(k_map, v_map, a, ctas, sms, stream);
        case 32: return launch_stream_typed<Policy, 32>(k_map, v_map, a, ctas, sms, stream);
        case 64: return launch_stream_typed<Policy, 64>(k_map, v_map, a, ctas, sms, stream);
        default: return launch_stream_typed<Policy, 128>(k_map, v_map, a, ctas, sms, stream);
    }
}

// Grid size and workspace carving shared by every policy; the policy for
// each query dtype is Policy<__half> / Policy<__nv_bfloat16>.
template <template <typename> class Policy>
cudaError_t launch_stream(const CUtensorMap& k_map, const CUtensorMap& v_map, DecodeArgs a,
                          pkv_dtype dtype, int block_size, cudaStream_t stream) {
    constexpr bool kFp8 = Policy<__half>::kFp8;
    constexpr int kTT = StreamLayout<kFp8, Policy<__half>::kWarps>::kTileTokens;
    int device = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&device);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (err != cudaSuccess) return err;
    // enough CTAs for ~kStreamTilesPerWarp tiles per warp, at most one per SM
    // (small batches are latency-bound: more warps, fewer tiles each)
    const int64_t max_tiles = static_cast<int64_t>(a.num_seqs) * a.num_kv_heads *
                              ((a.max_seq_len + kTT - 1) / kTT);
    constexpr int kWarps = Policy<__half>::kWarps;
    constexpr int64_t kPerCta = static_cast<int64_t>(kWarps) * kStreamTilesPerWarp;
    int64_t ctas = (max_tiles + kPerCta - 1) / kPerCta;
    const int cap = sms < kStreamMaxCtas ? sms : kStreamMaxCtas;
    if (ctas > cap) ctas = cap;
    if (ctas < 1) ctas = 1;
    a.num_warps = static_cast<int32_t>(ctas) * kWarps;
    // workspace layout: acc [rows][128], m [rows], l [rows]
    const size_t rows = (static_cast<size_t>(a.num_warps) +
                         static_cast<size_t>(a.num_seqs) * a.num_kv_heads) * a.group;
    float* ws = a.ws_acc;
    a.ws_m = ws + rows * kHeadDim;
    a.ws_l = a.ws_m + rows;
    return dtype == PKV_BF16
               ? launch_stream_block<Policy<__nv_bfloat16>>(k_map, v_map, a, block_size, (int)ctas,
                                                            sms, stream)
               : launch_stream_block<Policy<__half>>(k_map, v_map, a, block_size, (int)ctas, sms,
                                                     stream);
}

}  // namespace
}  // namespace pkv
