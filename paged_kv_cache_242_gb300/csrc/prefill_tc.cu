// Causal paged prefill attention on the fifth-generation tensor cores
// (tcgen05, operands and accumulators in tensor memory), for query groups
// that divide 128.
//
// What it computes is the same as prefill_attention.cu ("vLLM PagedAttention
// & continuous batching", "Prompt phase, decode phase"): the last q_len of
// sequence s's n cached tokens are queries at positions ctx + i
// (ctx = n - q_len), and query i attends to positions 0 .. ctx + i with
// softmax(scale * q K^T) V, accumulated key tile by key tile with the
// running max / running sum of Eq. (4) of "Serving Language Models Within a
// Memory Budget".
//
// Work items are (128-row tile, KV head, sequence); a row is one (query
// token, query head of the KV head's group) pair, token-major, so the group
// shares every key tile.  The grid is persistent (one CTA per SM): each CTA
// walks its share of the items with one running pipeline, so tensor memory,
// barriers and the K / V ring are set up once, and the next item's Q load
// and first S run while the previous item's output is written.  Ten warps
// with fixed roles:
//   warp 0     TMA producer: K and V tiles of 64 keys (64-column boxes of the
//              4-D pool view, 128-byte swizzle) into a six-stage ring;
//   warp 1     tensor-core issuer (one thread): S_j = Q K_j^T with Q read
//              from TMEM and K_j from shared memory, and O += P_j V_j with
//              P_j read from TMEM and V_j from shared memory, P split into a
//              bf16 / fp16 high part and the low part of the remainder (two
//              MMAs per step, so the weights keep about 16 significant bits);
//   warps 2-9  softmax, two threads per row (one TMEM lane each), each with
//              its own half of every key tile (keys 0-31 / 32-63), its own
//              running max / sum and its own O accumulator (the two halves
//              are split over keys and merged at the end by the same Eq. (4)
//              rule): read its 32 scores of S_j from TMEM, scale, causal mask,
//              max, weights, write P_j's two parts over those same 32 TMEM
//              columns, rescale the O row in TMEM when the max has grown by
//              more than 2^8 (until then the weights are taken against the
//              older, smaller max, which only lets them exceed 1); finally
//              merge and write O / l.
// S_{j+1} and P_{j-1} V_{j-1} run on the tensor cores while the softmax
// warps work on S_j.  Only K and V are read from shared memory by the MMAs.
//
// TMEM (32-bit columns): S_j / P_j buffers 0-63 and 64-127 (P as packed
// 16-bit pairs over the scores it replaces), the O of each key half 128-255
// and 256-383, Q 384-447 (packed pairs), the halves' final (m, l) 448-451.
// Shared memory: six stages of K + V (16 KiB each): 192 KiB.
#include <type_traits>

#include "pkv_internal.h"
#include "tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kRows = 128;                 // rows per CTA (the MMAs' M)
constexpr int kKeys = 64;                  // keys per tile (S's N, P V's K)
constexpr int kStages = 6;
constexpr int kKVHalf = kKeys * 128;       // 64 columns of a K or V tile: 8 KiB
constexpr int kTile = 2 * kKVHalf;         // a K or V tile: 16 KiB
constexpr int kCtlOff = kStages * 2 * kTile;  // 192 KiB
constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = (2 + kSoftmaxWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 128;      // O of key half c at + 128 c
constexpr uint32_t kQCol = 384;      // Q as 64 columns of packed pairs
constexpr uint32_t kStatCol = 448;   // (m, l) of key half c at + 2 c, + 2 c + 1
constexpr float kRescaleLog2 = 8.f;

struct alignas(8) TcControl {
    uint64_t q_full;
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_done[2];     // P_j V_j completed (j of that parity): O current, S / P buffer free
    uint64_t mma_done;
    uint64_t stat_ready;    // both halves of every row posted their (m, l)
    uint32_t tmem_base;
    int32_t valid[kStages];
};

constexpr size_t kSmemBytes = 1024 + kCtlOff + sizeof(TcControl);

// K tiles are the K-major B operand of S (64 dims per 128-byte row; k-step
// ks starts in half ks / 4 at byte (ks % 4) * 32); V tiles are the MN-major B
// operand of P V (rows are keys, the two halves hold dims 0-63 / 64-127 =
// the leading byte offset; k-step ks starts at key row 16 ks).  The issuer
// builds one descriptor per region and advances its address field by
// (bytes >> 4).

// The work list: item v = (h + H s) + H S x for row tile x (x = 0 is a
// sequence's last, longest row tile), KV head h and sequence s.  Every role
// of a CTA walks the same items v = blockIdx.x, + gridDim.x, ... and skips
// the same dead ones (x past the sequence's row tiles, or invalid lengths).
struct Item {
    int s, h, q0, ctx, rows_total, R0, n_tiles, first_lim, n;
};

__device__ __forceinline__ bool load_item(const PrefillArgs& a, int64_t v, int X, Item& it) {
    const int H = a.num_kv_heads;
    const int64_t hs = v % (static_cast<int64_t>(H) * a.num_seqs);
    const int x = static_cast<int>(v / (static_cast<int64_t>(H) * a.num_seqs));
    (void)X;
    it.s = static_cast<int>(hs / H);
    it.h = static_cast<int>(hs - static_cast<int64_t>(it.s) * H);
    it.q0 = __ldg(a.cu_q + it.s);
    const int q_len = __ldg(a.cu_q + it.s + 1) - it.q0;
    it.n = __ldg(a.seq_lens + it.s);
    if (it.n < 0 || it.n > a.max_seq_len || q_len < 0 || q_len > a.max_q_len || q_len > it.n)
        return false;
    const int g = a.group;
    it.ctx = it.n - q_len;
    it.rows_total = q_len * g;
    const int row_tiles = (it.rows_total + kRows - 1) / kRows;
    if (x >= row_tiles) return false;
    it.R0 = (row_tiles - 1 - x) * kRows;
    const int last_row = min(it.R0 + kRows, it.rows_total) - 1;
    it.n_tiles = (it.ctx + last_row / g + 1 + kKeys - 1) / kKeys;
    it.first_lim = it.ctx + it.R0 / g;
    return true;
}

template <typename T, int BS>
__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap k_map,
                            const __grid_constant__ CUtensorMap v_map, const PrefillArgs a,
                            int X) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    TcControl* ctl = reinterpret_cast<TcControl*>(sm + kCtlOff);
    const uint32_t s_base = smem_addr(sm);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = a.group;
    const int64_t n_items = static_cast<int64_t>(X) * a.num_kv_heads * a.num_seqs;

    if (threadIdx.x == 0) {
        prefetch_tensormap(&k_map);
        prefetch_tensormap(&v_map);
    }
    pdl_wait_prerequisites();
    pdl_allow_dependents();

    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&ctl->q_full), kSoftmaxWarps);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_addr(&ctl->kv_full[i]), 1);
            mbar_init(smem_addr(&ctl->kv_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&ctl->s_full[i]), 1);
            mbar_init(smem_addr(&ctl->p_full[i]), kSoftmaxWarps);
            mbar_init(smem_addr(&ctl->o_done[i]), 1);
        }
        mbar_init(smem_addr(&ctl->mma_done), 1);
        mbar_init(smem_addr(&ctl->stat_ready), kSoftmaxWarps);
        fence_barrier_init();
    }
    // every sequence's lengths are checked once, spread over the grid
    for (int s = blockIdx.x * kThreads + threadIdx.x; s < a.num_seqs; s += gridDim.x * kThreads) {
        const int q_len = __ldg(a.cu_q + s + 1) - __ldg(a.cu_q + s);
        const int n = __ldg(a.seq_lens + s);
        if (n < 0 || n > a.max_seq_len || q_len < 0 || q_len > a.max_q_len || q_len > n)
            report(a.err, PKV_DEVERR_BAD_SEQ_LEN);
    }
    if (warp == 1) tmem_alloc(smem_addr(&ctl->tmem_base), kTmemCols);
    tcgen05_before_sync();
    __syncthreads();
    tcgen05_after_sync();
    const uint32_t tmem = ctl->tmem_base;

    if (warp == 0) {
        // ============================ TMA producer ==============================
        constexpr int kBoxRows = BS < kKeys ? BS : kKeys;
        constexpr int kBlocksPerTile = BS < kKeys ? kKeys / BS : 1;
        int J = 0;  // tiles issued by this CTA over all its items
        bool alive = true;
        for (int64_t v = blockIdx.x; alive && v < n_items; v += gridDim.x) {
            Item it;
            if (!load_item(a, v, X, it)) continue;
            const int nblocks = (it.n + BS - 1) / BS;
            const int32_t* table = a.block_tables + static_cast<size_t>(it.s) * a.max_blocks_per_seq;
            int win_base = -(1 << 30), win_id = -1;
            for (int j = 0; j < it.n_tiles; ++j, ++J) {
                const int st = J % kStages;
                const int first_blk = (j * kKeys) / BS;
                const int last_blk = min(first_blk + kBlocksPerTile - 1, nblocks - 1);
                if (first_blk < win_base || last_blk >= win_base + 32) {
                    win_base = first_blk;
                    const int e = win_base + lane;
                    win_id = e < nblocks ? __ldg(table + e) : -1;
                }
                int ids[kBlocksPerTile];
                bool ok = true;
                uint32_t bytes = 0;
#pragma unroll
                for (int b = 0; b < kBlocksPerTile; ++b) {
                    const int blk = first_blk + b;
                    ids[b] = __shfl_sync(0xffffffffu, win_id, min(max(blk - win_base, 0), 31));
                    if (blk < nblocks) {  // blocks past the sequence end are not read
                        ok = ok && ids[b] >= 0 && ids[b] < a.num_blocks;
                        bytes += 4 * kBoxRows * 128;  // K and V, two halves each
                    }
                }
                int timed_out = 0;
                if (lane == 0 && J >= kStages &&
                    !mbar_wait(smem_addr(&ctl->kv_empty[st]), ((J - kStages) / kStages) & 1))
                    timed_out = 1;
                if (__shfl_sync(0xffffffffu, timed_out, 0)) {
                    if (lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
                    alive = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t full = smem_addr(&ctl->kv_full[st]);
                    ctl->valid[st] = ok ? 1 : 0;
                    if (ok) {
                        const uint32_t kb = s_base + st * 2 * kTile;
                        const uint32_t vb = kb + kTile;
                        const int row = (j * kKeys) % BS;  // 0 unless BS > 64
                        mbar_arrive_expect_tx(full, bytes);
#pragma unroll
                        for (int b = 0; b < kBlocksPerTile; ++b) {
                            if (first_blk + b >= nblocks) continue;
                            const uint32_t off = b * kBoxRows * 128;
                            tma_load_4d(kb + off, &k_map, full, 0, row, it.h, ids[b]);
                            tma_load_4d(kb + kKVHalf + off, &k_map, full, 64, row, it.h, ids[b]);
                            tma_load_4d(vb + off, &v_map, full, 0, row, it.h, ids[b]);
                            tma_load_4d(vb + kKVHalf + off, &v_map, full, 64, row, it.h, ids[b]);
                        }
                    } else {
                        report(a.err, PKV_DEVERR_BAD_BLOCK_ID);
                        mbar_arrive(full);
                    }
                }
                __syncwarp();
            }
        }
        if (lane == 0) {  // leave only once this CTA's copies have landed (bounded)
            const int first = J > kStages ? J - kStages : 0;
            for (int j = first; j < J; ++j)
                mbar_wait(smem_addr(&ctl->kv_full[j % kStages]), (j / kStages) & 1);
        }
    } else if (warp == 1) {
        // ============================ MMA issuer =================================
        // One stream of tiles J over all items: S_J is issued before
        // P_{J-1} V_{J-1}, except at the start of an item, where the last
        // P V of the previous item goes first (its epilogue is waiting for it).
        if (lane == 0) {
            constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
            constexpr uint32_t kIdS = umma_idesc_f16(kBf16, kRows, kKeys, false, false);
            constexpr uint32_t kIdO = umma_idesc_f16(kBf16, kRows, kHeadDim, false, true);
            const uint64_t dk = umma_desc_sw128(s_base, 16, 1024);
            const uint64_t dv = umma_desc_sw128(s_base + kTile, kKVHalf, 1024);
            const uint32_t k_lo = static_cast<uint32_t>(dk), k_hi = static_cast<uint32_t>(dk >> 32);
            const uint32_t v_lo = static_cast<uint32_t>(dv), v_hi = static_cast<uint32_t>(dv >> 32);
            bool alive = true;
            int J = 0, k = 0;
            bool pending = false;      // P_{J-1} V_{J-1} not issued yet
            bool pending_first = false;  // ... and it is its item's first tile
            auto issue_pv = [&](int jp, bool first_of_item) {
                const int stp = jp % kStages, pb = jp & 1;
                alive = mbar_wait(smem_addr(&ctl->p_full[pb]), (jp >> 1) & 1);
                if (!alive) return;
                tcgen05_after_sync();
                const uint32_t vs_lo = v_lo + ((stp * 2 * kTile) >> 4);
                const uint32_t first = first_of_item ? 0u : 1u;
                // P of key half c lives in columns 32 c .. + 31 of the buffer:
                // its high part in the first 16, the low part in the next 16
#pragma unroll
                for (int part = 0; part < 2; ++part) {
#pragma unroll
                    for (int ks = 0; ks < kKeys / 16; ++ks)
                        umma_f16_tmem_a(tmem + kOCol + 128 * (ks >> 1),
                                        tmem + pb * kKeys + 32 * (ks >> 1) + 16 * part + 8 * (ks & 1),
                                        vs_lo + ((ks * 16 * 128) >> 4), v_hi, kIdO,
                                        (part > 0 || (ks & 1)) ? 1u : first);
                }
                umma_commit(smem_addr(&ctl->o_done[pb]));
                umma_commit(smem_addr(&ctl->kv_empty[stp]));
            };
            for (int64_t v = blockIdx.x; alive && v < n_items; v += gridDim.x) {
                Item it;
                if (!load_item(a, v, X, it)) continue;
                // the previous item's last P V first, then this item's Q
                if (pending) {
                    issue_pv(J - 1, pending_first);
                    pending = false;
                    if (!alive) break;
                }
                alive = mbar_wait(smem_addr(&ctl->q_full), k & 1);
                if (!alive) break;
                tcgen05_after_sync();
                for (int j = 0; j < it.n_tiles; ++j, ++J) {
                    const int st = J % kStages, b = J & 1;
                    alive = mbar_wait(smem_addr(&ctl->kv_full[st]), (J / kStages) & 1);
                    // S / P buffer b is free once P_{J-2} V_{J-2} has completed
                    if (alive && J >= 2)
                        alive = mbar_wait(smem_addr(&ctl->o_done[b]), ((J - 2) >> 1) & 1);
                    if (!alive) break;
                    tcgen05_after_sync();
                    const uint32_t ks_lo = k_lo + ((st * 2 * kTile) >> 4);
#pragma unroll
                    for (int ks = 0; ks < kHeadDim / 16; ++ks)
                        umma_f16_tmem_a(tmem + b * kKeys, tmem + kQCol + 8 * ks,
                                        ks_lo + (((ks >> 2) * kKVHalf + (ks & 3) * 32) >> 4), k_hi,
                                        kIdS, ks > 0);
                    umma_commit(smem_addr(&ctl->s_full[b]));
                    if (pending) {  // P V of this item's previous tile
                        issue_pv(J - 1, pending_first);
                        if (!alive) break;
                    }
                    pending = true;
                    pending_first = j == 0;
                }
                ++k;
            }
            if (alive && pending) issue_pv(J - 1, pending_first);
            if (!alive) report(a.err, PKV_DEVERR_TIMEOUT);
            umma_commit(smem_addr(&ctl->mma_done));  // every MMA above has completed
            mbar_wait(smem_addr(&ctl->mma_done), 0);
        }
        __syncwarp();
    } else {
        // ============================ softmax warps ==============================
        // Warp 2 + 4 c + q (c = key half, q = lane quarter) owns TMEM lanes
        // 32 q .. + 31: S / P columns 32 c .. + 31 of each buffer, the O of key
        // half c, and Q / output dims 64 c .. + 63 (Q and the output only).
        const int quarter = warp & 3;  // TMEM lanes 32 quarter .. + 31 are this warp's
        const int half = (warp - 2) >> 2;
        const int r = quarter * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const float sl = a.scale_log2;
        bool alive = true;
        int J = 0, ep = 0;
        // the previous item's epilogue runs after the next item's Q is in place
        bool prev = false;
        bool prev_live = false;
        size_t prev_out = 0;
        float prev_m = -INFINITY, prev_l = 0.f;
        int prev_last = 0;  // global index of the previous item's last tile
        auto epilogue = [&]() {
            // ---- merge the two key halves (Eq. 4), O / l to the output ------
            const uint32_t st_addr = tmem + lane_base + kStatCol;
            alive = __all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->o_done[prev_last & 1]),
                                                      (prev_last >> 1) & 1));
            if (!alive) return;
            tcgen05_after_sync();
            tmem_st1(st_addr + 2 * half, __float_as_uint(prev_m));
            tmem_st1(st_addr + 2 * half + 1, __float_as_uint(prev_l));
            tmem_st_wait();
            tcgen05_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&ctl->stat_ready));
            alive = __all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->stat_ready), ep & 1));
            ++ep;
            if (!alive) return;
            tcgen05_after_sync();
            const float m0 = __uint_as_float(tmem_ld1(st_addr));
            const float l0 = __uint_as_float(tmem_ld1(st_addr + 1));
            const float m1 = __uint_as_float(tmem_ld1(st_addr + 2));
            const float l1 = __uint_as_float(tmem_ld1(st_addr + 3));
            tmem_ld_wait();
            const float mm = fmaxf(m0, m1);
            const float w0 = m0 == -INFINITY ? 0.f : ex2(m0 - mm);
            const float w1 = m1 == -INFINITY ? 0.f : ex2(m1 - mm);
            const float den = l0 * w0 + l1 * w1;
            const float inv = den > 0.f ? 1.f / den : 0.f;
            const float f0 = w0 * inv, f1 = w1 * inv;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(a.out) + prev_out) + 8 * half;
#pragma unroll 1
            for (int c2 = 0; c2 < 2; ++c2) {  // output dims 64 half + 32 c2 ..
                uint32_t oa[32], ob[32];
                tmem_ld32(tmem + lane_base + kOCol + 64 * half + 32 * c2, oa);
                tmem_ld32(tmem + lane_base + kOCol + 128 + 64 * half + 32 * c2, ob);
                tmem_ld_wait();
                if (prev_live) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = 8 * q + 2 * e;
                            w[e] = Mma<T>::pack(
                                __uint_as_float(oa[i]) * f0 + __uint_as_float(ob[i]) * f1,
                                __uint_as_float(oa[i + 1]) * f0 + __uint_as_float(ob[i + 1]) * f1);
                        }
                        dst[c2 * 4 + q] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            // O is read: the next item's first P V may overwrite it
            tcgen05_before_sync();
        };
        for (int64_t v = blockIdx.x; alive && v < n_items; v += gridDim.x) {
            Item it;
            if (!load_item(a, v, X, it)) continue;
            const int R = it.R0 + r;
            const bool live = R < it.rows_total;
            const int t = R / g;
            const int lim = live ? it.ctx + t : -1;  // last key this row sees
            const size_t out_row = (static_cast<size_t>(it.q0 + t) * a.num_q_heads +
                                    static_cast<size_t>(it.h) * g + R % g) *
                                   kHeadDim;
            // ---- dims 64 half .. + 63 of Q row r into TMEM (zeros past the last
            // row); every S of the previous item has completed (its last s_full
            // was waited for), so its Q may be overwritten
            {
                const uint4* src =
                    reinterpret_cast<const uint4*>(static_cast<const T*>(a.q) + out_row) + 8 * half;
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 q4 = live ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
                    w[4 * c] = q4.x;
                    w[4 * c + 1] = q4.y;
                    w[4 * c + 2] = q4.z;
                    w[4 * c + 3] = q4.w;
                }
                tmem_st32(tmem + lane_base + kQCol + 32 * half, w);
                tmem_st_wait();
                tcgen05_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&ctl->q_full));
            }
            if (prev) {
                epilogue();
                if (!alive) break;
            }
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < it.n_tiles; ++j, ++J) {
                const int b = J & 1, st = J % kStages;
                if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->s_full[b]), (J >> 1) & 1))) {
                    alive = false;
                    break;
                }
                tcgen05_after_sync();
                const int key0 = j * kKeys + 32 * half;
                const bool masked = j * kKeys + kKeys - 1 > it.first_lim;
                const uint32_t sp_addr = tmem + lane_base + b * kKeys + 32 * half;
                uint32_t v[32];
                tmem_ld32(sp_addr, v);
                tmem_ld_wait();
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float x = __uint_as_float(v[i]) * sl;
                    if (masked) x = key0 + i <= lim ? x : -INFINITY;  // also drops NaN
                    mx[i & 3] = fmaxf(mx[i & 3], x);
                }
                const float row_max = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                // lazy rescale: keep the older max until this half's max exceeds it by 2^8
                const float m_new = fmaxf(m_used, row_max);
                const bool bump = m_new > m_used + kRescaleLog2;  // true at the first finite max
                const float m_tgt = bump ? m_new : m_used;
                const float base = m_tgt == -INFINITY ? 0.f : m_tgt;
                const float alpha = bump ? ex2(m_used - base) : 1.f;  // 0 while m_used = -inf
                m_used = m_tgt;

                if (j >= 1 && __any_sync(0xffffffffu, bump)) {
                    // O must hold P_{J-1} V_{J-1} before it is rescaled
                    if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->o_done[(J - 1) & 1]),
                                                           ((J - 1) >> 1) & 1))) {
                        alive = false;
                        break;
                    }
                    tcgen05_after_sync();
#pragma unroll 1
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint32_t ov[32];
                        const uint32_t o_addr = tmem + lane_base + kOCol + 128 * half + 32 * c4;
                        tmem_ld32(o_addr, ov);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tmem_st32(o_addr, ov);
                    }
                    tmem_st_wait();
                }
                // V rows of keys past the sequence end hold stale bytes: zero them
                if (j * kKeys + kKeys > it.n) {
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(smem_addr(&ctl->kv_full[st]), (J / kStages) & 1))) {
                        alive = false;
                        break;
                    }
                    if (r < kKeys && j * kKeys + r >= it.n) {
                        const uint32_t vrow =
                            s_base + st * 2 * kTile + kTile + half * kKVHalf + r * 128;
                        asm volatile(
                            "{\n\t.reg .b32 z;\n\tmov.b32 z, 0;\n\t"
                            "st.shared.v4.b32 [%0], {z, z, z, z};\n\tst.shared.v4.b32 [%0+16], {z, z, z, z};\n\t"
                            "st.shared.v4.b32 [%0+32], {z, z, z, z};\n\tst.shared.v4.b32 [%0+48], {z, z, z, z};\n\t"
                            "st.shared.v4.b32 [%0+64], {z, z, z, z};\n\tst.shared.v4.b32 [%0+80], {z, z, z, z};\n\t"
                            "st.shared.v4.b32 [%0+96], {z, z, z, z};\n\tst.shared.v4.b32 [%0+112], {z, z, z, z};\n\t}"
                            ::"r"(vrow) : "memory");
                    }
                    fence_proxy_async_shared();
                }
                // ---- weights, their sum, P's high / low parts over these 32 columns ----
                float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float x = fmaf(__uint_as_float(v[i]), sl, -base);
                    if (masked) x = key0 + i <= lim ? x : -INFINITY;
                    const float p = ex2(x);
                    ps[i & 3] += p;
                    v[i] = __float_as_uint(p);
                }
                uint32_t pw[32];  // high parts of keys 0-31 of this half, then the low parts
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float p0 = __uint_as_float(v[2 * e]), p1 = __uint_as_float(v[2 * e + 1]);
                    pw[e] = Mma<T>::pack(p0, p1);
                    const float2 back = Mma<T>::unpack(pw[e]);
                    pw[16 + e] = Mma<T>::pack(p0 - back.x, p1 - back.y);
                }
                tmem_st32(sp_addr, pw);
                tmem_st_wait();
                l = l * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
                tcgen05_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&ctl->p_full[b]));
            }
            prev = true;
            prev_live = live;
            prev_out = out_row;
            prev_m = m_used;
            prev_l = l;
            prev_last = J - 1;
        }
        if (alive && prev) epilogue();
        if (!alive && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
    }

    // every role is done with TMEM (the issuer waited for its last MMA)
    tcgen05_before_sync();
    __syncthreads();
    if (warp == 1) {
        tcgen05_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <typename T, int BS>
cudaError_t launch_tc_typed(const CUtensorMap& k_map, const CUtensorMap& v_map,
                            const PrefillArgs& a, cudaStream_t stream) {
    cudaError_t err = ensure_smem_limit<paged_prefill_tc_kernel<T, BS>>(kSmemBytes);
    if (err != cudaSuccess) return err;
    const int64_t row_tiles = (static_cast<int64_t>(a.max_q_len) * a.group + kRows - 1) / kRows;
    const int X = static_cast<int>(row_tiles > 0 ? row_tiles : 1);
    const int64_t items = static_cast<int64_t>(X) * a.num_kv_heads * a.num_seqs;
    int device = 0, sms = 0;
    err = cudaGetDevice(&device);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (err != cudaSuccess) return err;
    // persistent: one CTA per SM walks the work list
    const int ctas = static_cast<int>(items < sms ? items : sms);
    return launch_pdl(paged_prefill_tc_kernel<T, BS>, dim3(ctas > 0 ? ctas : 1), dim3(kThreads),
                      kSmemBytes, stream, k_map, v_map, a, X);
}

template <typename T>
cudaError_t launch_tc_dtype(const CUtensorMap& k_map, const CUtensorMap& v_map,
                            const PrefillArgs& a, int block_size, cudaStream_t stream) {
    switch (block_size) {
        case 8: return launch_tc_typed<T, 8>(k_map, v_map, a, stream);
        case 16: return launch_tc_typed<T, 16>(k_map, v_map, a, stream);
        case 32: return launch_tc_typed<T, 32>(k_map, v_map, a, stream);
        case 64: return launch_tc_typed<T, 64>(k_map, v_map, a, stream);
        default: return launch_tc_typed<T, 128>(k_map, v_map, a, stream);
    }
}

}  // namespace

bool prefill_tc_supported(int group) { return group >= 1 && group <= kRows && kRows % group == 0; }

int prefill_tc_box_rows(int block_size) { return block_size < kKeys ? block_size : kKeys; }

cudaError_t launch_paged_prefill_tc(const CUtensorMap& k_map, const CUtensorMap& v_map,
                                    const PrefillArgs& args, pkv_dtype dtype, int block_size,
                                    cudaStream_t stream) {
    return dtype == PKV_BF16
               ? launch_tc_dtype<__nv_bfloat16>(k_map, v_map, args, block_size, stream)
               : launch_tc_dtype<__half>(k_map, v_map, args, block_size, stream);
}

}  // namespace pkv
