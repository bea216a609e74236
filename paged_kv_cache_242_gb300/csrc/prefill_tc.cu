// Causal paged prefill attention on the fifth-generation tensor cores
// (tcgen05, accumulators in tensor memory), for query groups that divide 128.
//
// What it computes is the same as prefill_attention.cu ("vLLM PagedAttention
// & continuous batching", "Prompt phase, decode phase"): the last q_len of
// sequence s's n cached tokens are queries at positions ctx + i
// (ctx = n - q_len), and query i attends to positions 0 .. ctx + i with
// softmax(scale * q K^T) V, accumulated key tile by key tile with the
// running max / running sum of Eq. (4) of "Serving Language Models Within a
// Memory Budget".
//
// Work items are (256-row tile, KV head, sequence); a row is one (query
// token, query head of the KV head's group) pair, token-major, so the group
// shares every key tile.  An item is two 128-row Q tiles, A and B, that share
// every K / V tile: one copy of a tile feeds both.  The grid is persistent
// (one CTA per SM): each CTA walks its share of the items with one running
// pipeline, so tensor memory, barriers and the K / V ring are set up once.
// Eleven warps with fixed roles:
//   warp 0     TMA producer: K and V tiles of 64 keys (64-column boxes of the
//              4-D pool view, 128-byte swizzle) into a four-stage ring; once a
//              copy holding keys past the sequence end has landed it zeroes
//              those V rows (stale slots may hold NaN), then releases the
//              stage to the P V MMAs;
//   warps 1-2  tensor-core issuers (one thread each), warp 1 for Q tile A and
//              warp 2 for B: for each key tile S = Q K^T (Q and K from shared
//              memory), then O += P V of the previous key tile (P read from
//              tensor memory, V from shared memory).  With bf16 inputs P is
//              split into a bf16 high part (its top 16 bits) and the rounded
//              remainder (two MMAs per step, so the weights keep about 16
//              significant bits); with fp16 inputs P is one binary16 value (11 bits).  With an
//              issuer per tile neither tile's S waits behind the other's
//              softmax;
//   warps 3-6  softmax of Q tile A, warps 7-10 of Q tile B, one thread per row
//              (one TMEM lane): read the row's 64 scores of S from TMEM,
//              scale, causal mask, weights, write P's parts over
//              those TMEM columns.  Once the row has a finite running max the
//              weights are taken against it without a max pass; a tile whose
//              weights would sum past kMaxTileSum moves the max (by the scores'
//              max, when it has grown by more than 2^8) and rescales the O row
//              in TMEM and the sum.  At the end of the item write O / l.
// While one Q tile's softmax runs, the tensor cores work on the other's S or
// P V and on the next S of the same tile (two S / P buffers per tile).
//
// TMEM (512 32-bit columns): Q tile q uses 256 q .. 256 q + 255: S / P
// buffers at + 0 and + 64, O at + 128.  Shared memory: four stages of K + V
// (16 KiB each) and the two 128 x 128 Q tiles: 192 KiB.
#include <type_traits>

#include "pkv_internal.h"
#include "tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kTileRows = 128;              // rows per Q tile (the MMAs' M)
constexpr int kItemRows = 2 * kTileRows;    // rows per work item
constexpr int kKeys = 64;                   // keys per tile (S's N, P V's K)
constexpr int kStages = 4;
constexpr int kKVHalf = kKeys * 128;        // 64 columns of a K or V tile: 8 KiB
constexpr int kTile = 2 * kKVHalf;          // a K or V tile: 16 KiB
constexpr int kQHalf = kTileRows * 128;     // 64 columns of a Q tile: 16 KiB
constexpr int kQBytes = 2 * kQHalf;         // a Q tile: 32 KiB
constexpr int kQOff = kStages * 2 * kTile;  // 128 KiB
constexpr int kCtlOff = kQOff + 2 * kQBytes;  // 192 KiB
constexpr int kSoftmaxWarps = 8;            // four per Q tile
constexpr int kFirstSoftmaxWarp = 3;        // warp 0 producer, warps 1-2 issuers
constexpr int kThreads = (kFirstSoftmaxWarp + kSoftmaxWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemPerTile = 256;      // S / P buffers + 0, + 64; O + 128
constexpr uint32_t kOCol = 128;
constexpr float kRescaleLog2 = 8.f;

// P's 16-bit parts: bf16 keeps 8 significant bits, so P is split into a high
// part (the top 16 bits of the fp32 weight, a bf16 value exactly) and the
// exact remainder rounded to bf16; binary16 keeps 11 and goes whole.
template <typename T>
constexpr int kPParts = std::is_same<T, __nv_bfloat16>::value ? 2 : 1;

// The largest sum of a tile's weights taken against a stale running max
// before the max is moved: weights stay well inside the 16-bit type's range
// (bf16: 2^127; binary16: 65504).
template <typename T>
constexpr float kMaxTileSum = std::is_same<T, __nv_bfloat16>::value ? 4294967296.f : 32768.f;

// max(a, b, c) in one instruction (sm_100+); a NaN input is ignored as in fmaxf.
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Packed two-lane fp32 arithmetic (one sm_100+ .f32x2 instruction for a
// pair).  A packed multiply whose result feeds a packed add or subtract may be
// evaluated as one fused operation, without the product's rounding, so they
// are used only where no multiply feeds an add: the scale before the max, the
// exponent argument (an explicit fma), the sums of weights and the low part
// of P (the weight minus its bit-truncated high part).
__device__ __forceinline__ void mul2(float& d0, float& d1, float a0, float a1, float b) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %4};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b));
}
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b, float c) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %4};\n\t"
        "mov.b64 rc, {%5, %5};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void sub2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

struct alignas(8) TcControl {
    uint64_t q_full[2];     // [Q tile]: its rows are in shared memory (4 warps)
    uint64_t kv_full[kStages];
    uint64_t v_clean[kStages];   // V rows past the sequence end are zero (producer)
    uint64_t kv_empty[kStages];  // both issuers' MMAs of the stage completed
    uint64_t s_full[2][2];  // [Q tile][buffer]
    uint64_t p_full[2][2];  // 4 warps
    uint64_t o_done[2][2];  // P V of that buffer completed: O current, buffer free
    uint64_t mma_done[2];   // [issuer]
    uint32_t tmem_base;
};

// Each sequence's number of row items, cached in shared memory so that dead
// items of the work list are skipped without global loads (up to
// kCachedSeqs sequences with fewer than 2^16 row items each).
constexpr int kCachedSeqs = 4096;
constexpr int kRowItemsOff = (kCtlOff + static_cast<int>(sizeof(TcControl)) + 15) / 16 * 16;
constexpr size_t kSmemMaxBytes = 1024 + kRowItemsOff + kCachedSeqs * sizeof(uint16_t);
static_assert(kSmemMaxBytes <= 232448, "shared memory per CTA");

// Dynamic shared memory of a launch: the cache holds this call's sequences.
inline size_t smem_bytes(int num_seqs) {
    const int cached = num_seqs <= kCachedSeqs ? num_seqs : 0;
    return 1024 + kRowItemsOff + static_cast<size_t>(cached) * sizeof(uint16_t);
}

// K tiles and Q tiles are K-major operands (64 dims per 128-byte row; k-step
// ks starts in half ks / 4 at byte (ks % 4) * 32); V tiles are the MN-major B
// operand of P V (rows are keys, the two halves hold dims 0-63 / 64-127 =
// the leading byte offset; k-step ks starts at key row 16 ks).  The issuer
// builds one descriptor per region and advances its address field by
// (bytes >> 4).

// The work list: item v = (h + H s) + H S x for row item x (x = 0 is a
// sequence's last, longest one), KV head h and sequence s.  Every role of a
// CTA walks the same items v = blockIdx.x, + gridDim.x, ... and skips the
// same dead ones (x past the sequence's rows, or invalid lengths).
struct Item {
    int s, h, q0, ctx, rows_total, R0, n, n_keys;
    int n_tiles[2];    // key tiles of Q tile A / B (0: B holds no row)
    int first_lim[2];  // the smallest causal limit among the tile's rows
};

// The row items of sequence s: ceil(q_len * group / 256), 0 when its lengths
// are invalid.
__device__ __forceinline__ int seq_row_items(const PrefillArgs& a, int s) {
    const int q_len = __ldg(a.cu_q + s + 1) - __ldg(a.cu_q + s);
    const int n = __ldg(a.seq_lens + s);
    if (n < 0 || n > a.max_seq_len || q_len < 0 || q_len > a.max_q_len || q_len > n) return 0;
    return static_cast<int>((static_cast<int64_t>(q_len) * a.group + kItemRows - 1) / kItemRows);
}

// `cache`: the shared-memory copy of seq_row_items, or null.
__device__ __forceinline__ bool load_item(const PrefillArgs& a, int64_t v, Item& it,
                                          const uint16_t* cache) {
    const int H = a.num_kv_heads;
    const int64_t hs = v % (static_cast<int64_t>(H) * a.num_seqs);
    const int x = static_cast<int>(v / (static_cast<int64_t>(H) * a.num_seqs));
    it.s = static_cast<int>(hs / H);
    it.h = static_cast<int>(hs - static_cast<int64_t>(it.s) * H);
    if (cache != nullptr && x >= cache[it.s]) return false;  // dead: no global loads
    it.q0 = __ldg(a.cu_q + it.s);
    const int q_len = __ldg(a.cu_q + it.s + 1) - it.q0;
    it.n = __ldg(a.seq_lens + it.s);
    if (it.n < 0 || it.n > a.max_seq_len || q_len < 0 || q_len > a.max_q_len || q_len > it.n)
        return false;
    const int g = a.group;
    it.ctx = it.n - q_len;
    it.rows_total = q_len * g;
    const int row_items = (it.rows_total + kItemRows - 1) / kItemRows;
    if (x >= row_items) return false;
    it.R0 = (row_items - 1 - x) * kItemRows;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int rq = it.R0 + q * kTileRows;
        if (rq >= it.rows_total) {
            it.n_tiles[q] = 0;
            it.first_lim[q] = 0;
        } else {
            const int last_row = min(rq + kTileRows, it.rows_total) - 1;
            it.n_tiles[q] = (it.ctx + last_row / g + 1 + kKeys - 1) / kKeys;
            it.first_lim[q] = it.ctx + rq / g;
        }
    }
    it.n_keys = max(it.n_tiles[0], it.n_tiles[1]);
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
        for (int q = 0; q < 2; ++q) {
            mbar_init(smem_addr(&ctl->q_full[q]), kSoftmaxWarps / 2);
            for (int b = 0; b < 2; ++b) {
                mbar_init(smem_addr(&ctl->s_full[q][b]), 1);
                mbar_init(smem_addr(&ctl->p_full[q][b]), kSoftmaxWarps / 2);
                mbar_init(smem_addr(&ctl->o_done[q][b]), 1);
            }
        }
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_addr(&ctl->kv_full[i]), 1);
            mbar_init(smem_addr(&ctl->v_clean[i]), 1);
            mbar_init(smem_addr(&ctl->kv_empty[i]), 2);
        }
        mbar_init(smem_addr(&ctl->mma_done[0]), 1);
        mbar_init(smem_addr(&ctl->mma_done[1]), 1);
        fence_barrier_init();
    }
    // every CTA caches the row items of every sequence (when they fit)
    uint16_t* row_items_smem = reinterpret_cast<uint16_t*>(sm + kRowItemsOff);
    const uint16_t* row_items = (a.num_seqs <= kCachedSeqs && X < 65536) ? row_items_smem : nullptr;
    if (row_items != nullptr) {
        for (int s = threadIdx.x; s < a.num_seqs; s += kThreads)
            row_items_smem[s] = static_cast<uint16_t>(min(seq_row_items(a, s), 65535));
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
        int J = 0;  // key tiles issued by this CTA over all its items
        bool alive = true;
        for (int64_t v = blockIdx.x; alive && v < n_items; v += gridDim.x) {
            Item it;
            if (!load_item(a, v, it, row_items)) continue;
            const int nblocks = (it.n + BS - 1) / BS;
            const int32_t* table = a.block_tables + static_cast<size_t>(it.s) * a.max_blocks_per_seq;
            int win_base = -(1 << 30), win_id = -1;
            for (int j = 0; j < it.n_keys; ++j, ++J) {
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
                // V rows of keys past the sequence end hold stale bytes: once the
                // copy has landed, zero them before any P V reads the stage
                const uint32_t clean = smem_addr(&ctl->v_clean[st]);
                if (j * kKeys + kKeys > it.n) {
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(smem_addr(&ctl->kv_full[st]), (J / kStages) & 1))) {
                        if (lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
                        alive = false;
                        break;
                    }
                    const int stale0 = it.n - j * kKeys;  // first stale key row (>= 0)
                    uint8_t* vt = sm + st * 2 * kTile + kTile;
                    for (int i = lane; i < 2 * kKeys * 8; i += 32) {  // (half, row, 16-byte chunk)
                        const int hf = i / (kKeys * 8), row = (i / 8) % kKeys, c = i % 8;
                        if (row >= stale0)
                            reinterpret_cast<uint4*>(vt + hf * kKVHalf + row * 128)[c] =
                                make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_shared();
                    __syncwarp();
                }
                if (lane == 0) mbar_arrive(clean);
                __syncwarp();
            }
        }
        if (lane == 0) {  // leave only once this CTA's copies have landed (bounded)
            const int first = J > kStages ? J - kStages : 0;
            for (int j = first; j < J; ++j)
                mbar_wait(smem_addr(&ctl->kv_full[j % kStages]), (j / kStages) & 1);
        }
    } else if (warp < kFirstSoftmaxWarp) {
        // ========================== MMA issuers (one per Q tile) ===================
        // Warp 1 issues Q tile A's MMAs, warp 2 Q tile B's: for each key tile,
        // S of this Q tile, then P V of its previous key tile.  Neither waits for
        // the other tile's softmax.  Each commits every key tile's stage release
        // once (after its last MMA that reads the stage, at once if it reads
        // none); waiting for every key tile's copy keeps both within one ring.
        const int q = warp - 1;
        if (lane == 0) {
            constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
            constexpr uint32_t kIdS = umma_idesc_f16(kBf16, kTileRows, kKeys, false, false);
            constexpr uint32_t kIdO = umma_idesc_f16(kBf16, kTileRows, kHeadDim, false, true);
            const uint64_t dq = umma_desc_sw128(s_base + kQOff + q * kQBytes, 16, 1024);
            const uint64_t dk = umma_desc_sw128(s_base, 16, 1024);
            const uint64_t dv = umma_desc_sw128(s_base + kTile, kKVHalf, 1024);
            const uint32_t q_lo = static_cast<uint32_t>(dq), q_hi = static_cast<uint32_t>(dq >> 32);
            const uint32_t k_lo = static_cast<uint32_t>(dk), k_hi = static_cast<uint32_t>(dk >> 32);
            const uint32_t v_lo = static_cast<uint32_t>(dv), v_hi = static_cast<uint32_t>(dv >> 32);
            const uint32_t tq = tmem + q * kTmemPerTile;
            bool alive = true;
            int J = 0;      // key tiles over all items (the ring)
            int Tq = 0;     // tiles of this Q tile over all items (its buffers)
            int Kq = 0;     // items in which this Q tile holds rows (q_full phases)
            bool pend = false, pend_first = false;
            int pend_t = 0, pend_j = 0;
            // P V of the pending tile, then the release of its stage
            auto flush = [&]() {
                if (!pend) return;
                const int stp = pend_j % kStages, pb = pend_t & 1;
                alive = mbar_wait(smem_addr(&ctl->p_full[q][pb]), (pend_t >> 1) & 1) &&
                        mbar_wait(smem_addr(&ctl->v_clean[stp]), (pend_j / kStages) & 1);
                if (!alive) return;
                tcgen05_after_sync();
                const uint32_t vs_lo = v_lo + ((stp * 2 * kTile) >> 4);
                const uint32_t first = pend_first ? 0u : 1u;
#pragma unroll
                for (int part = 0; part < kPParts<T>; ++part) {
#pragma unroll
                    for (int ks = 0; ks < kKeys / 16; ++ks)
                        umma_f16_tmem_a(tq + kOCol, tq + 64 * pb + 32 * part + 8 * ks,
                                        vs_lo + ((ks * 16 * 128) >> 4), v_hi, kIdO,
                                        (part > 0 || ks > 0) ? 1u : first);
                }
                umma_commit(smem_addr(&ctl->o_done[q][pb]));
                umma_commit(smem_addr(&ctl->kv_empty[stp]));
                pend = false;
            };
            for (int64_t v = blockIdx.x; alive && v < n_items; v += gridDim.x) {
                Item it;
                if (!load_item(a, v, it, row_items)) continue;
                flush();  // the previous item's last P V (its epilogue waits for it)
                if (!alive) break;
                const int n_t = q ? it.n_tiles[1] : it.n_tiles[0];
                if (n_t > 0) {
                    alive = mbar_wait(smem_addr(&ctl->q_full[q]), Kq & 1);
                    ++Kq;
                    if (!alive) break;
                    tcgen05_after_sync();
                }
                for (int j = 0; j < it.n_keys; ++j, ++J) {
                    const int st = J % kStages;
                    alive = mbar_wait(smem_addr(&ctl->kv_full[st]), (J / kStages) & 1);
                    if (!alive) break;
                    if (j < n_t) {
                        const int t = Tq, b = t & 1;
                        // S / P buffer b is free once the P V two tiles back has completed
                        if (t >= 2)
                            alive = mbar_wait(smem_addr(&ctl->o_done[q][b]), ((t - 2) >> 1) & 1);
                        if (!alive) break;
                        tcgen05_after_sync();
                        const uint32_t ks_lo = k_lo + ((st * 2 * kTile) >> 4);
#pragma unroll
                        for (int ks = 0; ks < kHeadDim / 16; ++ks) {
                            const uint32_t kadv = ((ks >> 2) * kKVHalf + (ks & 3) * 32) >> 4;
                            const uint32_t qadv = ((ks >> 2) * kQHalf + (ks & 3) * 32) >> 4;
                            umma_f16_lo(tq + 64 * b, q_lo + qadv, q_hi, ks_lo + kadv, k_hi, kIdS,
                                        ks > 0 ? 1u : 0u);
                        }
                        umma_commit(smem_addr(&ctl->s_full[q][b]));
                        flush();  // P V of this tile's previous key tile
                        if (!alive) break;
                        pend = true;
                        pend_first = j == 0;
                        pend_t = Tq++;
                        pend_j = J;
                    } else {
                        flush();
                        if (!alive) break;
                        umma_commit(smem_addr(&ctl->kv_empty[st]));  // reads nothing of it
                    }
                }
            }
            if (alive) flush();
            if (!alive) report(a.err, PKV_DEVERR_TIMEOUT);
            umma_commit(smem_addr(&ctl->mma_done[q]));  // every MMA above has completed
            mbar_wait(smem_addr(&ctl->mma_done[q]), 0);
        }
        __syncwarp();
    } else {
        // ============================ softmax warps ==============================
        // Warps 3-6 serve Q tile A, 7-10 Q tile B; warp w owns TMEM lanes
        // 32 (w % 4) .. + 31 = rows of its tile.
        const int qt = (warp - kFirstSoftmaxWarp) >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // row within the Q tile
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tbase = tmem + lane_base + qt * kTmemPerTile;
        const float sl = a.scale_log2;
        bool alive = true;
        int J = 0;    // key tiles over all items (ring stages)
        int Tt = 0;   // tiles of this Q tile over all items (its buffers)
        bool prev = false, prev_live = false;
        size_t prev_out = 0;
        float prev_l = 0.f;
        int prev_last = 0;
        auto epilogue = [&]() {
            // ---- O / l to the output row ----------------------------------------
            alive = __all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->o_done[qt][prev_last & 1]),
                                                      (prev_last >> 1) & 1));
            if (!alive) return;
            tcgen05_after_sync();
            const float inv = prev_l > 0.f ? 1.f / prev_l : 0.f;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(a.out) + prev_out);
#pragma unroll 1
            for (int c4 = 0; c4 < 4; ++c4) {  // output dims 32 c4 ..
                uint32_t o[32];
                tmem_ld32(tbase + kOCol + 32 * c4, o);
                tmem_ld_wait();
                if (prev_live) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = 8 * q + 2 * e;
                            w[e] = Mma<T>::pack(__uint_as_float(o[i]) * inv,
                                                __uint_as_float(o[i + 1]) * inv);
                        }
                        dst[c4 * 4 + q] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            // O is read: the next item's first P V may overwrite it
            tcgen05_before_sync();
        };
        for (int64_t v = blockIdx.x; alive && v < n_items; v += gridDim.x) {
            Item it;
            if (!load_item(a, v, it, row_items)) continue;
            J += it.n_keys;
            const int n_t = qt ? it.n_tiles[1] : it.n_tiles[0];
            const int first_lim = qt ? it.first_lim[1] : it.first_lim[0];
            if (n_t == 0) continue;  // this Q tile holds no row of the item
            const int R = it.R0 + qt * kTileRows + r;
            const bool live = R < it.rows_total;
            const int t = R / g;
            const int lim = live ? it.ctx + t : -1;  // last key this row sees
            const size_t out_row = (static_cast<size_t>(it.q0 + t) * a.num_q_heads +
                                    static_cast<size_t>(it.h) * g + R % g) *
                                   kHeadDim;
            // ---- Q row r into shared memory (128-byte swizzle: chunk c of row r
            // at chunk c ^ (r % 8)), zeros past the last row; every S of this
            // tile's previous item has completed, so its Q may be overwritten
            {
                const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(a.q) + out_row);
                uint8_t* qtile = sm + kQOff + qt * kQBytes + r * 128;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint4 q4 = live ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
                    reinterpret_cast<uint4*>(qtile + (c >> 3) * kQHalf)[(c & 7) ^ (r & 7)] = q4;
                }
                fence_proxy_async_shared();  // generic writes -> the tensor cores' reads
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&ctl->q_full[qt]));
            }
            if (prev) {
                epilogue();
                if (!alive) break;
            }
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < n_t; ++j, ++Tt) {
                const int b = Tt & 1;
                if (!__all_sync(0xffffffffu,
                                mbar_wait(smem_addr(&ctl->s_full[qt][b]), (Tt >> 1) & 1))) {
                    alive = false;
                    break;
                }
                tcgen05_after_sync();
                const int key0 = j * kKeys;
                const bool masked = j * kKeys + kKeys - 1 > first_lim;
                const uint32_t sp_addr = tbase + 64 * b;
                uint32_t v[64];
                tmem_ld32(sp_addr, *reinterpret_cast<uint32_t(*)[32]>(v));
                tmem_ld32(sp_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
                tmem_ld_wait();
                // ---- weights against the running max, and their sum ----
                // Once a row has a finite max, its weights are taken against it
                // without a max pass: they stay exact in fp32, and P keeps the same
                // relative precision at any size.  Only a tile whose weights sum past
                // kMaxTileSum (or a row without a finite max yet) takes the pass
                // below, which moves the max and rescales O and the sum.
                float ps[4] = {0.f, 0.f, 0.f, 0.f};
                auto weights = [&](float base) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) ps[k] = 0.f;
#pragma unroll
                    for (int i = 0; i < 64; i += 2) {
                        float x0, x1;
                        fma2(x0, x1, __uint_as_float(v[i]), __uint_as_float(v[i + 1]), sl, -base);
                        if (masked) {
                            x0 = key0 + i <= lim ? x0 : -INFINITY;
                            x1 = key0 + i + 1 <= lim ? x1 : -INFINITY;
                        }
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        const int a2 = (i >> 1) & 1;
                        add2(ps[2 * a2], ps[2 * a2 + 1], ps[2 * a2], ps[2 * a2 + 1], p0, p1);
                        v[i] = __float_as_uint(p0);
                        v[i + 1] = __float_as_uint(p1);
                    }
                };
                float alpha = 1.f;
                bool need_max = __any_sync(0xffffffffu, m_used == -INFINITY);
                if (!need_max) {
                    weights(m_used);
                    const float sum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
                    need_max = __any_sync(0xffffffffu, !(sum <= kMaxTileSum<T>));
                    if (need_max) {  // the scores again, for the pass below
                        tmem_ld32(sp_addr, *reinterpret_cast<uint32_t(*)[32]>(v));
                        tmem_ld32(sp_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
                        tmem_ld_wait();
                    }
                }
                if (need_max) {
                    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int i = 0; i < 64; i += 2) {
                        float x0, x1;
                        mul2(x0, x1, __uint_as_float(v[i]), __uint_as_float(v[i + 1]), sl);
                        if (masked) {
                            x0 = key0 + i <= lim ? x0 : -INFINITY;  // also drops NaN
                            x1 = key0 + i + 1 <= lim ? x1 : -INFINITY;
                        }
                        mx[(i >> 1) & 3] = max3(mx[(i >> 1) & 3], x0, x1);
                    }
                    const float row_max = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                    // lazy rescale: keep the older max until the row max exceeds it by 2^8
                    const float m_new = fmaxf(m_used, row_max);
                    const bool bump = m_new > m_used + kRescaleLog2;  // true at the first finite max
                    const float m_tgt = bump ? m_new : m_used;
                    const float base = m_tgt == -INFINITY ? 0.f : m_tgt;
                    alpha = bump ? ex2(m_used - base) : 1.f;  // 0 while m_used = -inf
                    m_used = m_tgt;
                    if (j >= 1 && __any_sync(0xffffffffu, bump)) {
                        // O must hold the previous tile's P V before it is rescaled
                        if (!__all_sync(0xffffffffu,
                                        mbar_wait(smem_addr(&ctl->o_done[qt][(Tt - 1) & 1]),
                                                  ((Tt - 1) >> 1) & 1))) {
                            alive = false;
                            break;
                        }
                        tcgen05_after_sync();
#pragma unroll 1
                        for (int c4 = 0; c4 < 4; ++c4) {
                            uint32_t ov[32];
                            const uint32_t o_addr = tbase + kOCol + 32 * c4;
                            tmem_ld32(o_addr, ov);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                            tmem_st32(o_addr, ov);
                        }
                        tmem_st_wait();
                    }
                    weights(base);
                }
                uint32_t pw[32];
                if constexpr (kPParts<T> == 2) {
                    // High part: the weight cut to its top 16 bits, a bf16 value
                    // exactly, paired by one byte permute.  Low part: the exact
                    // fp32 remainder (below 2^-7 of the weight), rounded to bf16,
                    // so the pair carries the weight within 2^-16 of it.  This takes
                    // one conversion per pair instead of two plus an unpack.
                    uint32_t lw[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const uint32_t h0 = v[2 * e] & 0xFFFF0000u, h1 = v[2 * e + 1] & 0xFFFF0000u;
                        pw[e] = __byte_perm(v[2 * e], v[2 * e + 1], 0x7632);
                        float r0, r1;
                        sub2(r0, r1, __uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]),
                             __uint_as_float(h0), __uint_as_float(h1));
                        lw[e] = Mma<T>::pack(r0, r1);
                    }
                    tmem_st32(sp_addr, pw);
                    tmem_st32(sp_addr + 32, lw);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        pw[e] = Mma<T>::pack(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
                    tmem_st32(sp_addr, pw);
                }
                tmem_st_wait();
                l = l * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
                tcgen05_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&ctl->p_full[qt][b]));
            }
            prev = true;
            prev_live = live;
            prev_out = out_row;
            prev_l = l;
            prev_last = Tt - 1;
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
    const size_t smem = smem_bytes(a.num_seqs);
    cudaError_t err = ensure_smem_limit<paged_prefill_tc_kernel<T, BS>>(smem);
    if (err != cudaSuccess) return err;
    const int64_t row_items = (static_cast<int64_t>(a.max_q_len) * a.group + kItemRows - 1) / kItemRows;
    const int X = static_cast<int>(row_items > 0 ? row_items : 1);
    const int64_t items = static_cast<int64_t>(X) * a.num_kv_heads * a.num_seqs;
    int device = 0, sms = 0;
    err = cudaGetDevice(&device);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (err != cudaSuccess) return err;
    // persistent: one CTA per SM walks the work list
    const int ctas = static_cast<int>(items < sms ? items : sms);
    return launch_pdl(paged_prefill_tc_kernel<T, BS>, dim3(ctas > 0 ? ctas : 1), dim3(kThreads),
                      smem, stream, k_map, v_map, a, X);
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

bool prefill_tc_supported(int group) {
    return group >= 1 && group <= kTileRows && kTileRows % group == 0;
}

int prefill_tc_box_rows(int block_size) { return block_size < kKeys ? block_size : kKeys; }

cudaError_t launch_paged_prefill_tc(const CUtensorMap& k_map, const CUtensorMap& v_map,
                                    const PrefillArgs& args, pkv_dtype dtype, int block_size,
                                    cudaStream_t stream) {
    return dtype == PKV_BF16
               ? launch_tc_dtype<__nv_bfloat16>(k_map, v_map, args, block_size, stream)
               : launch_tc_dtype<__half>(k_map, v_map, args, block_size, stream);
}

}  // namespace pkv
