// Paged decode attention for sm_103a.
//
// What it computes (vLLM PagedAttention & continuous batching,
// "PagedAttention" and "The kernel page"): one query token per sequence
// attends over that sequence's keys and values, which sit in fixed-size
// physical blocks reached through its block table; the attention formula is
// the ordinary softmax(scale * q K^T) V.  The softmax runs block by block with
// the running maximum / running sum recurrence of Eq. (4) of "Serving
// Language Models Within a Memory Budget".  Long sequences are split into
// partitions whose (max, sum, weighted sum) statistics are merged by the
// same rule in a second kernel.
//
// Work decomposition.  One CTA per (partition, KV head, sequence).  The CTA
// serves every query head of the KV head's group, so each K/V byte is read
// from HBM once.  Warp 4 is a TMA producer: it walks the partition's block
// table entries and streams each physical block's K tile and V tile
// ([block_size x 128] each, two 64-column boxes per tile, 128-byte swizzle)
// into a ring of shared-memory stages guarded by full / empty mbarriers.
// Warps 0-3 consume the stages round-robin:
//   S = Q K^T     mma.sync m16n8k16, A = the group's query heads (rows,
//                 zero-padded to 16 per m-tile, held in registers for the
//                 whole CTA), B = the K tile via ldmatrix (tokens as N);
//   softmax       fp32 running max / sum per query head (log2 domain);
//   O += P V      the score accumulator is re-packed in registers as the A
//                 operand, V via ldmatrix.trans (d as N); P is split into a
//                 high and a low 16-bit part so the weights keep ~16 bits.
// At the end the four warps' partial (m, l, O) are merged through shared
// memory (the ring, then idle) and written either as the final output
// (single partition) or as fp32 partition statistics for the merge kernel.
//
// The decode path moves ~1 flop per byte at 4 query heads per KV head, so
// it is bound by HBM bandwidth; the tensor cores only keep the CUDA cores
// free for the softmax and address arithmetic.
#include "decode_tile.cuh"

namespace pkv {
namespace {

// Shared-memory bookkeeping placed after the ring.
struct alignas(8) Control {
    uint64_t full[8];
    uint64_t empty[8];
    int32_t valid[8];
    volatile int32_t abort;
    float m[kConsumerWarps][16];
    float l[kConsumerWarps][16];
};

constexpr int kMergeRowFloats = 132;  // padded row of the cross-warp merge buffer

// MT = number of 16-row m-tiles that cover the query-head group.
template <typename T, int BS, int MT>
__global__ void __launch_bounds__(kDecodeThreads, 2)
    paged_decode_kernel(const __grid_constant__ CUtensorMap k_map,
                        const __grid_constant__ CUtensorMap v_map, const DecodeArgs a) {
    using G = Geometry<BS>;
    constexpr int NST = G::kStages;
    constexpr int kWarpsPerTile = kConsumerWarps / MT;
    constexpr bool kSplitP = true;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Control* ctl = reinterpret_cast<Control*>(ring + G::kRingBytes);

    const int p = blockIdx.x;
    const int h = blockIdx.y;
    const int s = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    pdl_wait_prerequisites();
    pdl_allow_dependents();
    const int n = clamped_len(a, s, p == 0 && h == 0 && threadIdx.x == 0);
    const int P = a.partition_size;
    const int np_s = n > 0 ? (n + P - 1) / P : 1;
    if (p >= np_s) return;  // uniform over the CTA
    const int tok0 = p * P;
    const int tok1 = min(tok0 + P, n);
    const int blk0 = tok0 / BS;
    const int nblk = tok1 > tok0 ? (tok1 - 1) / BS - blk0 + 1 : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(smem_addr(&ctl->full[i]), 1);
            mbar_init(smem_addr(&ctl->empty[i]), MT);
        }
        ctl->abort = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ======================= TMA producer warp =========================
        if (lane == 0) {
            prefetch_tensormap(&k_map);
            prefetch_tensormap(&v_map);
        }
        const int32_t* table = a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq + blk0;
        for (int jc = 0; jc < nblk; jc += 32) {
            const int j = jc + lane;
            int bid = 0;
            int ok = 0;
            if (j < nblk) {
                bid = __ldg(table + j);
                ok = (bid >= 0 && bid < a.num_blocks) ? 1 : 0;
                if (!ok) report(a.err, PKV_DEVERR_BAD_BLOCK_ID);
            }
            const int cnt = min(32, nblk - jc);
            for (int u = 0; u < cnt; ++u) {
                const int b = __shfl_sync(0xffffffffu, bid, u);
                const int okb = __shfl_sync(0xffffffffu, ok, u);
                if (lane == 0 && !ctl->abort) {
                    const int jj = jc + u;
                    const int st = jj % NST;
                    const int use = jj / NST;
                    bool ready = true;
                    if (use > 0) ready = mbar_wait(smem_addr(&ctl->empty[st]), (use - 1) & 1);
                    if (!ready) {
                        report(a.err, PKV_DEVERR_TIMEOUT);
                        ctl->abort = 1;
                    } else {
                        ctl->valid[st] = okb;
                        const uint32_t full = smem_addr(&ctl->full[st]);
                        if (okb) {
                            const uint32_t kt = smem_addr(ring + st * G::kStageBytes);
                            const uint32_t vt = kt + G::kTileBytes;
                            mbar_arrive_expect_tx(full, G::kStageBytes);
                            tma_load_4d(kt, &k_map, full, 0, 0, h, b);
                            tma_load_4d(kt + G::kHalfBytes, &k_map, full, 64, 0, h, b);
                            tma_load_4d(vt, &v_map, full, 0, 0, h, b);
                            tma_load_4d(vt + G::kHalfBytes, &v_map, full, 64, 0, h, b);
                        } else {
                            mbar_arrive(full);  // consumers skip an invalid block
                        }
                    }
                }
                __syncwarp();
            }
        }
        // Do not leave while copies into this CTA's shared memory are in
        // flight: wait (bounded) for the last use of every stage.
        if (lane == 0) {
            const int first = nblk > NST ? nblk - NST : 0;
            for (int jj = first; jj < nblk; ++jj)
                mbar_wait(smem_addr(&ctl->full[jj % NST]), (jj / NST) & 1);
        }
        return;
    }

    // ========================= consumer warps ==============================
    const int mt = warp % MT;
    const int wj = warp / MT;
    const int row0 = lane >> 2;
    const int quad = lane & 3;
    const int gl = min(16, a.group - mt * 16);  // live rows of this m-tile

    uint32_t qa[8][4];
    {
        const uint32_t* qw = reinterpret_cast<const uint32_t*>(
            static_cast<const T*>(a.q) +
            (static_cast<size_t>(s) * a.num_q_heads + static_cast<size_t>(h) * a.group + mt * 16) *
                kHeadDim);
        const bool live0 = row0 < gl, live1 = row0 + 8 < gl;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int w = ks * 8 + quad;  // 32-bit word of columns ks*16 + 2*quad
            qa[ks][0] = live0 ? __ldg(qw + row0 * 64 + w) : 0u;
            qa[ks][1] = live1 ? __ldg(qw + (row0 + 8) * 64 + w) : 0u;
            qa[ks][2] = live0 ? __ldg(qw + row0 * 64 + w + 4) : 0u;
            qa[ks][3] = live1 ? __ldg(qw + (row0 + 8) * 64 + w + 4) : 0u;
        }
    }

    float o[16][4];
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int j = wj; j < nblk; j += kWarpsPerTile) {
        const int st = j % NST;
        const int use = j / NST;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->full[st]), use & 1))) {
            if (lane == 0) {
                report(a.err, PKV_DEVERR_TIMEOUT);
                ctl->abort = 1;
            }
            break;  // the whole warp stops together
        }
        if (ctl->valid[st]) {
            const uint32_t kt = smem_addr(ring + st * G::kStageBytes);
            const int nvalid = min(BS, tok1 - (blk0 + j) * BS);
            attend_block<T, BS, kSplitP>(kt, kt + G::kTileBytes, nvalid, qa, o, m0, m1, l0, l1,
                                         a.scale_log2, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&ctl->empty[st]));
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    // ---- merge the consumer warps' partial results ---------------------------
    named_barrier_sync(1, kConsumerWarps * 32);  // every stage consumed: the ring is free
    float* mrg = reinterpret_cast<float*>(ring) + warp * 16 * kMergeRowFloats;
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
        const int col = nd * 8 + quad * 2;
        if (row0 < gl) *reinterpret_cast<float2*>(mrg + row0 * kMergeRowFloats + col) = make_float2(o[nd][0], o[nd][1]);
        if (row0 + 8 < gl)
            *reinterpret_cast<float2*>(mrg + (row0 + 8) * kMergeRowFloats + col) = make_float2(o[nd][2], o[nd][3]);
    }
    if (quad == 0) {
        ctl->m[warp][row0] = m0;
        ctl->l[warp][row0] = l0;
        ctl->m[warp][row0 + 8] = m1;
        ctl->l[warp][row0 + 8] = l1;
    }
    named_barrier_sync(1, kConsumerWarps * 32);

    const int d = threadIdx.x;  // 0..127: one output column per thread
    const float* ring_f = reinterpret_cast<const float*>(ring);
    for (int i = 0; i < a.group; ++i) {
        const int tile = i >> 4, lr = i & 15;
        float big = -INFINITY;
#pragma unroll
        for (int k = 0; k < kWarpsPerTile; ++k) big = fmaxf(big, ctl->m[tile + k * MT][lr]);
        float acc = 0.f, den = 0.f;
        if (big != -INFINITY) {
#pragma unroll
            for (int k = 0; k < kWarpsPerTile; ++k) {
                const int w = tile + k * MT;
                const float wgt = ex2(ctl->m[w][lr] - big);
                den += wgt * ctl->l[w][lr];
                acc += wgt * ring_f[(w * 16 + lr) * kMergeRowFloats + d];
            }
        }
        const size_t row = static_cast<size_t>(s) * a.num_q_heads + static_cast<size_t>(h) * a.group + i;
        if (np_s == 1) {
            const float val = den > 0.f ? acc / den : 0.f;
            static_cast<T*>(a.out)[row * kHeadDim + d] = Mma<T>::from_float(val);
        } else {
            const size_t idx = row * a.max_partitions + p;
            a.ws_acc[idx * kHeadDim + d] = acc;
            if (d == 0) {
                a.ws_m[idx] = big;
                a.ws_l[idx] = den;
            }
        }
    }
}

// Merge of partition statistics, Eq. (4) with each partition as one block:
// out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p,  M = max_p m_p.
template <typename T>
__global__ void __launch_bounds__(kHeadDim) merge_partitions_kernel(const DecodeArgs a) {
    pdl_wait_prerequisites();
    pdl_allow_dependents();
    const int i = blockIdx.x;  // query head
    const int s = blockIdx.y;
    const int d = threadIdx.x;
    const int n = clamped_len(a, s, false);
    const int P = a.partition_size;
    const int np_s = n > 0 ? (n + P - 1) / P : 1;
    if (np_s <= 1) return;  // written directly by the decode kernel
    const size_t row = static_cast<size_t>(s) * a.num_q_heads + i;
    const float* m = a.ws_m + row * a.max_partitions;
    const float* l = a.ws_l + row * a.max_partitions;
    const float* acc = a.ws_acc + row * a.max_partitions * kHeadDim;
    float big = -INFINITY;
    for (int p = 0; p < np_s; ++p) big = fmaxf(big, m[p]);
    float num = 0.f, den = 0.f;
    if (big != -INFINITY) {
        for (int p = 0; p < np_s; ++p) {
            const float w = ex2(m[p] - big);
            den += w * l[p];
            num += w * acc[static_cast<size_t>(p) * kHeadDim + d];
        }
    }
    static_cast<T*>(a.out)[row * kHeadDim + d] = Mma<T>::from_float(den > 0.f ? num / den : 0.f);
}

template <typename T, int BS, int MT>
cudaError_t launch_typed(const CUtensorMap& k_map, const CUtensorMap& v_map, const DecodeArgs& a,
                         cudaStream_t stream) {
    using G = Geometry<BS>;
    const size_t smem = 1024 + G::kRingBytes + sizeof(Control);
    auto kernel = paged_decode_kernel<T, BS, MT>;
    cudaError_t err = ensure_smem_limit<paged_decode_kernel<T, BS, MT>>(smem);
    if (err != cudaSuccess) return err;
    dim3 grid(static_cast<unsigned>(a.max_partitions), static_cast<unsigned>(a.num_kv_heads),
              static_cast<unsigned>(a.num_seqs));
    err = launch_pdl(kernel, grid, dim3(kDecodeThreads), smem, stream, k_map, v_map, a);
    if (err != cudaSuccess || a.max_partitions <= 1) return err;
    dim3 mgrid(static_cast<unsigned>(a.num_q_heads), static_cast<unsigned>(a.num_seqs));
    return launch_pdl(merge_partitions_kernel<T>, mgrid, dim3(kHeadDim), 0, stream, a);
}

template <typename T, int BS>
cudaError_t launch_bs(const CUtensorMap& k_map, const CUtensorMap& v_map, const DecodeArgs& a,
                      cudaStream_t stream) {
    if (a.group <= 16) return launch_typed<T, BS, 1>(k_map, v_map, a, stream);
    if (a.group <= 32) return launch_typed<T, BS, 2>(k_map, v_map, a, stream);
    return launch_typed<T, BS, 4>(k_map, v_map, a, stream);
}

}  // namespace

cudaError_t launch_paged_decode(const CUtensorMap& k_map, const CUtensorMap& v_map,
                                const DecodeArgs& args, pkv_dtype dtype, int block_size,
                                cudaStream_t stream) {
    if (dtype == PKV_BF16) {
        return block_size == 16 ? launch_bs<__nv_bfloat16, 16>(k_map, v_map, args, stream)
                                : launch_bs<__nv_bfloat16, 32>(k_map, v_map, args, stream);
    }
    return block_size == 16 ? launch_bs<__half, 16>(k_map, v_map, args, stream)
                            : launch_bs<__half, 32>(k_map, v_map, args, stream);
}

}  // namespace pkv
