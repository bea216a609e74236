// Per-warp attention state of the streaming decode kernel, one policy per
// pool format and query layout.  Each policy holds the query fragments, the
// output accumulator and the running max / running sum (Eq. (4) of "Serving
// Language Models Within a Memory Budget") of one (sequence, KV head)
// segment, and offers
//   reset(a, q_rows, g, lane)           load the group's queries, clear state
//   attend<kTT>(k_tile, v_tile, n, lane) fold one staged tile of kTT tokens in
//   flush(a, qrow, rbase, whole, g, lane) write the output rows (whole
//                                       segment) or the partial statistics
//
// Rows16Policy     16-bit pools; the group's query heads are the MMA rows.
// E4m3RowsPolicy   8-bit pools, query heads as MMA rows (groups of 9..16).
// E4m3ColsPolicy   8-bit pools, transposed: S^T = K Q^T and O^T = V^T P^T,
//                  tokens and head dims on the MMA rows and the query heads
//                  (up to 8) on its 8 columns, which halves the MMAs and the
//                  exponentials of the row form at groups of up to 8.
#pragma once

#include "decode_tile.cuh"

namespace pkv {

// ---- 16-bit pools ------------------------------------------------------------
template <typename T>
struct Rows16Policy {
    using Scalar = T;
    static constexpr bool kFp8 = false;
    static constexpr int kWarps = kStreamWarps;
    uint32_t qa[8][4];
    float o[16][4];
    float m0, m1, l0, l1;
    float sl;

    __device__ __forceinline__ void reset(const DecodeArgs& a, const T* q_rows, int g, int lane) {
        load_q_fragments<T>(qa, q_rows, g, lane);
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
        sl = a.scale_log2;
    }

    template <int kTT>
    __device__ __forceinline__ void attend(uint32_t k_tile, uint32_t v_tile, int nvalid, int lane) {
        attend_block<T, kTT, true>(k_tile, v_tile, nvalid, qa, o, m0, m1, l0, l1, sl, lane);
    }

    // n-tile nd holds dims nd * 8 + 2 quad + {0, 1} of rows lane / 4 and + 8.
    __device__ __forceinline__ void flush(const DecodeArgs& a, size_t qrow, size_t rbase,
                                          bool whole, int g, int lane) {
        const int row0 = lane >> 2, quad = lane & 3;
        float s0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
        s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
        float s1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
        if (whole) {
            const float inv0 = s0 > 0.f ? 1.f / s0 : 0.f;
            const float inv1 = s1 > 0.f ? 1.f / s1 : 0.f;
            T* out = static_cast<T*>(a.out);
#pragma unroll
            for (int nd = 0; nd < 16; ++nd) {
                const int col = nd * 8 + quad * 2;
                if (row0 < g)
                    *reinterpret_cast<uint32_t*>(out + (qrow + row0) * kHeadDim + col) =
                        Mma<T>::pack(o[nd][0] * inv0, o[nd][1] * inv0);
                if (row0 + 8 < g)
                    *reinterpret_cast<uint32_t*>(out + (qrow + row0 + 8) * kHeadDim + col) =
                        Mma<T>::pack(o[nd][2] * inv1, o[nd][3] * inv1);
            }
            return;
        }
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) {
            const int col = nd * 8 + quad * 2;
            if (row0 < g)
                *reinterpret_cast<float2*>(a.ws_acc + (rbase + row0) * kHeadDim + col) =
                    make_float2(o[nd][0], o[nd][1]);
            if (row0 + 8 < g)
                *reinterpret_cast<float2*>(a.ws_acc + (rbase + row0 + 8) * kHeadDim + col) =
                    make_float2(o[nd][2], o[nd][3]);
        }
        if (quad == 0) {
            if (row0 < g) {
                a.ws_m[rbase + row0] = m0;
                a.ws_l[rbase + row0] = s0;
            }
            if (row0 + 8 < g) {
                a.ws_m[rbase + row0 + 8] = m1;
                a.ws_l[rbase + row0 + 8] = s1;
            }
        }
    }
};

// ---- 8-bit pools, query heads as rows ----------------------------------------
template <typename T>
struct E4m3RowsPolicy {
    using Scalar = T;
    static constexpr bool kFp8 = true;
    static constexpr int kWarps = kStreamWarpsFp8;
    uint32_t qa[8][4];
    float o[16][4];
    float m0, m1, l0, l1;
    float sl0, sl1;

    __device__ __forceinline__ void reset(const DecodeArgs& a, const T* q_rows, int g, int lane) {
        load_q_fragments_e4m3<T>(qa, q_rows, g, lane, a.scale_log2, sl0, sl1);
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
    }

    template <int kTT>
    __device__ __forceinline__ void attend(uint32_t k_tile, uint32_t v_tile, int nvalid, int lane) {
        attend_tile_e4m3<kTT, kFp8SplitP>(k_tile, v_tile, nvalid, qa, o, m0, m1, l0, l1, sl0, sl1,
                                          lane);
    }

    // n-tiles 2c and 2c + 1 interleave dims 16 c + 4 quad + {0..3}.
    __device__ __forceinline__ void flush(const DecodeArgs& a, size_t qrow, size_t rbase,
                                          bool whole, int g, int lane) {
        const int row0 = lane >> 2, quad = lane & 3;
        float s0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
        s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
        float s1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
        const float vs = a.v_scale;
        if (whole) {
            const float inv0 = s0 > 0.f ? vs / s0 : 0.f;
            const float inv1 = s1 > 0.f ? vs / s1 : 0.f;
            T* out = static_cast<T*>(a.out);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int col = c * 16 + quad * 4;
                if (row0 < g)
                    *reinterpret_cast<uint2*>(out + (qrow + row0) * kHeadDim + col) =
                        make_uint2(Mma<T>::pack(o[2 * c][0] * inv0, o[2 * c + 1][0] * inv0),
                                   Mma<T>::pack(o[2 * c][1] * inv0, o[2 * c + 1][1] * inv0));
                if (row0 + 8 < g)
                    *reinterpret_cast<uint2*>(out + (qrow + row0 + 8) * kHeadDim + col) =
                        make_uint2(Mma<T>::pack(o[2 * c][2] * inv1, o[2 * c + 1][2] * inv1),
                                   Mma<T>::pack(o[2 * c][3] * inv1, o[2 * c + 1][3] * inv1));
            }
            return;
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int col = c * 16 + quad * 4;
            if (row0 < g)
                *reinterpret_cast<float4*>(a.ws_acc + (rbase + row0) * kHeadDim + col) =
                    make_float4(o[2 * c][0] * vs, o[2 * c + 1][0] * vs, o[2 * c][1] * vs,
                                o[2 * c + 1][1] * vs);
            if (row0 + 8 < g)
                *reinterpret_cast<float4*>(a.ws_acc + (rbase + row0 + 8) * kHeadDim + col) =
                    make_float4(o[2 * c][2] * vs, o[2 * c + 1][2] * vs, o[2 * c][3] * vs,
                                o[2 * c + 1][3] * vs);
        }
        if (quad == 0) {
            if (row0 < g) {
                a.ws_m[rbase + row0] = m0;
                a.ws_l[rbase + row0] = s0;
            }
            if (row0 + 8 < g) {
                a.ws_m[rbase + row0 + 8] = m1;
                a.ws_l[rbase + row0 + 8] = s1;
            }
        }
    }
};

// ---- 8-bit pools, transposed (groups of up to 8 query heads) ----------------
// Lane (n = lane / 4, quad = lane & 3).  Query head n supplies the B operand
// of S^T = K Q^T: k-step s holds dims 16 s + 4 quad + {0, 1} and + {2, 3},
// the order in which ldmatrix delivers K's codes (the A operand, tokens on
// the rows).  The S^T accumulator of a 16-token M-tile gives the lane tokens
// n and n + 8 of heads 2 quad ("A") and 2 quad + 1 ("B"); movmatrix turns
// the binary16 P^T of those 8 x 8 blocks into the B operand of
// O^T = V^T P^T, whose A operand comes from ldmatrix.trans of V's codes
// with a byte permute: M-tile c (one 16-dim chunk) has dims 16 c + 2 n on
// rows n and 16 c + 2 n + 1 on rows n + 8.  So the lane's O^T accumulator
// ot[c] holds dims 16 c + 2 n (+ 1) of heads A and B.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

template <typename T>
struct E4m3ColsPolicy {
    using Scalar = T;
    static constexpr bool kFp8 = true;
    static constexpr int kWarps = kStreamWarpsFp8Cols;
    uint32_t qb[8][2];
    float ot[8][4];
    float mA, mB, lA, lB;  // running max / this lane's part of the running sum
    float slA, slB;        // score factors (log2 units) of heads A and B

    __device__ __forceinline__ void reset(const DecodeArgs& a, const T* q_rows, int g, int lane) {
        const int n = lane >> 2, quad = lane & 3;
        const bool live = n < g;
        const uint2* qr = reinterpret_cast<const uint2*>(q_rows + n * kHeadDim);
        uint2 w[8];
#pragma unroll
        for (int s = 0; s < 8; ++s) w[s] = live ? __ldg(qr + s * 4 + quad) : make_uint2(0u, 0u);
        float sl = a.scale_log2;
        if constexpr (std::is_same<T, __half>::value) {
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                qb[s][0] = w[s].x;
                qb[s][1] = w[s].y;
            }
        } else {
            // bfloat16 row: scale by 2^e so that its largest magnitude lands in
            // [2^14, 2^15) (exact), round to binary16, divide 2^e out of the scores
            float big = 0.f;
#pragma unroll
            for (int s = 0; s < 8; ++s)
                big = fmaxf(big, fmaxf(fmaxf(fabsf(__uint_as_float(w[s].x << 16)),
                                             fabsf(__uint_as_float(w[s].x & 0xffff0000u))),
                                       fmaxf(fabsf(__uint_as_float(w[s].y << 16)),
                                             fabsf(__uint_as_float(w[s].y & 0xffff0000u)))));
            big = fmaxf(big, __shfl_xor_sync(0xffffffffu, big, 1));
            big = fmaxf(big, __shfl_xor_sync(0xffffffffu, big, 2));
            int x = 0;
            frexpf(big, &x);
            const int e = min(max(15 - x, -100), 100);
            const float up = __int_as_float((127 + e) << 23);
            sl = a.scale_log2 * __int_as_float((127 - e) << 23);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const __half2 h0 = __floats2half2_rn(__uint_as_float(w[s].x << 16) * up,
                                                     __uint_as_float(w[s].x & 0xffff0000u) * up);
                const __half2 h1 = __floats2half2_rn(__uint_as_float(w[s].y << 16) * up,
                                                     __uint_as_float(w[s].y & 0xffff0000u) * up);
                qb[s][0] = *reinterpret_cast<const uint32_t*>(&h0);
                qb[s][1] = *reinterpret_cast<const uint32_t*>(&h1);
            }
        }
        slA = __shfl_sync(0xffffffffu, sl, 8 * quad);      // head 2 quad lives on lanes 8 quad ..
        slB = __shfl_sync(0xffffffffu, sl, 8 * quad + 4);  // head 2 quad + 1 on lanes 8 quad + 4 ..
#pragma unroll
        for (int c = 0; c < 8; ++c) ot[c][0] = ot[c][1] = ot[c][2] = ot[c][3] = 0.f;
        mA = mB = -INFINITY;
        lA = lB = 0.f;
    }

    template <int kTT>
    __device__ __forceinline__ void attend(uint32_t k_tile, uint32_t v_tile, int nvalid, int lane) {
        using M = Mma<__half>;
        constexpr int MT = kTT / 16;  // 16-token M-tiles (and k-steps of P V)
        const int mi = lane >> 3, r = lane & 7;
        const int n = lane >> 2, quad = lane & 3;
        const int row = (mi & 1) * 8 + r;  // row within 16 this lane addresses for ldmatrix

        // ---- S^T = K Q^T, two partial accumulators per M-tile ---------------
        float d[MT][2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) d[mt][h][0] = d[mt][h][1] = d[mt][h][2] = d[mt][h][3] = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int sp = 0; sp < 4; ++sp) {
                const int chunk = 2 * sp + (mi >> 1);
                uint32_t x[4];
                ldsm_x4(k_tile + (mt * 16 + row) * 128 + ((chunk ^ r) << 4), x[0], x[1], x[2], x[3]);
                // x[0] / x[1]: tokens 0-7 / 8-15 at chunk 2 sp; x[2] / x[3] at chunk 2 sp + 1
#pragma unroll
                for (int hs = 0; hs < 2; ++hs) {
                    uint32_t af[4];
                    e4m3x4_to_f16x2(x[2 * hs], af[0], af[2]);
                    e4m3x4_to_f16x2(x[2 * hs + 1], af[1], af[3]);
                    M::run(d[mt][sp & 1], af, qb[2 * sp + hs][0], qb[2 * sp + hs][1]);
                }
            }
        }

        // ---- mask, online softmax per head (Eq. 4) -----------------------------
        float sc[MT][4];  // [token n: head A, head B | token n + 8: head A, head B]
        float bmA = -INFINITY, bmB = -INFINITY;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int t0 = mt * 16 + n;
            const bool v0 = t0 < nvalid, v1 = t0 + 8 < nvalid;
            sc[mt][0] = v0 ? (d[mt][0][0] + d[mt][1][0]) * slA : -INFINITY;
            sc[mt][1] = v0 ? (d[mt][0][1] + d[mt][1][1]) * slB : -INFINITY;
            sc[mt][2] = v1 ? (d[mt][0][2] + d[mt][1][2]) * slA : -INFINITY;
            sc[mt][3] = v1 ? (d[mt][0][3] + d[mt][1][3]) * slB : -INFINITY;
            bmA = fmaxf(bmA, fmaxf(sc[mt][0], sc[mt][2]));
            bmB = fmaxf(bmB, fmaxf(sc[mt][1], sc[mt][3]));
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {  // lanes of the same quad share heads A, B
            bmA = fmaxf(bmA, __shfl_xor_sync(0xffffffffu, bmA, off));
            bmB = fmaxf(bmB, __shfl_xor_sync(0xffffffffu, bmB, off));
        }
        const float mnA = fmaxf(mA, bmA), mnB = fmaxf(mB, bmB);
        const float baseA = mnA == -INFINITY ? 0.f : mnA;
        const float baseB = mnB == -INFINITY ? 0.f : mnB;
        const float alphaA = ex2(mA - baseA), alphaB = ex2(mB - baseB);
        const bool rescale = mnA != mA || mnB != mB;
        mA = mnA;
        mB = mnB;
        float psA = 0.f, psB = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            sc[mt][0] = ex2(sc[mt][0] - baseA);
            sc[mt][1] = ex2(sc[mt][1] - baseB);
            sc[mt][2] = ex2(sc[mt][2] - baseA);
            sc[mt][3] = ex2(sc[mt][3] - baseB);
            psA += sc[mt][0] + sc[mt][2];
            psB += sc[mt][1] + sc[mt][3];
        }
        lA = lA * alphaA + psA;
        lB = lB * alphaB + psB;
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                ot[c][0] *= alphaA;
                ot[c][1] *= alphaB;
                ot[c][2] *= alphaA;
                ot[c][3] *= alphaB;
            }
        }

        // ---- O^T += V^T P^T ---------------------------------------------------------
        const bool partial = nvalid < kTT;
#pragma unroll
        for (int kk = 0; kk < MT; ++kk) {
            // P^T B fragments: tokens 2 quad, 2 quad + 1 (and + 8) of head n
            const uint32_t pb0 = movmatrix_trans(M::pack(sc[kk][0], sc[kk][1]));
            const uint32_t pb1 = movmatrix_trans(M::pack(sc[kk][2], sc[kk][3]));
            const int t0 = kk * 16 + quad * 2;
            const uint32_t keep0 =
                ((t0 < nvalid) ? 0x0000ffffu : 0u) | ((t0 + 1 < nvalid) ? 0xffff0000u : 0u);
            const uint32_t keep1 =
                ((t0 + 8 < nvalid) ? 0x0000ffffu : 0u) | ((t0 + 9 < nvalid) ? 0xffff0000u : 0u);
#pragma unroll
            for (int cp = 0; cp < 4; ++cp) {
                const int chunk = 2 * cp + (mi >> 1);
                uint32_t x[4];
                ldsm_x4_trans(v_tile + (kk * 16 + row) * 128 + ((chunk ^ r) << 4), x[0], x[1], x[2],
                              x[3]);
                // x[j]: tokens 8 (j & 1) .. + 7 of the k-step, chunk 2 cp + (j >> 1); bytes
                // [tok 2quad: dim 2n, dim 2n+1 | tok 2quad+1: dim 2n, dim 2n+1]
#pragma unroll
                for (int hc = 0; hc < 2; ++hc) {
                    uint32_t af[4];  // rows n: dim 16c + 2n; rows n + 8: dim 16c + 2n + 1
                    e4m3x4_to_f16x2(__byte_perm(x[2 * hc], 0, 0x3120), af[0], af[1]);
                    e4m3x4_to_f16x2(__byte_perm(x[2 * hc + 1], 0, 0x3120), af[2], af[3]);
                    if (partial) {  // unfilled rows may hold any codes (NaN too): zero them
                        af[0] &= keep0;
                        af[1] &= keep0;
                        af[2] &= keep1;
                        af[3] &= keep1;
                    }
                    M::run(ot[2 * cp + hc], af, pb0, pb1);
                }
            }
        }
    }

    __device__ __forceinline__ void flush(const DecodeArgs& a, size_t qrow, size_t rbase,
                                          bool whole, int g, int lane) {
        const int n = lane >> 2, quad = lane & 3;
        float sA = lA, sB = lB;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            sA += __shfl_xor_sync(0xffffffffu, sA, off);
            sB += __shfl_xor_sync(0xffffffffu, sB, off);
        }
        const int hA = 2 * quad, hB = 2 * quad + 1;
        const float vs = a.v_scale;
        if (whole) {
            const float invA = sA > 0.f ? vs / sA : 0.f;
            const float invB = sB > 0.f ? vs / sB : 0.f;
            T* out = static_cast<T*>(a.out);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int col = c * 16 + 2 * n;
                if (hA < g)
                    *reinterpret_cast<uint32_t*>(out + (qrow + hA) * kHeadDim + col) =
                        Mma<T>::pack(ot[c][0] * invA, ot[c][2] * invA);
                if (hB < g)
                    *reinterpret_cast<uint32_t*>(out + (qrow + hB) * kHeadDim + col) =
                        Mma<T>::pack(ot[c][1] * invB, ot[c][3] * invB);
            }
            return;
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int col = c * 16 + 2 * n;
            if (hA < g)
                *reinterpret_cast<float2*>(a.ws_acc + (rbase + hA) * kHeadDim + col) =
                    make_float2(ot[c][0] * vs, ot[c][2] * vs);
            if (hB < g)
                *reinterpret_cast<float2*>(a.ws_acc + (rbase + hB) * kHeadDim + col) =
                    make_float2(ot[c][1] * vs, ot[c][3] * vs);
        }
        if (n == 0) {
            if (hA < g) {
                a.ws_m[rbase + hA] = mA;
                a.ws_l[rbase + hA] = sA;
            }
            if (hB < g) {
                a.ws_m[rbase + hB] = mB;
                a.ws_l[rbase + hB] = sB;
            }
        }
    }
};

}  // namespace pkv
