// Per-tile attention math shared by the decode kernels: one [rows x 128]
// K tile and V tile in shared memory (two 64-column boxes each, 128-byte
// swizzle, as written by a TMA tile load) against the register-resident
// query fragments of up to 16 query heads, with the running max / running
// sum softmax of Eq. (4) of "Serving Language Models Within a Memory Budget".
#pragma once

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

template <int BS>
struct Geometry {
    static constexpr int kHalfBytes = BS * 128;        // one 64-column box: BS rows x 128 B
    static constexpr int kTileBytes = 2 * kHalfBytes;  // [BS x 128] tile of K or V
    static constexpr int kStageBytes = 2 * kTileBytes; // K tile + V tile
    static constexpr int kStages = 65536 / kStageBytes;  // 64 KiB ring
    static constexpr int kRingBytes = kStages * kStageBytes;
};

// Clamp a device-side sequence length into what the launch covers.
__device__ __forceinline__ int clamped_len(const DecodeArgs& a, int s, bool report_error) {
    int n = __ldg(a.seq_lens + s);
    const int cap = a.max_seq_len;  // the host checked max_seq_len <= table capacity
    if (n < 0 || n > cap) {
        if (report_error) report(a.err, PKV_DEVERR_BAD_SEQ_LEN);
        n = n < 0 ? 0 : cap;
    }
    return n;
}

template <typename T, int BS, bool kSplitP>
__device__ __forceinline__ void attend_block(uint32_t k_tile, uint32_t v_tile, int nvalid,
                                             const uint32_t (&qa)[8][4], float (&o)[16][4],
                                             float& m0, float& m1, float& l0, float& l1,
                                             float scale_log2, int lane) {
    using G = Geometry<BS>;
    constexpr int NT = BS / 8;   // n-tiles of 8 tokens
    constexpr int KK = BS / 16;  // k-steps of 16 tokens for P V
    const int mi = lane >> 3;    // which 8x8 matrix this lane addresses
    const int r = lane & 7;      // row within it (token % 8)
    const int quad = lane & 3;

    // ---- S = Q K^T ------------------------------------------------------
    float sc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int tg = 0; tg < BS / 16; ++tg) {
            const int token = tg * 16 + (mi >> 1) * 8 + r;
            const int chunk = (ks & 3) * 2 + (mi & 1);
            const uint32_t addr = k_tile + (ks >> 2) * G::kHalfBytes + token * 128 + ((chunk ^ r) << 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(addr, b0, b1, b2, b3);
            Mma<T>::run(sc[2 * tg], qa[ks], b0, b1);
            Mma<T>::run(sc[2 * tg + 1], qa[ks], b2, b3);
        }
    }

    // ---- scale, mask the unfilled tail, online softmax (Eq. 4) ------------
    float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int col = nt * 8 + quad * 2 + (e & 1);
            const float x = sc[nt][e] * scale_log2;
            sc[nt][e] = col < nvalid ? x : -INFINITY;
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

    // ---- P as the A operand (accumulator layout == A-fragment layout) -----
    uint32_t pa[KK][4];
    uint32_t pl[KK][4];
#pragma unroll
    for (int kk = 0; kk < KK; ++kk) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            // e: 0 = rows g, tokens 0-7; 1 = rows g+8, tokens 0-7;
            //    2 = rows g, tokens 8-15; 3 = rows g+8, tokens 8-15
            const int nt = 2 * kk + (e >> 1);
            const int c = (e & 1) * 2;
            pa[kk][e] = Mma<T>::pack(sc[nt][c], sc[nt][c + 1]);
            if (kSplitP) {
                const float2 hi = Mma<T>::unpack(pa[kk][e]);
                pl[kk][e] = Mma<T>::pack(sc[nt][c] - hi.x, sc[nt][c + 1] - hi.y);
            }
        }
    }

    // ---- O += P V ------------------------------------------------------------
    const bool partial = nvalid < BS;
#pragma unroll
    for (int kk = 0; kk < KK; ++kk) {
#pragma unroll
        for (int np = 0; np < 8; ++np) {
            const int token = kk * 16 + (mi & 1) * 8 + r;
            const int d8 = 2 * np + (mi >> 1);  // 8-column group of head_dim
            const uint32_t addr =
                v_tile + (d8 >> 3) * G::kHalfBytes + token * 128 + (((d8 & 7) ^ r) << 4);
            uint32_t v0, v1, v2, v3;
            ldsm_x4_trans(addr, v0, v1, v2, v3);
            if (partial) {
                // Unfilled slots may hold any bits (even NaN); zero them so that
                // their zero weights contribute exactly zero.
                const int t0 = kk * 16 + quad * 2;
                const uint32_t keep_lo0 = (t0 < nvalid) ? 0x0000ffffu : 0u;
                const uint32_t keep_hi0 = (t0 + 1 < nvalid) ? 0xffff0000u : 0u;
                const uint32_t keep_lo1 = (t0 + 8 < nvalid) ? 0x0000ffffu : 0u;
                const uint32_t keep_hi1 = (t0 + 9 < nvalid) ? 0xffff0000u : 0u;
                v0 &= keep_lo0 | keep_hi0;
                v2 &= keep_lo0 | keep_hi0;
                v1 &= keep_lo1 | keep_hi1;
                v3 &= keep_lo1 | keep_hi1;
            }
            Mma<T>::run(o[2 * np], pa[kk], v0, v1);
            Mma<T>::run(o[2 * np + 1], pa[kk], v2, v3);
            if (kSplitP) {
                Mma<T>::run(o[2 * np], pl[kk], v0, v1);
                Mma<T>::run(o[2 * np + 1], pl[kk], v2, v3);
            }
        }
    }
}


// Query fragments (A operand of m16n8k16) of up to 16 query heads: rows
// [0, live) of the [16 x 128] tile starting at `q_rows`, zero beyond.
template <typename T>
__device__ __forceinline__ void load_q_fragments(uint32_t (&qa)[8][4], const T* q_rows, int live,
                                                 int lane) {
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(q_rows);
    const int row0 = lane >> 2, quad = lane & 3;
    const bool live0 = row0 < live, live1 = row0 + 8 < live;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const int w = ks * 8 + quad;  // 32-bit word of columns ks*16 + 2*quad
        qa[ks][0] = live0 ? __ldg(qw + row0 * 64 + w) : 0u;
        qa[ks][1] = live1 ? __ldg(qw + (row0 + 8) * 64 + w) : 0u;
        qa[ks][2] = live0 ? __ldg(qw + row0 * 64 + w + 4) : 0u;
        qa[ks][3] = live1 ? __ldg(qw + (row0 + 8) * 64 + w + 4) : 0u;
    }
}

}  // namespace pkv
