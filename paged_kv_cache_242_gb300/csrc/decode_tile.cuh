// Per-tile attention math shared by the decode kernels: one [rows x 128]
// K tile and V tile in shared memory (two 64-column boxes each, 128-byte
// swizzle, as written by a TMA tile load) against the register-resident
// query fragments of up to 16 query heads, with the running max / running
// sum softmax of Eq. (4) of "Serving Language Models Within a Memory Budget".
#pragma once

#include <cuda_fp8.h>

#include <type_traits>

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
    const bool rescale = mn0 != m0 || mn1 != m1;
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
    if (__any_sync(0xffffffffu, rescale)) {  // some row's running maximum moved
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) {
            o[nd][0] *= alpha0;
            o[nd][1] *= alpha0;
            o[nd][2] *= alpha1;
            o[nd][3] *= alpha1;
        }
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

// ---- 8-bit (E4M3) pools ------------------------------------------------------
// A streamed tile is 16 or 32 token rows of 128 one-byte codes (128-byte TMA
// boxes, 128-byte swizzle: the 16-byte chunk c of row t sits at chunk
// c ^ (t & 7)).  Codes are widened to binary16 in registers, which is exact
// (every E4M3 value is a binary16 value), and multiplied with binary16 query
// fragments by mma.sync m16n8k16; the pool scales are applied to the fp32
// scores and to the output.
//
// Q K^T.  ldmatrix of the tile viewed as 16-bit pairs gives lane
// (row t = lane / 4, quad) the four codes of dims 4 quad .. 4 quad + 3 of a
// 16-dim chunk.  They fill k = 2 quad, 2 quad + 1, 2 quad + 8, 2 quad + 9 of
// that k16 step, so the query fragment of step s holds dims
// 16 s + 4 quad + {0, 1} in registers 0 / 1 and + {2, 3} in registers 2 / 3:
// the same dot product summed in another order.
//
// P V.  ldmatrix.trans of 8 rows gives lane (quad, n = lane / 4) the codes of
// tokens 2 quad and 2 quad + 1 at dims 2 n and 2 n + 1 of a chunk; a byte
// permute splits them into the B fragments of two n8 tiles, one holding the
// even and one the odd dims of the chunk.  Output n-tile 2 c + p therefore
// holds dims 16 c + 2 n + p, and lane quad's accumulators cover the four
// consecutive dims 16 c + 4 quad .. + 3.

// Four codes (bytes 0..3) -> binary16 pairs (bytes 0, 1) and (bytes 2, 3),
// lower byte to the lower half (cvt.rn.f16x2.e4m3x2, exact).
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t x, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(x));
}

// One tile of kTokens (16 or 32) token rows of E4M3 codes.  sl0 / sl1: score
// factors (log2 units) of this lane's two rows.
template <int kTokens, bool kSplitP>
__device__ __forceinline__ void attend_tile_e4m3(uint32_t k_tile, uint32_t v_tile, int nvalid,
                                                 const uint32_t (&qa)[8][4], float (&o)[16][4],
                                                 float& m0, float& m1, float& l0, float& l1,
                                                 float sl0, float sl1, int lane) {
    using M = Mma<__half>;
    constexpr int NT = kTokens / 8;   // n-tiles of 8 tokens
    constexpr int KK = kTokens / 16;  // k-steps of 16 tokens for P V
    const int mi = lane >> 3;
    const int r = lane & 7;
    const int quad = lane & 3;
    const int row = (mi & 1) * 8 + r;  // row (within 16) this lane addresses for ldmatrix

    // ---- S = Q K^T: each ldmatrix.x4 covers 2 n-tiles x 2 k-steps -----------
    float sc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int th = 0; th < KK; ++th) {
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
            const int chunk = 2 * kp + (mi >> 1);
            uint32_t d[4];
            ldsm_x4(k_tile + (th * 16 + row) * 128 + ((chunk ^ r) << 4), d[0], d[1], d[2], d[3]);
            // d[j]: n-tile 2 th + (j & 1), k-step 2 kp + (j >> 1)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t b0, b1;
                e4m3x4_to_f16x2(d[j], b0, b1);
                M::run(sc[2 * th + (j & 1)], qa[2 * kp + (j >> 1)], b0, b1);
            }
        }
    }

    // ---- mask the unfilled tail, online softmax (Eq. 4) ------------------------
    float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int col = nt * 8 + quad * 2 + (e & 1);
            const float x = sc[nt][e] * (e < 2 ? sl0 : sl1);
            sc[nt][e] = col < nvalid ? x : -INFINITY;  // select: drops NaN of unfilled rows
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
    const bool rescale = mn0 != m0 || mn1 != m1;
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
    if (__any_sync(0xffffffffu, rescale)) {  // some row's running maximum moved
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) {
            o[nd][0] *= alpha0;
            o[nd][1] *= alpha0;
            o[nd][2] *= alpha1;
            o[nd][3] *= alpha1;
        }
    }

    // ---- P (binary16, optionally split into high and low parts) -------------
    uint32_t pa[KK][4], pl[KK][4];
#pragma unroll
    for (int kk = 0; kk < KK; ++kk) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int nt = 2 * kk + (e >> 1);
            const int c = (e & 1) * 2;
            pa[kk][e] = M::pack(sc[nt][c], sc[nt][c + 1]);
            if (kSplitP) {
                const float2 hi = M::unpack(pa[kk][e]);
                pl[kk][e] = M::pack(sc[nt][c] - hi.x, sc[nt][c + 1] - hi.y);
            }
        }
    }

    // ---- O += P V -----------------------------------------------------------------
    const bool partial = nvalid < kTokens;
#pragma unroll
    for (int kk = 0; kk < KK; ++kk) {
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
            // x[j]: tokens 16 kk + 8 (j & 1) .. + 7, chunk 2 cp + (j >> 1); bytes
            // [tok 2quad: dim 2n, dim 2n+1 | tok 2quad+1: dim 2n, dim 2n+1]
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                uint32_t even0, odd0, even1, odd1;
                e4m3x4_to_f16x2(__byte_perm(x[2 * hc], 0, 0x3120), even0, odd0);
                e4m3x4_to_f16x2(__byte_perm(x[2 * hc + 1], 0, 0x3120), even1, odd1);
                if (partial) {  // unfilled rows may hold any codes (NaN too): zero them
                    even0 &= keep0;
                    odd0 &= keep0;
                    even1 &= keep1;
                    odd1 &= keep1;
                }
                const int ch = 2 * cp + hc;
                M::run(o[2 * ch], pa[kk], even0, even1);
                M::run(o[2 * ch + 1], pa[kk], odd0, odd1);
                if (kSplitP) {
                    M::run(o[2 * ch], pl[kk], even0, even1);
                    M::run(o[2 * ch + 1], pl[kk], odd0, odd1);
                }
            }
        }
    }
}

// Query fragments for attend_tile_e4m3 (dims 16 s + 4 quad .. + 3 per k-step
// s), as binary16, and each row's score factor.  A bfloat16 row is scaled by
// 2^e, e chosen so that its largest magnitude lands in [2^14, 2^15) (exact),
// then rounded to binary16; 2^-e goes into the row's factor.
template <typename T>
__device__ __forceinline__ void load_q_fragments_e4m3(uint32_t (&qa)[8][4], const T* q_rows,
                                                      int live, int lane, float scale_log2,
                                                      float& sl0, float& sl1) {
    const int row0 = lane >> 2, quad = lane & 3;
    const bool live0 = row0 < live, live1 = row0 + 8 < live;
    const uint2* r0 = reinterpret_cast<const uint2*>(q_rows + row0 * kHeadDim);
    const uint2* r1 = reinterpret_cast<const uint2*>(q_rows + (row0 + 8) * kHeadDim);
    uint2 w0[8], w1[8];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const int idx = ks * 4 + quad;  // 8-byte word of dims 16 ks + 4 quad
        w0[ks] = live0 ? __ldg(r0 + idx) : make_uint2(0u, 0u);
        w1[ks] = live1 ? __ldg(r1 + idx) : make_uint2(0u, 0u);
    }
    if constexpr (std::is_same<T, __half>::value) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            qa[ks][0] = w0[ks].x;
            qa[ks][1] = w1[ks].x;
            qa[ks][2] = w0[ks].y;
            qa[ks][3] = w1[ks].y;
        }
        sl0 = sl1 = scale_log2;
    } else {
        float big0 = 0.f, big1 = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            big0 = fmaxf(big0, fmaxf(fmaxf(fabsf(__uint_as_float(w0[ks].x << 16)),
                                           fabsf(__uint_as_float(w0[ks].x & 0xffff0000u))),
                                     fmaxf(fabsf(__uint_as_float(w0[ks].y << 16)),
                                           fabsf(__uint_as_float(w0[ks].y & 0xffff0000u)))));
            big1 = fmaxf(big1, fmaxf(fmaxf(fabsf(__uint_as_float(w1[ks].x << 16)),
                                           fabsf(__uint_as_float(w1[ks].x & 0xffff0000u))),
                                     fmaxf(fabsf(__uint_as_float(w1[ks].y << 16)),
                                           fabsf(__uint_as_float(w1[ks].y & 0xffff0000u)))));
        }
        big0 = fmaxf(big0, __shfl_xor_sync(0xffffffffu, big0, 1));
        big0 = fmaxf(big0, __shfl_xor_sync(0xffffffffu, big0, 2));
        big1 = fmaxf(big1, __shfl_xor_sync(0xffffffffu, big1, 1));
        big1 = fmaxf(big1, __shfl_xor_sync(0xffffffffu, big1, 2));
        // big = f * 2^x, f in [0.5, 1): multiply by 2^(15 - x); a zero row keeps x = 0
        int x0 = 0, x1 = 0;
        frexpf(big0, &x0);
        frexpf(big1, &x1);
        const int e0 = min(max(15 - x0, -100), 100);
        const int e1 = min(max(15 - x1, -100), 100);
        const float up0 = __int_as_float((127 + e0) << 23), up1 = __int_as_float((127 + e1) << 23);
        sl0 = scale_log2 * __int_as_float((127 - e0) << 23);
        sl1 = scale_log2 * __int_as_float((127 - e1) << 23);
        auto to_f16 = [](uint32_t w, float up) {
            const __half2 h = __floats2half2_rn(__uint_as_float(w << 16) * up,
                                                __uint_as_float(w & 0xffff0000u) * up);
            return *reinterpret_cast<const uint32_t*>(&h);
        };
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            qa[ks][0] = to_f16(w0[ks].x, up0);
            qa[ks][1] = to_f16(w1[ks].x, up1);
            qa[ks][2] = to_f16(w0[ks].y, up0);
            qa[ks][3] = to_f16(w1[ks].y, up1);
        }
    }
}

}  // namespace pkv
