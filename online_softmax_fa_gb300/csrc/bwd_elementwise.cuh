// bwd_elementwise.cuh -- the elementwise step of the backward kernels
// (fa_bwd_sm103.cu, fa_bwd256_sm103.cu): from a 32-column slice of the
// recomputed scores S (or S^T) and of dP (or dP^T), the probabilities
// P = exp(S - L) of "Fix 2" of "FlashAttention-2 -- Deeper Math" and
// dS = P * (dP - D) of "Understanding FlashAttention Pt 1" (wpnews.pro),
// section 3.6, both rounded to packed bf16 pairs for the MMAs that read them
// from TMEM.  Base 2: p = 2^(s * scale * log2 e - L log2 e).
#pragma once

#include <cstdint>

#include "sm103_primitives.cuh"

namespace fa {

// Elementwise part shared by both kernels, for 32 consecutive columns:
// p = 2^(s*c - lse2), ds = p * (dp - D), returned as packed bf16 pairs.  The
// statistics come negated (nl2 = -lse2, nd = -D): per column from shared
// memory in dkdv (col_stats), per row in registers in dq.
// Fast path (no column masked): packed fp32x2 arithmetic, 16-byte loads.
__device__ __forceinline__ void p_ds_fast(const uint32_t (&s)[32], const uint32_t (&dp)[32],
                                          const float *nl2, const float *nd, bool col_stats,
                                          float my_nl2, float my_nd, float cs,
                                          uint32_t (&pp)[16], uint32_t (&pds)[16]) {
    const uint64_t cs2 = f2_pack(cs, cs);
#pragma unroll
    for (int t4 = 0; t4 < 8; ++t4) {  // four columns at a time
        float4 l4, d4;
        if (col_stats) {
            l4 = *reinterpret_cast<const float4 *>(nl2 + 4 * t4);
            d4 = *reinterpret_cast<const float4 *>(nd + 4 * t4);
        } else {
            l4 = make_float4(my_nl2, my_nl2, my_nl2, my_nl2);
            d4 = make_float4(my_nd, my_nd, my_nd, my_nd);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int t = 2 * t4 + h, e = 2 * t;
            const uint64_t nl = h ? f2_pack(l4.z, l4.w) : f2_pack(l4.x, l4.y);
            const uint64_t nm = h ? f2_pack(d4.z, d4.w) : f2_pack(d4.x, d4.y);
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), cs2, nl),
                      x0, x1);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            const uint64_t p2 = f2_pack(p0, p1);
            float ds0, ds1;
            f2_unpack(f2_mul(p2, f2_add(f2_pack(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])),
                                        nm)),
                      ds0, ds1);
            pp[t] = pack_bf16x2(p0, p1);
            pds[t] = pack_bf16x2(ds0, ds1);
        }
    }
}

// Fast path with the 32 columns' statistics already in registers.
__device__ __forceinline__ void p_ds_fast_reg(const uint32_t (&s)[32], const uint32_t (&dp)[32],
                                              const float4 (&l4)[8], const float4 (&d4)[8],
                                              float cs, uint32_t (&pp)[16], uint32_t (&pds)[16]) {
    const uint64_t cs2 = f2_pack(cs, cs);
#pragma unroll
    for (int t4 = 0; t4 < 8; ++t4) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int t = 2 * t4 + h, e = 2 * t;
            const uint64_t nl = h ? f2_pack(l4[t4].z, l4[t4].w) : f2_pack(l4[t4].x, l4[t4].y);
            const uint64_t nm = h ? f2_pack(d4[t4].z, d4[t4].w) : f2_pack(d4[t4].x, d4[t4].y);
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), cs2, nl),
                      x0, x1);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            const uint64_t p2 = f2_pack(p0, p1);
            float ds0, ds1;
            f2_unpack(f2_mul(p2, f2_add(f2_pack(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])),
                                        nm)),
                      ds0, ds1);
            pp[t] = pack_bf16x2(p0, p1);
            pds[t] = pack_bf16x2(ds0, ds1);
        }
    }
}

// Masked path (diagonal or ragged block): column col0 + e is kept iff
// lim_lo <= col0 + e < lim_hi; p = 0 elsewhere.
__device__ __forceinline__ void p_ds_masked(const uint32_t (&s)[32], const uint32_t (&dp)[32],
                                            const float *nl2, const float *nd, bool col_stats,
                                            float my_nl2, float my_nd, float cs, int lim_lo,
                                            int lim_hi, int col0, uint32_t (&pp)[16],
                                            uint32_t (&pds)[16]) {
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        float p[2], ds[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int e = 2 * t + u;
            const int col = col0 + e;
            const float l2 = col_stats ? nl2[e] : my_nl2;
            const float dv = col_stats ? nd[e] : my_nd;
            const bool keep = col >= lim_lo && col < lim_hi;
            p[u] = keep ? ex2_approx(fmaf(__uint_as_float(s[e]), cs, l2)) : 0.f;
            ds[u] = p[u] * (__uint_as_float(dp[e]) + dv);
        }
        pp[t] = pack_bf16x2(p[0], p[1]);
        pds[t] = pack_bf16x2(ds[0], ds[1]);
    }
}


// P alone (the d = 256 dV kernel role, which needs no dS): p = 2^(s*c -
// lse2) for 32 consecutive columns as packed bf16 pairs, the columns'
// negated statistics nl2 in registers; masked, column col0 + e is kept iff
// lim_lo <= col0 + e < lim_hi (p = 0 elsewhere).
__device__ __forceinline__ float f4_at(const float4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ void p_only_reg(const uint32_t (&s)[32], const float4 (&l4)[8],
                                           float cs, bool masked, int lim_lo, int lim_hi,
                                           int col0, uint32_t (&pp)[16]) {
    if (!masked) {
        const uint64_t cs2 = f2_pack(cs, cs);
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            const int e = 2 * t;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), cs2,
                             f2_pack(f4_at(l4[e >> 2], e & 3), f4_at(l4[e >> 2], (e & 3) + 1))),
                      x0, x1);
            pp[t] = pack_bf16x2(ex2_approx(x0), ex2_approx(x1));
        }
    } else {
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            float pv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int e = 2 * t + u, col = col0 + e;
                const bool keep = col >= lim_lo && col < lim_hi;
                pv[u] = keep ? ex2_approx(fmaf(__uint_as_float(s[e]), cs, f4_at(l4[e >> 2], e & 3)))
                             : 0.f;
            }
            pp[t] = pack_bf16x2(pv[0], pv[1]);
        }
    }
}

}  // namespace fa
