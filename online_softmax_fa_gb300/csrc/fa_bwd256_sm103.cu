// fa_bwd256_sm103.cu -- attention backward pass at head dimension 256 for
// sm_103a (GB300).
//
// Same gradients as fa_bwd_sm103.cu ("Understanding FlashAttention Pt 1",
// wpnews.pro, section 3.6, recomputation from the saved LSE of "Fix 2" of
// "FlashAttention-2 -- Deeper Math"):
//   P = exp(S - L),  dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),
//   dQ = scale * dS K,  dK = scale * dS^T Q,     D = rowsum(dO * O),
// laid out for d = 256, which the pages list beside 64 and 128.
//
// At d = 256 the tiles outgrow the SM.  A 128-row fp32 accumulator of width
// 256 is half of TMEM, so dV and dK of one key block (512 columns) cannot
// share an SM with the S^T / dP^T tiles, and 128-row K, V, Q, dO tiles are
// 64 KB each in shared memory.  So:
//   * dkdv: two CTAs per 128-key block, one per 128-column slice of dV and
//     dK (S^T and dP^T need all of d, so both CTAs compute them).  V_j stays
//     in shared memory (64 KB) and K_j in TMEM columns [128, 256) (copied
//     there once, with tcgen05.cp, through a shared-memory stage), where the
//     S^T MMAs read it as their A operand; the query rows stream in 64-row
//     halves (Q and dO, 64 KB) through two stages, so a half's loads overlap
//     the previous half's MMAs.  Per half: S^T = K_j Q_h^T and dP^T = V_j
//     dO_h^T (16 K-steps each, N = 64), P^T and dS^T by eight elementwise
//     warps (thread = key row, 32 query columns per warp), then dV_s +=
//     P^T dO_h[:, s] and dK_s += dS^T Q_h[:, s] (N = 128, A from TMEM).
//     TMEM: S^T [0, 64), dP^T [64, 128), K_j [128, 256), dV_s [256, 384),
//     dK_s [384, 512); P^T and dS^T as bf16 pairs over S^T's columns.
//   * dq: one CTA per 128-query block; dO_i stays in shared memory and Q_i
//     in TMEM [128, 256) the same way; the keys stream in 64-row halves (K
//     and V, 64 KB) through two stages.  Per half: S and dP (N = 64), dS
//     (thread = query row), then dQ += dS K_h as one M128 x N256 MMA per 16
//     keys.  TMEM: S [0, 64), dP [64, 128), Q_i [128, 256), dQ [256, 512).
// TMEM holds one S^T / dP^T pair, so a half's MMAs wait for the elementwise
// step of the previous half.  The kernels are deterministic (no atomics,
// fixed order).  Causal: blocks above the diagonal are skipped, the
// diagonal block and a ragged last block masked per element.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_internal.h"
#include "sm103_primitives.cuh"
#include "bwd_elementwise.cuh"

namespace fa {

__device__ int g_fa_status_bwd256;  // bounded-wait timeouts of these kernels

namespace b256 {

constexpr int kD = 256;
constexpr int kBlk = 128;           // keys (dkdv) or queries (dq) per CTA
constexpr int kHalf = 64;           // streamed rows per stage
constexpr int kBox = 128 * 128;     // 128 rows x 64 bf16 (one 128-byte swizzle chunk)
constexpr int kHBox = 64 * 128;     // 64 rows x 64 bf16
constexpr int kTile = 4 * kBox;     // [128 x 256] bf16, four chunks
constexpr int kHTile = 4 * kHBox;   // [64 x 256] bf16, four chunks
constexpr int kThreads = 384;       // 8 elementwise warps, MMA (8), TMA (9), 2 idle
constexpr int kEwWarps = 8;
constexpr int kMmaWarp = 8, kTmaWarp = 9;
constexpr uint32_t kRegsEw = 216, kRegsCtl = 72;  // 128 x (216 + 216 + 72) = 384 x 168
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmS = 0, kTmP = 64, kTmOp = 128, kTmAcc = 256;  // kTmOp: K_j or Q_i
constexpr float kLog2e = 1.4426950408889634f;

// shared memory: the resident tile A (V_j or dO_i); two stages, each the
// streamed half-tiles C (Q_h or K_h) and E (dO_h or V_h); the stages' row
// statistics (dkdv); barriers.  Stage 1 first holds the tile that goes to
// TMEM (K_j or Q_i, 64 KB = one stage).
constexpr int kStages = 2;
constexpr int kStage = 2 * kHTile;
constexpr int kOffA = 0, kOffStage = kTile;
constexpr int kOffRows = kOffStage + kStages * kStage;  // dkdv: per stage -LSE2[64], -D[64]
constexpr int kOffBar = kOffRows + kStages * 2 * kHalf * 4;
// once, full[2], empty[2], s_full, p_full, o_full
constexpr int kNumBars = 8;
constexpr int kOffMisc = kOffBar + 8 * kNumBars;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kIdescSdp = idesc_bf16_f32(kBlk, kHalf, false);      // M128 N64, K-major
constexpr uint32_t kIdescSlice = idesc_bf16_f32(kBlk, 128, true);       // M128 N128, B MN-major
constexpr uint32_t kIdescDq = idesc_bf16_f32(kBlk, kD, true);           // M128 N256, B MN-major

enum : int { kSiteOnce = 0x51, kSiteFull, kSiteEmpty, kSiteS, kSiteP, kSiteO };

struct Params {
    __nv_bfloat16 *g0, *g1;  // dkdv: dK, dV; dq: dQ
    const float *lse2;       // -LSE * log2(e), rows padded to n_blocks * 128 per head
    const float *dd;         // -D
    int N, n_blocks;
    int H, group;            // query heads per batch; query heads per K/V head
    int grid_heads;          // K/V heads (dkdv) or query heads (dq)
    int head_group;          // causal CTA order: heads per group
    float scale, scale_log2;
    uint64_t limit_ns;
};

struct View {
    uint8_t *a, *stage;  // stage s at stage + s * kStage: C, then E
    float *rows;         // stage s's statistics at rows + s * 2 * kHalf
    uint64_t *once, *full, *empty, *s_full, *p_full, *o_full;  // full, empty: [2]
    uint32_t *tmem_slot;
    volatile int *abort_flag;
    __device__ uint8_t *c(int s) const { return stage + s * kStage; }
    __device__ uint8_t *e(int s) const { return stage + s * kStage + kHTile; }
};

__device__ __forceinline__ View view() {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    View v;
    v.a = smem + kOffA;
    v.stage = smem + kOffStage;
    v.rows = reinterpret_cast<float *>(smem + kOffRows);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kOffBar);
    v.once = bar;
    v.full = bar + 1;
    v.empty = bar + 3;
    v.s_full = bar + 5;
    v.p_full = bar + 6;
    v.o_full = bar + 7;
    v.tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    v.abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    return v;
}

// CTA -> (head row, block), causal in cost order within head groups (the
// d <= 128 backward's order); dkdv CTAs come in pairs, one per d-slice.
template <bool CAUSAL, bool KEY_BLOCKS>
__device__ __forceinline__ void block_of(const Params &p, int x, int &bh, int &blk) {
    if (CAUSAL) {
        const int per_group = p.head_group * p.n_blocks;
        const int grp = x / per_group;
        const int in = x - grp * per_group;
        const int h0 = grp * p.head_group;
        const int gsize = min(p.head_group, p.grid_heads - h0);
        const int rank = in / gsize;
        bh = h0 + (in - rank * gsize);
        blk = KEY_BLOCKS ? rank : p.n_blocks - 1 - rank;
    } else {
        bh = x / p.n_blocks;
        blk = x - bh * p.n_blocks;
    }
}

__device__ __forceinline__ int q_head(const Params &p, int kv, int g) {
    const int hkv = p.H / p.group;
    const int b = kv / hkv;
    return b * p.H + (kv - b * hkv) * p.group + g;
}
__device__ __forceinline__ int kv_head(const Params &p, int bh) {
    const int b = bh / p.H;
    return b * (p.H / p.group) + (bh - b * p.H) / p.group;
}

// D[M128 x N64] = A[128 rows x 256] * B[64 rows x 256]^T, both K-major in
// four 64-column swizzled chunks (A chunks 16 KB apart, B chunks 8 KB).
// Unrolled one chunk at a time: the control warps run at 72 registers.
__device__ __forceinline__ void mma_rows_k256(uint32_t d_tm, uint64_t da, uint64_t db) {
#pragma unroll 4
    for (int kk = 0; kk < kD / 16; ++kk) {
        const uint32_t in = (kk & 3) * 32;
        const uint64_t oa = static_cast<uint64_t>(((kk >> 2) * kBox + in) >> 4);
        const uint64_t ob = static_cast<uint64_t>(((kk >> 2) * kHBox + in) >> 4);
        mma_ss_elect(d_tm, da + oa, db + ob, kIdescSdp, kk > 0 ? 1u : 0u);
    }
}

// D[M128 x N64] = A[tmem, 128 x 256 bf16 at kTmOp] * B[64 rows x 256]^T, B
// K-major in four 64-column swizzled chunks 8 KB apart.
__device__ __forceinline__ void mma_tmem_rows_k256(uint32_t d_tm, uint32_t a_tm, uint64_t db) {
#pragma unroll 4
    for (int kk = 0; kk < kD / 16; ++kk) {
        const uint64_t ob = static_cast<uint64_t>(((kk >> 2) * kHBox + (kk & 3) * 32) >> 4);
        mma_ts_elect(d_tm, a_tm + 8 * kk, db + ob, kIdescSdp, kk > 0 ? 1u : 0u);
    }
}

// Copies a [128 x 256] bf16 tile (K-major, four 64-column swizzled chunks
// 16 KB apart, descriptor da) into TMEM columns [a_tm, a_tm + 128) as an A
// operand: K-step kk (16 elements) into columns a_tm + 8 kk.
__device__ __forceinline__ void copy_tile_to_tmem(uint32_t a_tm, uint64_t da) {
#pragma unroll 4
    for (int kk = 0; kk < kD / 16; ++kk) {
        const uint64_t oa = static_cast<uint64_t>(((kk >> 2) * kBox + (kk & 3) * 32) >> 4);
        tmem_cp_128x256b_elect(a_tm + 8 * kk, da + oa);
    }
}

// The producer's wait before it loads half u into stage u & 1.  Stage 0
// holds halves 0, 2, 4, ...; stage 1 first holds the tile copied into TMEM
// (its release is the first completion of empty[1]), then halves 1, 3, ...
__device__ __forceinline__ bool wait_stage_free(const View &v, int u, const WaitCtl &ctl) {
    const int s = u & 1, use = u >> 1;
    if (s == 0) return use == 0 || mbar_wait(&v.empty[0], (use - 1) & 1, ctl, kSiteEmpty);
    return mbar_wait(&v.empty[1], use & 1, ctl, kSiteEmpty);
}

// Drain of the producer's copies on the way out: the resident tiles and the
// last two halves issued (one per stage).
__device__ __forceinline__ void drain_loads(const View &v, int issued, uint64_t limit_ns) {
    mbar_wait_drain(v.once, 0, limit_ns);
    for (int u = max(0, issued - kStages); u < issued; ++u)
        mbar_wait_drain(&v.full[u & 1], (u >> 1) & 1, limit_ns);
}

// acc (+)= A[tmem, 128 x 64 bf16] * B[64 rows x N, MN-major], the A pairs
// of K-steps 0-1 at [a, a + 16), 2-3 at [a + 32, a + 48) (each column-half
// warp writes its 32 columns' bf16 pairs over its first 16).  B's row
// (K-step) stride is 16 rows x 128 bytes.
__device__ __forceinline__ void mma_tmem_k64(uint32_t d_tm, uint32_t a_tm, uint64_t db,
                                             uint32_t idesc, bool acc) {
#pragma unroll
    for (int kk = 0; kk < kHalf / 16; ++kk)
        mma_ts_elect(d_tm, a_tm + (kk >> 1) * 32 + (kk & 1) * 8,
                     db + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc,
                     (acc || kk > 0) ? 1u : 0u);
}

__device__ __forceinline__ void load_rows(uint8_t *dst, int chunk_bytes, const CUtensorMap *m,
                                          uint64_t *bar, int row, int bh, uint64_t pol) {
#pragma unroll
    for (int c = 0; c < 4; ++c) tma_load_3d(dst + c * chunk_bytes, m, bar, 64 * c, row, bh, pol);
}

__device__ __forceinline__ void setup(const View &v) {
    mbar_init(v.once, 1);
    for (int s = 0; s < kStages; ++s) {
        mbar_init(&v.full[s], 1);
        mbar_init(&v.empty[s], 1);
    }
    mbar_init(v.s_full, 1);
    mbar_init(v.p_full, kEwWarps);
    mbar_init(v.o_full, 1);
    *v.abort_flag = 0;
    fence_mbarrier_init();
}

// ============================== dK / dV kernel ==============================
template <bool CAUSAL>
__device__ __forceinline__ void dkdv_producer(const CUtensorMap *tmQh, const CUtensorMap *tmK,
                                            const CUtensorMap *tmV, const CUtensorMap *tmdOh,
                                            const Params &p, int bh, int jb, int lane) {
    if (lane != 0) return;
    const View v = view();
    const WaitCtl ctl{v.abort_flag, &g_fa_status_bwd256, p.limit_ns};
    const int i0 = CAUSAL ? jb : 0;
    const int n_q = p.n_blocks - i0;
    const int n_u = 2 * p.group * n_q;
    const uint64_t pol = l2_policy_evict_last();
    mbar_arrive_expect_tx(v.once, 2 * kTile);
    load_rows(v.a, kBox, tmV, v.once, jb * kBlk, bh, pol);         // V_j, resident
    load_rows(v.c(1), kBox, tmK, v.once, jb * kBlk, bh, pol);      // K_j, for TMEM
    int issued = 0;
    for (int u = 0; u < n_u; ++u) {
        if (!wait_stage_free(v, u, ctl)) break;
        const int s = u & 1;
        const int t = u >> 1, g = t / n_q;
        const int qr = (i0 + t - g * n_q) * kBlk + (u & 1) * kHalf;  // the half's first query
        const int bq = q_head(p, bh, g);
        const size_t prow = static_cast<size_t>(bq) * p.n_blocks * kBlk + qr;
        float *rows = v.rows + s * 2 * kHalf;
        mbar_arrive_expect_tx(&v.full[s], 2 * kHTile + 2 * kHalf * 4);
        load_rows(v.c(s), kHBox, tmQh, &v.full[s], qr, bq, pol);
        load_rows(v.e(s), kHBox, tmdOh, &v.full[s], qr, bq, pol);
        bulk_load(rows, p.lse2 + prow, kHalf * 4, &v.full[s], pol);
        bulk_load(rows + kHalf, p.dd + prow, kHalf * 4, &v.full[s], pol);
        ++issued;
    }
    drain_loads(v, issued, p.limit_ns);
}

template <bool CAUSAL>
__device__ __forceinline__ void dkdv_mma(const Params &p, int jb, int slice) {
    const View v = view();
    const WaitCtl ctl{v.abort_flag, &g_fa_status_bwd256, p.limit_ns};
    const int n_u = 2 * p.group * (p.n_blocks - (CAUSAL ? jb : 0));
    const uint32_t tmem = *v.tmem_slot;
    const auto wait = [&](uint64_t *bar, uint32_t par, int site) {
        return __all_sync(0xffffffffu, mbar_wait(bar, par, ctl, site));
    };
    const uint64_t dV = sdesc_sw128(smem_u32(v.a), 16, 1024);
    // K_j, staged in stage 1, into TMEM; its copies complete (and stage 1 is
    // free) at the first completion of empty[1]
    bool ok = wait(v.once, 0, kSiteOnce);
    if (ok) {
        tc_fence_after();
        copy_tile_to_tmem(tmem + kTmOp, sdesc_sw128(smem_u32(v.c(1)), 16, 1024));
        mma_commit_elect(&v.empty[1]);
        ok = wait(&v.empty[1], 0, kSiteEmpty);
    }
    for (int u = 0; u < n_u && ok; ++u) {
        const int s = u & 1;
        ok = wait(&v.full[s], (u >> 1) & 1, kSiteFull);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dQh = sdesc_sw128(smem_u32(v.c(s)), 16, 1024);
        const uint64_t ddOh = sdesc_sw128(smem_u32(v.e(s)), 16, 1024);
        // the slice's two chunks of Q_h / dO_h as MN-major B operands (N =
        // 128: chunks 2 slice and 2 slice + 1, kHBox apart)
        const uint64_t dQs = sdesc_sw128(smem_u32(v.c(s) + 2 * slice * kHBox), kHBox, 1024);
        const uint64_t ddOs = sdesc_sw128(smem_u32(v.e(s) + 2 * slice * kHBox), kHBox, 1024);
        // S^T and dP^T of this half (the previous half's dV / dK, which read
        // the same TMEM columns, were issued before by this thread)
        mma_tmem_rows_k256(tmem + kTmS, tmem + kTmOp, dQh);
        mma_rows_k256(tmem + kTmP, dV, ddOh);
        mma_commit_elect(v.s_full);
        ok = wait(v.p_full, u & 1, kSiteP);
        if (!ok) break;
        tc_fence_after();
        mma_tmem_k64(tmem + kTmAcc, tmem + kTmS, ddOs, kIdescSlice, u > 0);             // dV_s
        mma_tmem_k64(tmem + kTmAcc + 128, tmem + kTmS + 16, dQs, kIdescSlice, u > 0);  // dK_s
        mma_commit_elect(&v.empty[s]);  // the stage is read
    }
    mma_commit_elect(v.o_full);
    mbar_wait_drain(v.o_full, 0, p.limit_ns);
}

template <bool CAUSAL>
__device__ __forceinline__ void dkdv_elementwise(const Params &p, int bh, int jb, int slice,
                                                 int warp, int lane) {
    const View v = view();
    const WaitCtl ctl{v.abort_flag, &g_fa_status_bwd256, p.limit_ns};
    const int N = p.N;
    const int i0 = CAUSAL ? jb : 0;
    const int n_q = p.n_blocks - i0;
    const int n_u = 2 * p.group * n_q;
    const uint32_t tmem = *v.tmem_slot;
    const int quarter = warp & 3, c = warp >> 2;  // c: queries [32c, 32c + 32) of each half
    const int key = jb * kBlk + quarter * 32 + lane;
    const uint32_t lb = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    for (int u = 0; u < n_u && ok; ++u) {
        const float *rows = v.rows + (u & 1) * 2 * kHalf + 32 * c;
        ok = mbar_wait(&v.full[u & 1], (u >> 1) & 1, ctl, kSiteFull);  // the half's statistics
        if (!ok) break;
        // this warp's 32 columns' statistics into registers before S^T is
        // ready (read during the math, they would wait on shared memory)
        float4 l4[8], d4[8];
#pragma unroll
        for (int t4 = 0; t4 < 8; ++t4) {
            l4[t4] = *reinterpret_cast<const float4 *>(rows + 4 * t4);
            d4[t4] = *reinterpret_cast<const float4 *>(rows + kHalf + 4 * t4);
        }
        ok = mbar_wait(v.s_full, u & 1, ctl, kSiteS);
        if (!ok) break;
        tc_fence_after();
        const int t = u >> 1;
        const int qi = t % n_q;
        const int qh0 = (i0 + qi) * kBlk + (u & 1) * kHalf;  // the half's first query
        // column (query) qh0 + e kept iff qh0 + e < N and, causal, >= key
        const int lim_lo = CAUSAL ? key - qh0 : 0;
        const int lim_hi = N - qh0;
        const bool masked = (CAUSAL && qi == 0) || qh0 + kHalf > N;
        uint32_t sv[32], dv[32], pp[16], pds[16];
        const uint32_t ts = tmem + lb + kTmS + 32 * c, tp = tmem + lb + kTmP + 32 * c;
        tmem_ld32x2(ts, tp, sv, dv);
        if (masked)
            p_ds_masked(sv, dv, rows, rows + kHalf, true, 0.f, 0.f, p.scale_log2, lim_lo, lim_hi,
                        32 * c, pp, pds);
        else
            p_ds_fast_reg(sv, dv, l4, d4, p.scale_log2, pp, pds);
        tmem_st16(ts, pp);         // P^T over the first 16 of this warp's columns
        tmem_st16(ts + 16, pds);   // dS^T over the next 16
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(v.p_full);
    }
    if (ok) ok = mbar_wait(v.o_full, 0, ctl, kSiteO);
    if (ok) {
        tc_fence_after();
        // every lane takes part in the TMEM loads (warp-collective); only
        // rows below N are stored
        const bool in = key < N;
        const size_t row = (static_cast<size_t>(bh) * N + key) * kD + 128 * slice;
        __nv_bfloat16 *dvp = p.g1 + row, *dkp = p.g0 + row;
#pragma unroll 1
        for (int g = 2 * c; g < 2 * c + 2; ++g) {  // 64 of the slice's 128 columns
            uint32_t a[32], b[32], pa[16], pb[16];
            tmem_ld32(tmem + lb + kTmAcc + 32 * g, a);
            tmem_ld32(tmem + lb + kTmAcc + 128 + 32 * g, b);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                pa[e] = pack_bf16x2(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
                pb[e] = pack_bf16x2(__uint_as_float(b[2 * e]) * p.scale,
                                    __uint_as_float(b[2 * e + 1]) * p.scale);
            }
            if (in) {
                uint4 *o0 = reinterpret_cast<uint4 *>(dvp + 32 * g);
                uint4 *o1 = reinterpret_cast<uint4 *>(dkp + 32 * g);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    o0[e] = make_uint4(pa[4 * e], pa[4 * e + 1], pa[4 * e + 2], pa[4 * e + 3]);
                    o1[e] = make_uint4(pb[4 * e], pb[4 * e + 1], pb[4 * e + 2], pb[4 * e + 3]);
                }
            }
        }
    }
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv256_kernel(const __grid_constant__ CUtensorMap tmQh,
                   const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmdOh, const Params p) {
    const View v = view();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slice = static_cast<int>(blockIdx.x & 1);  // the pair of a key block's slices
    int bh, jb;
    block_of<CAUSAL, true>(p, static_cast<int>(blockIdx.x >> 1), bh, jb);
    if (threadIdx.x == 0) setup(v);
    if (warp == kMmaWarp) {
        tmem_alloc(v.tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp >= kMmaWarp) {
        regs_decrease<kRegsCtl>();
        if (warp == kTmaWarp)
            dkdv_producer<CAUSAL>(&tmQh, &tmK, &tmV, &tmdOh, p, bh, jb, lane);
        else if (warp == kMmaWarp)
            dkdv_mma<CAUSAL>(p, jb, slice);
        __syncwarp();
    } else {
        regs_increase<kRegsEw>();
        dkdv_elementwise<CAUSAL>(p, bh, jb, slice, warp, lane);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(*view().tmem_slot, kTmemCols);
    }
}

// ================================= dQ kernel =================================
template <bool CAUSAL>
__device__ __forceinline__ void dq_producer(const CUtensorMap *tmQ, const CUtensorMap *tmKh,
                                          const CUtensorMap *tmVh, const CUtensorMap *tmdO,
                                          const Params &p, int bh, int ib, int lane) {
    if (lane != 0) return;
    const View v = view();
    const WaitCtl ctl{v.abort_flag, &g_fa_status_bwd256, p.limit_ns};
    const int n_u = 2 * (CAUSAL ? ib + 1 : p.n_blocks);
    const int bk = kv_head(p, bh);
    const uint64_t pol_q = l2_policy_evict_first(), pol_kv = l2_policy_evict_last();
    mbar_arrive_expect_tx(v.once, 2 * kTile);
    load_rows(v.a, kBox, tmdO, v.once, ib * kBlk, bh, pol_q);    // dO_i, resident
    load_rows(v.c(1), kBox, tmQ, v.once, ib * kBlk, bh, pol_q);  // Q_i, for TMEM
    int issued = 0;
    for (int u = 0; u < n_u; ++u) {
        if (!wait_stage_free(v, u, ctl)) break;
        const int s = u & 1;
        mbar_arrive_expect_tx(&v.full[s], 2 * kHTile);
        load_rows(v.c(s), kHBox, tmKh, &v.full[s], u * kHalf, bk, pol_kv);
        load_rows(v.e(s), kHBox, tmVh, &v.full[s], u * kHalf, bk, pol_kv);
        ++issued;
    }
    drain_loads(v, issued, p.limit_ns);
}

template <bool CAUSAL>
__device__ __forceinline__ void dq_mma(const Params &p, int ib) {
    const View v = view();
    const WaitCtl ctl{v.abort_flag, &g_fa_status_bwd256, p.limit_ns};
    const int n_u = 2 * (CAUSAL ? ib + 1 : p.n_blocks);
    const uint32_t tmem = *v.tmem_slot;
    const auto wait = [&](uint64_t *bar, uint32_t par, int site) {
        return __all_sync(0xffffffffu, mbar_wait(bar, par, ctl, site));
    };
    const uint64_t ddO = sdesc_sw128(smem_u32(v.a), 16, 1024);
    // Q_i, staged in stage 1, into TMEM (as in the dK / dV kernel)
    bool ok = wait(v.once, 0, kSiteOnce);
    if (ok) {
        tc_fence_after();
        copy_tile_to_tmem(tmem + kTmOp, sdesc_sw128(smem_u32(v.c(1)), 16, 1024));
        mma_commit_elect(&v.empty[1]);
        ok = wait(&v.empty[1], 0, kSiteEmpty);
    }
    for (int u = 0; u < n_u && ok; ++u) {
        const int s = u & 1;
        ok = wait(&v.full[s], (u >> 1) & 1, kSiteFull);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dKh = sdesc_sw128(smem_u32(v.c(s)), 16, 1024);
        const uint64_t dVh = sdesc_sw128(smem_u32(v.e(s)), 16, 1024);
        const uint64_t dKmn = sdesc_sw128(smem_u32(v.c(s)), kHBox, 1024);  // MN-major B, N = 256
        mma_tmem_rows_k256(tmem + kTmS, tmem + kTmOp, dKh);  // S = Q K_h^T
        mma_rows_k256(tmem + kTmP, ddO, dVh);                // dP = dO V_h^T
        mma_commit_elect(v.s_full);
        ok = wait(v.p_full, u & 1, kSiteP);
        if (!ok) break;
        tc_fence_after();
        mma_tmem_k64(tmem + kTmAcc, tmem + kTmS, dKmn, kIdescDq, u > 0);  // dQ += dS K_h
        mma_commit_elect(&v.empty[s]);
    }
    mma_commit_elect(v.o_full);
    mbar_wait_drain(v.o_full, 0, p.limit_ns);
}

template <bool CAUSAL>
__device__ __forceinline__ void dq_elementwise(const Params &p, int bh, int ib, int warp,
                                               int lane) {
    const View v = view();
    const WaitCtl ctl{v.abort_flag, &g_fa_status_bwd256, p.limit_ns};
    const int N = p.N;
    const int n_u = 2 * (CAUSAL ? ib + 1 : p.n_blocks);
    const uint32_t tmem = *v.tmem_slot;
    const int quarter = warp & 3, c = warp >> 2;  // c: keys [32c, 32c + 32) of each half
    const int q = ib * kBlk + quarter * 32 + lane;
    const uint32_t lb = static_cast<uint32_t>(quarter * 32) << 16;
    const size_t prow = static_cast<size_t>(bh) * p.n_blocks * kBlk + q;  // padded row
    const float my_nl2 = p.lse2[prow], my_nd = p.dd[prow];
    bool ok = true;
    for (int u = 0; u < n_u && ok; ++u) {
        ok = mbar_wait(v.s_full, u & 1, ctl, kSiteS);
        if (!ok) break;
        tc_fence_after();
        const int k0 = u * kHalf;  // the half's first key
        // key k0 + e kept iff k0 + e < N and, causal, k0 + e <= q
        const int lim_hi = CAUSAL ? min(N - k0, q - k0 + 1) : N - k0;
        const bool masked = (CAUSAL && k0 + kHalf - 1 > ib * kBlk) || k0 + kHalf > N;
        uint32_t sv[32], dv[32], pp[16], pds[16];
        const uint32_t ts = tmem + lb + kTmS + 32 * c, tp = tmem + lb + kTmP + 32 * c;
        tmem_ld32x2(ts, tp, sv, dv);
        if (masked)
            p_ds_masked(sv, dv, nullptr, nullptr, false, my_nl2, my_nd, p.scale_log2, 0, lim_hi,
                        32 * c, pp, pds);
        else
            p_ds_fast(sv, dv, nullptr, nullptr, false, my_nl2, my_nd, p.scale_log2, pp, pds);
        tmem_st16(ts, pds);  // dS over the first 16 of this warp's columns
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(v.p_full);
    }
    if (ok) ok = mbar_wait(v.o_full, 0, ctl, kSiteO);
    if (ok) {
        tc_fence_after();
        // every lane takes part in the TMEM loads (warp-collective); only
        // rows below N are stored
        const bool in = q < N;
        __nv_bfloat16 *dq = p.g0 + (static_cast<size_t>(bh) * N + q) * kD;
#pragma unroll 1
        for (int g = 4 * c; g < 4 * c + 4; ++g) {  // half of the 256 columns
            uint32_t a[32], pa[16];
            tmem_ld32(tmem + lb + kTmAcc + 32 * g, a);
#pragma unroll
            for (int e = 0; e < 16; ++e)
                pa[e] = pack_bf16x2(__uint_as_float(a[2 * e]) * p.scale,
                                    __uint_as_float(a[2 * e + 1]) * p.scale);
            if (in) {
                uint4 *o = reinterpret_cast<uint4 *>(dq + 32 * g);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    o[e] = make_uint4(pa[4 * e], pa[4 * e + 1], pa[4 * e + 2], pa[4 * e + 3]);
            }
        }
    }
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    dq256_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKh,
                 const __grid_constant__ CUtensorMap tmVh,
                 const __grid_constant__ CUtensorMap tmdO, const Params p) {
    const View v = view();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int bh, ib;
    block_of<CAUSAL, false>(p, static_cast<int>(blockIdx.x), bh, ib);
    if (threadIdx.x == 0) setup(v);
    if (warp == kMmaWarp) {
        tmem_alloc(v.tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp >= kMmaWarp) {
        regs_decrease<kRegsCtl>();
        if (warp == kTmaWarp)
            dq_producer<CAUSAL>(&tmQ, &tmKh, &tmVh, &tmdO, p, bh, ib, lane);
        else if (warp == kMmaWarp)
            dq_mma<CAUSAL>(p, ib);
        __syncwarp();
    } else {
        regs_increase<kRegsEw>();
        dq_elementwise<CAUSAL>(p, bh, ib, warp, lane);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(*view().tmem_slot, kTmemCols);
    }
}

}  // namespace b256

template <bool CAUSAL>
static int launch_bwd256_t(const BwdArgs &a, const float *lse2, const float *dd, int n_blocks) {
    static std::atomic<int> configured1[kMaxDevices], configured2[kMaxDevices];
    int dev = 0;
    FA_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_ARCH;
    auto k1 = b256::dkdv256_kernel<CAUSAL>;
    auto k2 = b256::dq256_kernel<CAUSAL>;
    int rc = set_smem_once(configured1, dev, k1, b256::kSmemBytes);
    if (rc == FA_OK) rc = set_smem_once(configured2, dev, k2, b256::kSmemBytes);
    if (rc != FA_OK) return rc;
    const int sms = device_sm_count(dev);
    b256::Params p;
    p.lse2 = lse2;
    p.dd = dd;
    p.N = a.N;
    p.n_blocks = n_blocks;
    p.H = a.H;
    p.group = a.H / a.Hkv;
    p.scale = a.scale;
    p.scale_log2 = a.scale * b256::kLog2e;
    p.limit_ns = a.limit_ns;
    // causal cost order in head groups, as in the d <= 128 backward
    const long long hg = (3LL * (sms > 0 ? sms : 1) + n_blocks) / (n_blocks + 1);
    const auto set_heads = [&](long long heads) {
        p.grid_heads = static_cast<int>(heads);
        p.head_group = static_cast<int>(hg < 1 ? 1 : (hg > heads ? heads : hg));
        return static_cast<long long>(n_blocks) * heads;
    };
    const long long bh_kv = a.BH / p.group;
    // dK / dV: two CTAs (d-slices) per (K/V head, key block)
    const long long grid1 = 2 * set_heads(bh_kv);
    if (grid1 > 0x7FFFFFFFLL) return FA_ERR_SHAPE;
    p.g0 = static_cast<__nv_bfloat16 *>(a.dK);
    p.g1 = static_cast<__nv_bfloat16 *>(a.dV);
    k1<<<static_cast<unsigned>(grid1), b256::kThreads, b256::kSmemBytes, a.stream>>>(
        *a.tmQ64, *a.tmK, *a.tmV, *a.tmdO64, p);
    FA_CUDA_TRY(cudaGetLastError());
    // dQ: one CTA per (query head, query block)
    const long long grid2 = set_heads(a.BH);
    p.g0 = static_cast<__nv_bfloat16 *>(a.dQ);
    p.g1 = nullptr;
    k2<<<static_cast<unsigned>(grid2), b256::kThreads, b256::kSmemBytes, a.stream>>>(
        *a.tmQ, *a.tmK64, *a.tmV64, *a.tmdO, p);
    FA_CUDA_TRY(cudaGetLastError());
    return FA_OK;
}

int launch_bwd256(const BwdArgs &a, const float *lse2, const float *dd, int n_blocks) {
    return a.causal ? launch_bwd256_t<true>(a, lse2, dd, n_blocks)
                    : launch_bwd256_t<false>(a, lse2, dd, n_blocks);
}

int bwd256_read_and_clear_status(int *status) {
    int v = 0;
    FA_CUDA_TRY(cudaMemcpyFromSymbol(&v, g_fa_status_bwd256, sizeof v));
    if (v != 0) {
        const int zero = 0;
        FA_CUDA_TRY(cudaMemcpyToSymbol(g_fa_status_bwd256, &zero, sizeof zero));
    }
    *status = v;
    return FA_OK;
}

}  // namespace fa
