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
//   * dkdv: two CTAs per 128-key block, one for dV and one for dK, each
//     with its 256-column accumulator in TMEM [256, 512) (S^T needs all of
//     d, so both compute it).  Both hold K_j in TMEM columns [128, 256)
//     (copied there once, with tcgen05.cp, through a shared-memory stage),
//     where the S^T MMAs read it as their A operand, and stream the query
//     rows in 64-row halves (Q and dO, 64 KB) through shared-memory stages,
//     so a half's loads overlap the previous half's MMAs.  Per half: S^T =
//     K_j Q_h^T (16 K-steps, N = 64); the dV CTA forms P^T (thread = key
//     row, 32 query columns per warp) and adds P^T dO_h (N = 256, A from
//     TMEM), with S^T double-buffered in [0, 64) and [64, 128) so the next
//     half's S^T overlaps the elementwise step, over three stages; the dK
//     CTA also computes dP^T = V_j dO_h^T (V_j resident in shared memory),
//     forms dS^T and adds dS^T Q_h, with one S^T / dP^T pair ([0, 64),
//     [64, 128)) over two stages.  P^T and dS^T are bf16 pairs written over
//     S^T's columns.
//   * dq: one CTA per 128-query block; dO_i stays in shared memory and Q_i
//     in TMEM [128, 256) the same way; the keys stream in 64-row halves (K
//     and V, 64 KB) through two stages.  Per half: S and dP (N = 64), dS
//     (thread = query row), then dQ += dS K_h as one M128 x N256 MMA per 16
//     keys.  TMEM: S [0, 64), dP [64, 128), Q_i [128, 256), dQ [256, 512).
// In the dK CTA and in dQ, TMEM holds one S^T / dP^T (S / dP) pair, so a
// half's MMAs wait for the elementwise step of the previous half.  The
// kernels are deterministic (no atomics, fixed order).  Causal: blocks above
// the diagonal are skipped, the diagonal block and a ragged last block
// masked per element.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_internal.h"
#include "sm103_primitives.cuh"
#include "bwd_elementwise.cuh"
#include "debug_checks.cuh"

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

// shared memory: three 64 KB regions R0-R2, the row statistics of each
// region (dkdv: -LSE2[64], -D[64]), barriers.  A stage is a region holding
// the streamed half-tiles C (Q_h or K_h) and E (dO_h or V_h).  The dK CTA
// and dQ keep their resident tile (V_j or dO_i) in R0 and stream through
// R1, R2; the dV CTA streams through all three.  R2 first holds the tile
// that goes to TMEM (K_j or Q_i), then serves as the last stage.
constexpr int kRegion = 2 * kHTile;  // 64 KB = one [128 x 256] bf16 tile
constexpr int kRegions = 3;
constexpr int kOffRows = kRegions * kRegion;
constexpr int kOffBar = kOffRows + kRegions * 2 * kHalf * 4;
// once, full[3], empty[3], s_full[2], p_full[2], o_full
constexpr int kNumBars = 12;
constexpr int kOffMisc = kOffBar + 8 * kNumBars;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kIdescSdp = idesc_bf16_f32(kBlk, kHalf, false);      // M128 N64, K-major
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
    uint8_t *base;     // region r at base + r * kRegion: C, then E
    float *rows_base;  // region r's statistics at rows_base + r * 2 * kHalf
    // full, empty: [3], per stage; s_full, p_full: [2], per S^T buffer (the
    // dV CTA double-buffers S^T; the others use [0])
    uint64_t *once, *full, *empty, *s_full, *p_full, *o_full;
    uint32_t *tmem_slot;
    volatile int *abort_flag;
    __device__ uint8_t *c(int r) const { return base + r * kRegion; }
    __device__ uint8_t *e(int r) const { return base + r * kRegion + kHTile; }
    __device__ float *rows(int r) const { return rows_base + r * 2 * kHalf; }
};

__device__ __forceinline__ View view() {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    View v;
    v.base = smem;
    v.rows_base = reinterpret_cast<float *>(smem + kOffRows);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kOffBar);
    v.once = bar;
    v.full = bar + 1;
    v.empty = bar + 4;
    v.s_full = bar + 7;
    v.p_full = bar + 9;
    v.o_full = bar + 11;
    v.tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    v.abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    return v;
}

// CTA -> (head row, block), causal in cost order within head groups (the
// d <= 128 backward's order); dkdv CTAs come in pairs, dV's and dK's.
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

// A ring of STAGES stages over the last STAGES regions: half u goes to
// stage u % STAGES = region (3 - STAGES) + u % STAGES, and is that stage's
// (u / STAGES)-th half.
template <int STAGES>
__device__ __forceinline__ int region_of(int u) {
    return (kRegions - STAGES) + u % STAGES;
}

// The producer's wait before it loads half u.  A stage below the last one
// is free for its k-th half once its (k-1)-th half is released; the last
// stage (R2) first holds the tile copied into TMEM, whose release is the
// first completion of its empty barrier.
template <int STAGES>
__device__ __forceinline__ bool wait_stage_free(const View &v, int u, const WaitCtl &ctl) {
    const int s = u % STAGES, use = u / STAGES;
    const int done = (s == STAGES - 1) ? use : use - 1;  // 0-based completion of empty[s]
    return done < 0 || mbar_wait(&v.empty[s], done & 1, ctl, kSiteEmpty);
}

// Drain of the producer's copies on the way out: the resident tiles and the
// last halves issued (one per stage).
template <int STAGES>
__device__ __forceinline__ void drain_loads(const View &v, int issued, uint64_t limit_ns) {
    mbar_wait_drain(v.once, 0, limit_ns);
    for (int u = max(0, issued - STAGES); u < issued; ++u)
        mbar_wait_drain(&v.full[u % STAGES], (u / STAGES) & 1, limit_ns);
}

// Copies the tile staged in R2 into TMEM [kTmOp, kTmOp + 128) and frees R2:
// the copies complete at the first completion of the last stage's empty
// barrier, which the issuing warp then waits for.
template <int STAGES>
__device__ __forceinline__ bool stage_to_tmem(const View &v, uint32_t tmem, const WaitCtl &ctl) {
    tc_fence_after();
    copy_tile_to_tmem(tmem + kTmOp, sdesc_sw128(smem_u32(v.c(kRegions - 1)), 16, 1024));
    mma_commit_elect(&v.empty[STAGES - 1]);
    return __all_sync(0xffffffffu, mbar_wait(&v.empty[STAGES - 1], 0, ctl, kSiteEmpty));
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
    for (int s = 0; s < 3; ++s) {
        mbar_init(&v.full[s], 1);
        mbar_init(&v.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
        mbar_init(&v.s_full[b], 1);
        mbar_init(&v.p_full[b], kEwWarps);
    }
    mbar_init(v.o_full, 1);
    *v.abort_flag = 0;
    fence_mbarrier_init();
}

// ============================== dK / dV kernel ==============================
// Two CTAs per (K/V head, key block j): the dV CTA (even blockIdx) and the
// dK CTA (odd).  Both hold K_j in TMEM [128, 256) and stream Q and dO in
// 64-query halves; both compute S^T = K_j Q_h^T.
//   * dV CTA: P^T = 2^(S^T c - LSE2) and dV += P^T dO_h (no dP, no dS).  S^T
//     is double-buffered in TMEM ([0, 64) and [64, 128)), so S^T of the next
//     half runs while the elementwise warps work on this one; three stages.
//     TMEM: S^T x 2, K_j, dV [256, 512).
//   * dK CTA: dP^T = V_j dO_h^T (V_j resident in R0), dS^T = P^T (dP^T - D),
//     dK += dS^T Q_h.  TMEM: S^T [0, 64), dP^T [64, 128), K_j, dK [256, 512);
//     one S^T / dP^T pair, so the elementwise step waits for the MMAs and
//     the MMAs for it; two stages.
template <bool DV>
struct Role {
    static constexpr int kStages = DV ? 3 : 2;
};

template <bool CAUSAL, bool DV>
__device__ __forceinline__ void dkdv_producer(const CUtensorMap *tmQh, const CUtensorMap *tmK,
                                            const CUtensorMap *tmV, const CUtensorMap *tmdOh,
                                            const Params &p, int bh, int jb, int lane) {
    constexpr int S = Role<DV>::kStages;
    if (lane != 0) return;
    const View v = view();
    const WaitCtl ctl{v.abort_flag, &g_fa_status_bwd256, p.limit_ns};
    const int i0 = CAUSAL ? jb : 0;
    const int n_q = p.n_blocks - i0;
    const int n_u = 2 * p.group * n_q;
    if (!dbg_ok(bh >= 0 && bh < p.grid_heads && jb >= 0 && jb < p.n_blocks &&
                    in_smem(v.c(0), kRegions * kRegion, kSmemBytes),
                ctl, kChkItem))
        return;
    const uint64_t pol = l2_policy_evict_last();
    mbar_arrive_expect_tx(v.once, DV ? kTile : 2 * kTile);
    if (!DV) load_rows(v.c(0), kBox, tmV, v.once, jb * kBlk, bh, pol);  // V_j, resident
    load_rows(v.c(kRegions - 1), kBox, tmK, v.once, jb * kBlk, bh, pol);  // K_j, for TMEM
    int issued = 0;
    for (int u = 0; u < n_u; ++u) {
        if (!wait_stage_free<S>(v, u, ctl)) break;
        const int s = u % S, r = region_of<S>(u);
        const int t = u >> 1, g = t / n_q;
        const int qr = (i0 + t - g * n_q) * kBlk + (u & 1) * kHalf;  // the half's first query
        const int bq = q_head(p, bh, g);
        const size_t prow = static_cast<size_t>(bq) * p.n_blocks * kBlk + qr;
        float *rows = v.rows(r);
        if (!dbg_ok(bq >= 0 && bq < p.grid_heads * p.group && qr >= 0 &&
                        qr < p.n_blocks * kBlk &&
                        prow + kHalf <= static_cast<size_t>(p.grid_heads) * p.group *
                                            p.n_blocks * kBlk,
                    ctl, kChkTmaQ) ||
            !dbg_ok(in_smem(rows, 2 * kHalf * 4, kSmemBytes), ctl, kChkSmem))
            break;
        mbar_arrive_expect_tx(&v.full[s], 2 * kHTile + (DV ? 1 : 2) * kHalf * 4);
        load_rows(v.c(r), kHBox, tmQh, &v.full[s], qr, bq, pol);
        load_rows(v.e(r), kHBox, tmdOh, &v.full[s], qr, bq, pol);
        bulk_load(rows, p.lse2 + prow, kHalf * 4, &v.full[s], pol);
        if (!DV) bulk_load(rows + kHalf, p.dd + prow, kHalf * 4, &v.full[s], pol);
        ++issued;
    }
    drain_loads<S>(v, issued, p.limit_ns);
}

template <bool CAUSAL, bool DV>
__device__ __forceinline__ void dkdv_mma(const Params &p, int jb) {
    constexpr int S = Role<DV>::kStages;
    const View v = view();
    const WaitCtl ctl{v.abort_flag, &g_fa_status_bwd256, p.limit_ns};
    const int n_u = 2 * p.group * (p.n_blocks - (CAUSAL ? jb : 0));
    const uint32_t tmem = *v.tmem_slot;
    const auto wait = [&](uint64_t *bar, uint32_t par, int site) {
        return __all_sync(0xffffffffu, mbar_wait(bar, par, ctl, site));
    };
    bool ok = dbg_ok(whole_tmem(tmem), ctl, kChkTmem) && wait(v.once, 0, kSiteOnce);
    if (ok) ok = stage_to_tmem<S>(v, tmem, ctl);  // K_j
    if (DV) {
        // S^T(u + 1) into the other buffer before dV(u): the buffer last
        // held P^T(u - 1), read by dV(u - 1), issued before by this thread
        const auto issue_s = [&](int u) {
            const bool good = wait(&v.full[u % S], (u / S) & 1, kSiteFull);
            if (good) {
                tc_fence_after();
                mma_tmem_rows_k256(tmem + kTmS + 64 * (u & 1), tmem + kTmOp,
                                   sdesc_sw128(smem_u32(v.c(region_of<S>(u))), 16, 1024));
                mma_commit_elect(&v.s_full[u & 1]);
            }
            return good;
        };
        if (ok && n_u > 0) ok = issue_s(0);
        for (int u = 0; u < n_u && ok; ++u) {
            if (u + 1 < n_u) ok = issue_s(u + 1);
            if (ok) ok = wait(&v.p_full[u & 1], (u >> 1) & 1, kSiteP);
            if (!ok) break;
            tc_fence_after();
            // dV += P^T dO_h: dO_h as the MN-major B operand, N = 256
            mma_tmem_k64(tmem + kTmAcc, tmem + kTmS + 64 * (u & 1),
                         sdesc_sw128(smem_u32(v.e(region_of<S>(u))), kHBox, 1024), kIdescDq,
                         u > 0);
            mma_commit_elect(&v.empty[u % S]);  // the stage is read
        }
    } else {
        const uint64_t dV = sdesc_sw128(smem_u32(v.c(0)), 16, 1024);
        for (int u = 0; u < n_u && ok; ++u) {
            const int s = u % S, r = region_of<S>(u);
            ok = wait(&v.full[s], (u / S) & 1, kSiteFull);
            if (!ok) break;
            tc_fence_after();
            // S^T and dP^T of this half (the previous half's dK, which read
            // the same TMEM columns, was issued before by this thread)
            mma_tmem_rows_k256(tmem + kTmS, tmem + kTmOp, sdesc_sw128(smem_u32(v.c(r)), 16, 1024));
            mma_rows_k256(tmem + kTmP, dV, sdesc_sw128(smem_u32(v.e(r)), 16, 1024));
            mma_commit_elect(&v.s_full[0]);
            ok = wait(&v.p_full[0], u & 1, kSiteP);
            if (!ok) break;
            tc_fence_after();
            // dK += dS^T Q_h: Q_h as the MN-major B operand, N = 256
            mma_tmem_k64(tmem + kTmAcc, tmem + kTmS, sdesc_sw128(smem_u32(v.c(r)), kHBox, 1024),
                         kIdescDq, u > 0);
            mma_commit_elect(&v.empty[s]);  // the stage is read
        }
    }
    mma_commit_elect(v.o_full);
    mbar_wait_drain(v.o_full, 0, p.limit_ns);
}

template <bool CAUSAL, bool DV>
__device__ __forceinline__ void dkdv_elementwise(const Params &p, int bh, int jb, int warp,
                                                 int lane) {
    constexpr int S = Role<DV>::kStages;
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
    // wait results made warp-uniform: the warp reaches its collective TMEM
    // loads together or not at all
    const auto wait = [&](uint64_t *bar, uint32_t par, int site) {
        return __all_sync(0xffffffffu, mbar_wait(bar, par, ctl, site));
    };
    bool ok = dbg_ok(whole_tmem(tmem), ctl, kChkTmem);
    for (int u = 0; u < n_u && ok; ++u) {
        const float *rows = v.rows(region_of<S>(u)) + 32 * c;
        ok = wait(&v.full[u % S], (u / S) & 1, kSiteFull);  // the half's statistics
        if (!ok) break;
        // this warp's 32 columns' statistics into registers before S^T is
        // ready (read during the math, they would wait on shared memory)
        float4 l4[8], d4[8];
#pragma unroll
        for (int t4 = 0; t4 < 8; ++t4) {
            l4[t4] = *reinterpret_cast<const float4 *>(rows + 4 * t4);
            if (!DV) d4[t4] = *reinterpret_cast<const float4 *>(rows + kHalf + 4 * t4);
        }
        const int b = DV ? (u & 1) : 0;
        ok = wait(&v.s_full[b], (DV ? (u >> 1) : u) & 1, kSiteS);
        if (!ok) break;
        tc_fence_after();
        const int t = u >> 1;
        const int qi = t % n_q;
        const int qh0 = (i0 + qi) * kBlk + (u & 1) * kHalf;  // the half's first query
        // column (query) qh0 + e kept iff qh0 + e < N and, causal, >= key
        const int lim_lo = CAUSAL ? key - qh0 : 0;
        const int lim_hi = N - qh0;
        const bool masked = (CAUSAL && qi == 0) || qh0 + kHalf > N;
        const uint32_t ts = tmem + lb + kTmS + 64 * b + 32 * c;
        uint32_t pp[16];
        if (DV) {
            uint32_t sv[32];
            tmem_ld32(ts, sv);
            p_only_reg(sv, l4, p.scale_log2, masked, lim_lo, lim_hi, 32 * c, pp);
            tmem_st16(ts, pp);  // P^T over the first 16 of this warp's columns
        } else {
            uint32_t sv[32], dv[32], pds[16];
            tmem_ld32x2(ts, tmem + lb + kTmP + 32 * c, sv, dv);
            if (masked)
                p_ds_masked(sv, dv, rows, rows + kHalf, true, 0.f, 0.f, p.scale_log2, lim_lo,
                            lim_hi, 32 * c, pp, pds);
            else
                p_ds_fast_reg(sv, dv, l4, d4, p.scale_log2, pp, pds);
            tmem_st16(ts, pds);  // dS^T over the first 16 of this warp's columns
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&v.p_full[b]);
    }
    if (ok) ok = wait(v.o_full, 0, kSiteO);
    if (ok) {
        tc_fence_after();
        // every lane takes part in the TMEM loads (warp-collective); only
        // rows below N are stored.  dV unscaled, dK times the scale.
        const bool in = key < N;
        const float mul = DV ? 1.f : p.scale;
        __nv_bfloat16 *dst = (DV ? p.g1 : p.g0) + (static_cast<size_t>(bh) * N + key) * kD;
#pragma unroll 1
        for (int g = 4 * c; g < 4 * c + 4; ++g) {  // half of the 256 columns
            uint32_t a[32], pa[16];
            tmem_ld32(tmem + lb + kTmAcc + 32 * g, a);
#pragma unroll
            for (int e = 0; e < 16; ++e)
                pa[e] = pack_bf16x2(__uint_as_float(a[2 * e]) * mul,
                                    __uint_as_float(a[2 * e + 1]) * mul);
            if (in && dbg_ok(static_cast<size_t>(bh) * N + key <
                                     static_cast<size_t>(p.grid_heads) * N &&
                                 (reinterpret_cast<uintptr_t>(dst + 32 * g) & 15u) == 0,
                             ctl, kChkStoreO)) {
                uint4 *o = reinterpret_cast<uint4 *>(dst + 32 * g);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    o[e] = make_uint4(pa[4 * e], pa[4 * e + 1], pa[4 * e + 2], pa[4 * e + 3]);
            }
        }
    }
}

template <bool CAUSAL, bool DV>
__device__ __forceinline__ void dkdv_role(const CUtensorMap *tmQh, const CUtensorMap *tmK,
                                          const CUtensorMap *tmV, const CUtensorMap *tmdOh,
                                          const Params &p, int bh, int jb, int warp, int lane) {
    if (warp >= kMmaWarp) {
        regs_decrease<kRegsCtl>();
        if (warp == kTmaWarp)
            dkdv_producer<CAUSAL, DV>(tmQh, tmK, tmV, tmdOh, p, bh, jb, lane);
        else if (warp == kMmaWarp)
            dkdv_mma<CAUSAL, DV>(p, jb);
        __syncwarp();
    } else {
        regs_increase<kRegsEw>();
        dkdv_elementwise<CAUSAL, DV>(p, bh, jb, warp, lane);
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
    const bool dv_cta = (blockIdx.x & 1) == 0;  // the pair of a key block: dV, then dK
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
    if (dv_cta)
        dkdv_role<CAUSAL, true>(&tmQh, &tmK, &tmV, &tmdOh, p, bh, jb, warp, lane);
    else
        dkdv_role<CAUSAL, false>(&tmQh, &tmK, &tmV, &tmdOh, p, bh, jb, warp, lane);
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
    if (!dbg_ok(bh >= 0 && bh < p.grid_heads && ib >= 0 && ib < p.n_blocks &&
                    in_smem(v.c(0), kRegions * kRegion, kSmemBytes),
                ctl, kChkItem))
        return;
    const uint64_t pol_q = l2_policy_evict_first(), pol_kv = l2_policy_evict_last();
    mbar_arrive_expect_tx(v.once, 2 * kTile);
    load_rows(v.c(0), kBox, tmdO, v.once, ib * kBlk, bh, pol_q);             // dO_i, resident
    load_rows(v.c(kRegions - 1), kBox, tmQ, v.once, ib * kBlk, bh, pol_q);  // Q_i, for TMEM
    int issued = 0;
    for (int u = 0; u < n_u; ++u) {
        if (!wait_stage_free<2>(v, u, ctl)) break;
        const int s = u & 1, r = region_of<2>(u);
        if (!dbg_ok(u * kHalf < p.n_blocks * kBlk && bk >= 0 && bk < p.grid_heads / p.group,
                    ctl, kChkTmaKV))
            break;
        mbar_arrive_expect_tx(&v.full[s], 2 * kHTile);
        load_rows(v.c(r), kHBox, tmKh, &v.full[s], u * kHalf, bk, pol_kv);
        load_rows(v.e(r), kHBox, tmVh, &v.full[s], u * kHalf, bk, pol_kv);
        ++issued;
    }
    drain_loads<2>(v, issued, p.limit_ns);
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
    const uint64_t ddO = sdesc_sw128(smem_u32(v.c(0)), 16, 1024);
    bool ok = dbg_ok(whole_tmem(tmem), ctl, kChkTmem) && wait(v.once, 0, kSiteOnce);
    if (ok) ok = stage_to_tmem<2>(v, tmem, ctl);  // Q_i
    for (int u = 0; u < n_u && ok; ++u) {
        const int s = u & 1, r = region_of<2>(u);
        ok = wait(&v.full[s], (u >> 1) & 1, kSiteFull);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dKh = sdesc_sw128(smem_u32(v.c(r)), 16, 1024);
        const uint64_t dVh = sdesc_sw128(smem_u32(v.e(r)), 16, 1024);
        const uint64_t dKmn = sdesc_sw128(smem_u32(v.c(r)), kHBox, 1024);  // MN-major B, N = 256
        mma_tmem_rows_k256(tmem + kTmS, tmem + kTmOp, dKh);  // S = Q K_h^T
        mma_rows_k256(tmem + kTmP, ddO, dVh);                // dP = dO V_h^T
        mma_commit_elect(&v.s_full[0]);
        ok = wait(&v.p_full[0], u & 1, kSiteP);
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
    bool ok = dbg_ok(whole_tmem(tmem), ctl, kChkTmem);
    for (int u = 0; u < n_u && ok; ++u) {
        ok = __all_sync(0xffffffffu, mbar_wait(&v.s_full[0], u & 1, ctl, kSiteS));
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
        if (lane == 0) mbar_arrive(&v.p_full[0]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(v.o_full, 0, ctl, kSiteO));
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
            if (in && dbg_ok(static_cast<size_t>(bh) * N + q <
                                     static_cast<size_t>(p.grid_heads) * N &&
                                 (reinterpret_cast<uintptr_t>(dq + 32 * g) & 15u) == 0,
                             ctl, kChkStoreO)) {
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
    // dK / dV: two CTAs (dV's, then dK's) per (K/V head, key block)
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
