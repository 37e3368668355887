// fa_bwd_sm103.cu -- attention backward pass for sm_103a (GB300).
//
// Gradients of O = softmax(scale * Q K^T [+causal]) V for an output gradient
// dO, by recomputation ("Understanding FlashAttention Pt 1", wpnews.pro,
// section 3.6 "Backward Pass: Recompute Instead of Save"): the probability
// tiles are rebuilt from the saved per-row LSE ("Fix 2" of "FlashAttention-2
// -- Deeper Math": P_ij = exp(S_ij - L_i)) instead of being stored, and
//   dV += P^T dO,  dP = dO V^T,  dS = P * (dP - D_i),
//   dQ += scale * dS K,  dK += scale * dS^T Q,
// with D_i = sum_r dO_ir O_ir.
//
// Three kernels, all deterministic (no atomics, fixed summation order):
//   * pre:  D = rowsum(dO * O) in fp32 and LSE * log2(e), one warp per row,
//           into rows padded to a multiple of 128 per head (the workspace)
//           so that the dkdv producer fetches a block's rows with bulk copies.
//   * dkdv: one CTA per (b, K/V head, 128-key block j), the query blocks i
//           of every query head of the K/V head's group as the inner loop
//           (one head per group without grouped-query attention), each
//           taken in two 64-query halves.  On tcgen05 with TMEM
//           accumulators: S^T = K_j Q_h^T and dP^T = V_j dO_h^T (keys are
//           the MMA rows) for one half while eight elementwise warps
//           (thread = key row = TMEM lane, two warps per row, 32 columns
//           each) form P^T and dS^T in bf16 for the previous half, then
//           dV_j += P^T dO_h and dK_j += dS^T Q_h read them from TMEM.
//           Two warps issue the MMAs: one S^T / dP^T, one dV / dK.
//   * dq:   one CTA per (b, h, 128-query block i), key blocks j of K/V head
//           h / group inner:
//           S = Q_i K_j^T and dP = dO_i V_j^T, then dS (thread = query row),
//           then dQ_i += dS K_j; S is double-buffered, so the next block's S
//           and dP run on the tensor pipe while the warps work on this one.
// Causal: blocks entirely above the diagonal are skipped; the diagonal block
// is masked.  Causal CTAs run in cost order (heaviest first) within groups
// of heads small enough to share L2.  TMEM (dkdv): S^T of the two halves at
// [0,64) and [64,128), dP^T at [128,192) and [192,256), dV [256,256+d),
// dK [256+d, 256+2d); P^T and
// dS^T of a half are bf16 pairs over its S^T columns, each column-half warp
// writing over its own 32 columns (P^T over the first 16, dS^T over the
// next 16).  TMEM (dq): S [0,128) and [128,256), dP [256,384), dQ [384,384+d).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_internal.h"
#include "sm103_primitives.cuh"
#include "bwd_elementwise.cuh"
#include "debug_checks.cuh"

namespace fa {

// Device status word of the backward kernels (read with the forward's by
// fa_device_error): 0 or the site of the first bounded wait that expired.
__device__ int g_fa_status_bwd;

namespace bwd {

constexpr int kBlk = 128;             // rows per block (keys or queries)
constexpr int kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 64 bf16
constexpr int kEwWarps = 8;           // elementwise warps: 4 lane quarters x 2 column halves
constexpr int kThreads = 384;         // 3 warpgroups: 8 elementwise warps, MMA (warp 8; dkdv also 10), TMA (9)
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
// Registers after reallocation: 128 x (216 + 216 + 72) = 64512 = 384 x 168.
constexpr uint32_t kRegsEw = 216;
constexpr uint32_t kRegsCtl = 72;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

enum : int { kSiteKV = 0x21, kSiteQ, kSiteS, kSiteP, kSiteO, kSiteEmpty };

template <int D>
struct Cfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kTile = kChunks * kBoxBytes;  // one [128 x D] bf16 tile
    // dkdv: K_j, V_j once; a ring of kStages stages of (Q_i, dO_i) tiles and
    // their LSE2 / D rows.  dq: Q_i, dO_i once; a ring of kStagesK K tiles and
    // one of kStagesV V tiles (V is released as soon as dP has read it, K only
    // after dQ, so K runs a stage further ahead).
    static constexpr int kStages = 2;
    static constexpr int kStagesK = 3, kStagesV = 2;
    static constexpr int kOffA = 0;                 // K_j (dkdv) / Q_i (dq)
    static constexpr int kOffB = kTile;             // V_j (dkdv) / dO_i (dq)
    static constexpr int kOffRing = 2 * kTile;
    static constexpr int kOffRows = kOffRing + kStages * 2 * kTile;  // dkdv: LSE2, D per stage
    static constexpr int kRingDkdv = kStages * 2 * kTile + kStages * 2 * kBlk * 4;
    static constexpr int kRingDq = (kStagesK + kStagesV) * kTile;
    static constexpr int kOffVq = kOffRing + kStagesK * kTile;      // dq: V ring
    static constexpr int kOffBar = kOffRing + (kRingDkdv > kRingDq ? kRingDkdv : kRingDq);
    // once, full/empty[3] (dkdv: stages; dq: K ring), vfull/vempty[2] (dq: V
    // ring; dkdv: vfull[2] = buf_free of the two S^T/dP^T half buffers),
    // s_full[2], p_full[2], o_full, dp_free (dq)
    static constexpr int kNumBars = 1 + 2 * 3 + 2 * 2 + 6;
    static_assert(kStages <= 3 && kStagesK <= 3 && kStagesV <= 2, "barrier slots");
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
    static constexpr uint32_t kTmS = 0, kTmP = 128, kTmAcc0 = 256, kTmAcc1 = 256 + D;
    static constexpr uint32_t kIdescS = idesc_bf16_f32(kBlk, kBlk, false);
    static constexpr uint32_t kIdescHalf = idesc_bf16_f32(kBlk, kBlk / 2, false);
    static constexpr uint32_t kIdescAcc = idesc_bf16_f32(kBlk, D, true);
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// TMEM of the dQ kernel: S double-buffered, dP, dQ.
constexpr uint32_t kTmSq = 0, kTmPq = 256, kTmAccq = 384;
static_assert(kTmAccq + 128 <= kTmemCols, "TMEM budget of the dQ kernel");

struct Params {
    __nv_bfloat16 *g0, *g1;  // dkdv: dK, dV; dq: dQ
    // per query row, padded to n_blocks * 128 rows per head (zeros past N),
    // negated so that the elementwise step adds them:
    const float *lse2;  // -LSE * log2(e)
    const float *dd;    // -D, D = rowsum(dO * O)
    int N, BH, n_blocks;
    int H, group;     // query heads per batch; query heads per K/V head
    int grid_heads;   // heads the grid walks: K/V heads (dkdv) or query heads (dq)
    int head_group;   // causal CTA order: heads per group (see block_of)
    float scale, scale_log2;
    uint64_t limit_ns;
};

template <int D>
struct View {
    uint8_t *a, *b, *ring;
    float *rows;
    uint8_t *vring;  // dq: V ring
    uint64_t *once, *full, *empty, *vfull, *vempty, *s_full, *p_full, *o_full, *dp_free;
    uint32_t *tmem_slot;
    volatile int *abort_flag;
};

template <int D>
__device__ __forceinline__ View<D> view() {
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    View<D> v;
    v.a = smem + C::kOffA;
    v.b = smem + C::kOffB;
    v.ring = smem + C::kOffRing;
    v.vring = smem + C::kOffVq;
    v.rows = reinterpret_cast<float *>(smem + C::kOffRows);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    v.once = bar;
    v.full = bar + 1;
    v.empty = v.full + 3;
    v.vfull = v.empty + 3;
    v.vempty = v.vfull + 2;
    v.s_full = v.vempty + 2;
    v.p_full = v.s_full + 2;
    v.o_full = v.p_full + 2;
    v.dp_free = v.o_full + 1;
    v.tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    v.abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    return v;
}

// M128 x N128 x K(D) with both operands K-major [rows x D] in swizzled chunks.
template <int D>
__device__ __forceinline__ void mma_rows_rows(uint32_t d_tm, uint64_t da, uint64_t db) {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
        mma_ss_elect(d_tm, da + off, db + off, Cfg<D>::kIdescS, kk > 0 ? 1u : 0u);
    }
}

// acc[M128 x N(D)] (+)= A[tmem, 128 x 128 bf16] * B[128 rows x D, MN-major].
// A's bf16 pairs sit in two column groups (written by the two column-half
// warps over their own fp32 columns): K-steps 0-3 at columns [a_off,
// a_off + 32), 4-7 at [64 + a_off, 96 + a_off) of the region.
template <int D>
__device__ __forceinline__ void mma_tmem_rows(uint32_t d_tm, uint32_t a_tm, uint64_t db, bool acc,
                                              uint32_t a_off = 0) {
#pragma unroll
    for (int kk = 0; kk < kBlk / 16; ++kk)
        mma_ts_elect(d_tm, a_tm + (kk >> 2) * 64 + a_off + (kk & 3) * 8,
                     db + static_cast<uint64_t>((kk * 16 * 128) >> 4), Cfg<D>::kIdescAcc,
                     (acc || kk > 0) ? 1u : 0u);
}

// M128 x N64 x K(D) for one 64-query half of a block: A = K_j or V_j,
// B = the half's 64 rows of Q_i or dO_i (both K-major; the caller adds the
// half's row offset, 64 rows = 8192 bytes = whole swizzle atoms, to B).
template <int D>
__device__ __forceinline__ void mma_rows_half(uint32_t d_tm, uint64_t da, uint64_t db) {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
        mma_ss_elect(d_tm, da + off, db + off, Cfg<D>::kIdescHalf, kk > 0 ? 1u : 0u);
    }
}

// acc[M128 x N(D)] (+)= A[tmem, 128 x 64 bf16] * B[64 rows x D, MN-major]
// for one 64-query half.  A's bf16 pairs sit in two column groups (each
// written by one column-half warp over its own 32 fp32 columns): K-steps 0-1
// at [a, a + 16), 2-3 at [a + 32, a + 48).
template <int D>
__device__ __forceinline__ void mma_tmem_half(uint32_t d_tm, uint32_t a_tm, uint64_t db,
                                              bool acc) {
#pragma unroll
    for (int kk = 0; kk < kBlk / 32; ++kk)
        mma_ts_elect(d_tm, a_tm + (kk >> 1) * 32 + (kk & 1) * 8,
                     db + static_cast<uint64_t>((kk * 16 * 128) >> 4), Cfg<D>::kIdescAcc,
                     (acc || kk > 0) ? 1u : 0u);
}

template <int D>
__device__ __forceinline__ void load_tile(uint8_t *dst, const CUtensorMap *m, uint64_t *bar,
                                          int row, int bh, uint64_t pol) {
#pragma unroll
    for (int c = 0; c < Cfg<D>::kChunks; ++c)
        tma_load_3d(dst + c * kBoxBytes, m, bar, 64 * c, row, bh, pol);
}

__device__ __forceinline__ void setup_barriers(uint64_t *once, uint64_t *full, uint64_t *empty,
                                               uint64_t *vfull, uint64_t *vempty,
                                               uint64_t *s_full, uint64_t *p_full,
                                               uint64_t *o_full, uint64_t *dp_free,
                                               volatile int *abort_flag) {
    mbar_init(once, 1);
    for (int s = 0; s < 3; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
        mbar_init(&vfull[s], 1);
        mbar_init(&vempty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(&p_full[0], kEwWarps);
    mbar_init(&p_full[1], kEwWarps);
    mbar_init(o_full, 1);
    mbar_init(dp_free, kEwWarps);
    *abort_flag = 0;
    fence_mbarrier_init();
}

// CTA -> (batch x head row, block).  Causal: the heads are taken in groups
// of head_group, and within a group the CTAs run in cost order, heaviest
// first (key block jb is used by n_blocks - jb query blocks, query block ib
// by ib + 1 key blocks), so the longest CTAs start early instead of in the
// last wave, while the CTAs in flight share a group's K/V/Q/dO in L2 (the
// host sizes the group so that its heaviest CTAs still start early enough).
// Otherwise head-major.
template <bool CAUSAL, bool KEY_BLOCKS>
__device__ __forceinline__ void block_of(const Params &p, int &bh, int &blk) {
    const int x = static_cast<int>(blockIdx.x);
    if (CAUSAL) {
        const int per_group = p.head_group * p.n_blocks;
        const int grp = x / per_group;
        const int in = x - grp * per_group;
        const int h0 = grp * p.head_group;
        const int gsize = min(p.head_group, p.grid_heads - h0);  // the last group may be smaller
        const int rank = in / gsize;
        bh = h0 + (in - rank * gsize);
        blk = KEY_BLOCKS ? rank : p.n_blocks - 1 - rank;
    } else {
        bh = x / p.n_blocks;
        blk = x - bh * p.n_blocks;
    }
}

// Grouped-query attention: query head q_head(p, kv, g) is member g of K/V
// head kv's group (query head h of a batch uses K/V head h / group).
__device__ __forceinline__ int q_head(const Params &p, int kv, int g) {
    const int hkv = p.H / p.group;  // K/V heads per batch
    const int b = kv / hkv;
    return b * p.H + (kv - b * hkv) * p.group + g;
}
__device__ __forceinline__ int kv_head(const Params &p, int bh) {
    const int b = bh / p.H;
    return b * (p.H / p.group) + (bh - b * p.H) / p.group;
}

// ============================== dK / dV kernel ==============================
template <int D, bool CAUSAL>
__device__ __forceinline__ void dkdv_producer(const CUtensorMap *tmQ, const CUtensorMap *tmK,
                                            const CUtensorMap *tmV, const CUtensorMap *tmdO,
                                            const Params &p, int lane) {
    using C = Cfg<D>;
    const View<D> v = view<D>();
    int bh, jb;  // bh: K/V head; jb: key block
    block_of<CAUSAL, true>(p, bh, jb);
    const int i0 = CAUSAL ? jb : 0;          // first query block touching this key block
    const int n_q = p.n_blocks - i0;         // query blocks per query head
    const WaitCtl ctl{v.abort_flag, &g_fa_status_bwd, p.limit_ns};
    // ---- producer: K_j, V_j once; then, for each query head of the K/V
    // head's group in turn, per query block Q_i, dO_i (TMA) and the block's
    // LSE2 and D rows (bulk copies of the padded rows), all completing the
    // stage's barrier
    if (lane == 0 &&
        dbg_ok(bh >= 0 && bh < p.grid_heads && jb >= 0 && jb < p.n_blocks &&
                   in_smem(v.a, 2 * C::kTile, C::kSmemBytes),
               ctl, kChkItem)) {
        const uint64_t pol = l2_policy_evict_last();
        mbar_arrive_expect_tx(v.once, 2 * C::kTile);
        load_tile<D>(v.a, tmK, v.once, jb * kBlk, bh, pol);
        load_tile<D>(v.b, tmV, v.once, jb * kBlk, bh, pol);
        int issued = 0;
        bool ok = true;
        for (int t = 0; t < p.group * n_q && ok; ++t) {
            const int s = t % C::kStages;
            if (t >= C::kStages)
                ok = mbar_wait(&v.empty[s], ((t / C::kStages) & 1) ^ 1, ctl, kSiteEmpty);
            if (!ok) break;
            const int g = t / n_q;
            const int q0 = (i0 + t - g * n_q) * kBlk;
            const int bq = q_head(p, bh, g);
            const size_t prow = static_cast<size_t>(bq) * p.n_blocks * kBlk;
            float *lse2 = v.rows + s * 2 * kBlk, *dd = lse2 + kBlk;
            uint8_t *st = v.ring + s * 2 * C::kTile;
            if (!dbg_ok(bq >= 0 && bq < p.BH && q0 >= 0 && q0 < p.n_blocks * kBlk &&
                            prow + q0 + kBlk <= static_cast<size_t>(p.BH) * p.n_blocks * kBlk,
                        ctl, kChkTmaQ) ||
                !dbg_ok(in_smem(st, 2 * C::kTile, C::kSmemBytes) &&
                            in_smem(lse2, 2 * kBlk * 4, C::kSmemBytes),
                        ctl, kChkSmem)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(&v.full[s], 2 * C::kTile + 2 * kBlk * 4);
            load_tile<D>(st, tmQ, &v.full[s], q0, bq, pol);
            load_tile<D>(st + C::kTile, tmdO, &v.full[s], q0, bq, pol);
            bulk_load(lse2, p.lse2 + prow + q0, kBlk * 4, &v.full[s], pol);
            bulk_load(dd, p.dd + prow + q0, kBlk * 4, &v.full[s], pol);
            ++issued;
        }
        // drain the loads in flight
        mbar_wait_drain(v.once, 0, p.limit_ns);
        for (int t = max(0, issued - C::kStages); t < issued; ++t)
            mbar_wait_drain(&v.full[t % C::kStages], (t / C::kStages) & 1, p.limit_ns);
    }
    __syncwarp();
}

// Each 128-query block i is taken in two 64-query halves u = 2t + h, and
// the halves alternate between two TMEM buffers (buffer h): S^T at
// [64h, 64h + 64), dP^T at [128 + 64h, 192 + 64h).  The tensor pipe computes
// S^T and dP^T of half u + 1 while the elementwise warps turn half u into
// P^T and dS^T, then runs dV / dK of half u, so neither side waits for the
// other's whole block.
// Two issuing warps: warp 8 issues S^T / dP^T of each half, warp 10 the dV
// / dK of each half once its P^T / dS^T are in TMEM.  S^T / dP^T(u) go into
// buffer u & 1 after dV / dK(u - 2), which read that buffer, have completed
// (buf_free, committed by warp 10; the dkdv kernel uses the dq kernel's V
// ring barriers vfull[2] for it).  Warp 10's commit after the second half's
// dV / dK releases the block's stage: that dV / dK followed the half's
// p_full, so the S^T / dP^T that read the stage had completed too.
template <int D, bool CAUSAL>
__device__ __forceinline__ void dkdv_issue_sdp(const Params &p) {
    using C = Cfg<D>;
    const View<D> v = view<D>();
    int bh, jb;  // jb: key block
    block_of<CAUSAL, true>(p, bh, jb);
    const int i0 = CAUSAL ? jb : 0;
    const int n_u = 2 * p.group * (p.n_blocks - i0);  // 64-query halves
    const uint32_t tmem = *v.tmem_slot;
    const WaitCtl ctl{v.abort_flag, &g_fa_status_bwd, p.limit_ns};
    (void)bh;
    const uint64_t dK = sdesc_sw128(smem_u32(v.a), 16, 1024);
    const uint64_t dV = sdesc_sw128(smem_u32(v.b), 16, 1024);
    const uint64_t ring_k = sdesc_sw128(smem_u32(v.ring), 16, 1024);
    const auto wait = [&](uint64_t *bar, uint32_t par, int site) {
        return __all_sync(0xffffffffu, mbar_wait(bar, par, ctl, site));
    };
    const uint64_t to = static_cast<uint64_t>(C::kTile >> 4);
    const uint64_t ho = static_cast<uint64_t>((64 * 128) >> 4);
    uint64_t *buf_free = v.vfull;
    bool ok = dbg_ok(whole_tmem(tmem), ctl, kChkTmem) && wait(v.once, 0, kSiteKV);
    for (int u = 0; u < n_u && ok; ++u) {
        const int t = u >> 1;
        if ((u & 1) == 0) {
            ok = wait(&v.full[t % C::kStages], (t / C::kStages) & 1, kSiteQ);
            if (!ok) break;
        }
        if (u >= 2) {
            ok = wait(&buf_free[u & 1], ((u - 2) >> 1) & 1, kSiteP);
            if (!ok) break;
        }
        tc_fence_after();
        const uint64_t so =
            static_cast<uint64_t>(((t % C::kStages) * 2 * C::kTile) >> 4) + (u & 1) * ho;
        mma_rows_half<D>(tmem + C::kTmS + (u & 1) * 64, dK, ring_k + so);
        mma_rows_half<D>(tmem + C::kTmP + (u & 1) * 64, dV, ring_k + so + to);
        mma_commit_elect(&v.s_full[u & 1]);
    }
    // every MMA of this warp had completed before the other issuer's last
    // dV / dK (it followed the last p_full); wait for that one
    mbar_wait_drain(v.o_full, 0, p.limit_ns);
}

template <int D, bool CAUSAL>
__device__ __forceinline__ void dkdv_issue_acc(const Params &p) {
    using C = Cfg<D>;
    const View<D> v = view<D>();
    int bh, jb;  // jb: key block
    block_of<CAUSAL, true>(p, bh, jb);
    const int i0 = CAUSAL ? jb : 0;
    const int n_u = 2 * p.group * (p.n_blocks - i0);
    const uint32_t tmem = *v.tmem_slot;
    const WaitCtl ctl{v.abort_flag, &g_fa_status_bwd, p.limit_ns};
    (void)bh;
    const uint64_t ring_mn = sdesc_sw128(smem_u32(v.ring), kBoxBytes, 1024);
    const auto wait = [&](uint64_t *bar, uint32_t par, int site) {
        return __all_sync(0xffffffffu, mbar_wait(bar, par, ctl, site));
    };
    const uint64_t to = static_cast<uint64_t>(C::kTile >> 4);
    const uint64_t ho = static_cast<uint64_t>((64 * 128) >> 4);
    uint64_t *buf_free = v.vfull;
    bool ok = dbg_ok(whole_tmem(tmem), ctl, kChkTmem);
    for (int u = 0; u < n_u && ok; ++u) {
        ok = wait(&v.p_full[u & 1], (u >> 1) & 1, kSiteP);
        if (!ok) break;
        tc_fence_after();
        const int t = u >> 1;
        const uint64_t so =
            static_cast<uint64_t>(((t % C::kStages) * 2 * C::kTile) >> 4) + (u & 1) * ho;
        const uint32_t a = tmem + C::kTmS + (u & 1) * 64;
        mma_tmem_half<D>(tmem + C::kTmAcc0, a, ring_mn + so + to, u > 0);  // dV += P^T dO_h
        mma_tmem_half<D>(tmem + C::kTmAcc1, a + 16, ring_mn + so, u > 0);  // dK += dS^T Q_h
        mma_commit_elect(&buf_free[u & 1]);
        if (u & 1) mma_commit_elect(&v.empty[t % C::kStages]);
    }
    mma_commit_elect(v.o_full);
    mbar_wait_drain(v.o_full, 0, p.limit_ns);
}

template <int D, bool CAUSAL>
__device__ __forceinline__ void dkdv_elementwise(const Params &p, int warp, int lane) {
    using C = Cfg<D>;
    const View<D> v = view<D>();
    int bh, jb;  // bh: K/V head; jb: key block
    block_of<CAUSAL, true>(p, bh, jb);
    const int N = p.N;
    const int i0 = CAUSAL ? jb : 0;  // first query block touching this key block
    const int n_q = p.n_blocks - i0;  // query blocks per query head of the group
    const int n_u = 2 * p.group * n_q;
    const uint32_t tmem = *v.tmem_slot;
    const WaitCtl ctl{v.abort_flag, &g_fa_status_bwd, p.limit_ns};
    // ---- elementwise: thread = key row of this block (TMEM lane); warp
    // column half c = queries [32c, 32c + 32) of each 64-query half
    const int quarter = warp & 3, c = warp >> 2;
    const int row = quarter * 32 + lane;
    const int key = jb * kBlk + row;
    const uint32_t lb = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = dbg_ok(whole_tmem(tmem), ctl, kChkTmem);
    for (int u = 0; u < n_u && ok; ++u) {
        const int t = u >> 1, h = u & 1, s = t % C::kStages;
        // the stage's LSE2/D rows landed with its tiles (the stage cannot
        // be refilled before this block's last dV / dK); this warp's 32
        // columns of them go to registers before S^T / dP^T are waited for
        ok = __all_sync(0xffffffffu, mbar_wait(&v.full[s], (t / C::kStages) & 1, ctl, kSiteQ));
        if (!ok) break;
        const int qi = t % n_q;  // query block within the current query head
        const int q0 = (i0 + qi) * kBlk;
        const int cb = 64 * h + 32 * c;  // this warp's first column within the block
        const float *lse2 = v.rows + s * 2 * kBlk + cb, *dd = lse2 + kBlk;
        float4 l4[8], d4[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            l4[e] = reinterpret_cast<const float4 *>(lse2)[e];
            d4[e] = reinterpret_cast<const float4 *>(dd)[e];
        }
        ok = __all_sync(0xffffffffu, mbar_wait(&v.s_full[h], (u >> 1) & 1, ctl, kSiteS));
        if (!ok) break;
        tc_fence_after();
        // column (query) q kept iff q < N and, causal, q >= key
        const int lim_lo = CAUSAL ? key - q0 : 0;
        const int lim_hi = N - q0;
        uint32_t sv[32], dv[32], pp[16], pds[16];
        const uint32_t ts = tmem + lb + C::kTmS + 64 * h + 32 * c;
        const uint32_t tp = tmem + lb + C::kTmP + 64 * h + 32 * c;
        tmem_ld32x2(ts, tp, sv, dv);
        // masked only on the diagonal block (causal) and a ragged last block
        const bool masked = (CAUSAL && qi == 0) || q0 + kBlk > N;
        if (masked)
            p_ds_masked(sv, dv, lse2, dd, true, 0.f, 0.f, p.scale_log2, lim_lo, lim_hi, cb, pp,
                        pds);
        else
            p_ds_fast_reg(sv, dv, l4, d4, p.scale_log2, pp, pds);
        // P^T over the first 16 of this warp's 32 S^T columns, dS^T over the
        // next 16
        tmem_st16(ts, pp);
        tmem_st16(ts + 16, pds);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&v.p_full[h]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(v.o_full, 0, ctl, kSiteO));
    if (ok) {
        tc_fence_after();
        const bool in = key < N;
        const bool row_ok =
            static_cast<size_t>(bh) * N + key < static_cast<size_t>(p.grid_heads) * N;
        __nv_bfloat16 *dvp = p.g1 + (static_cast<size_t>(bh) * N + key) * D;
        __nv_bfloat16 *dkp = p.g0 + (static_cast<size_t>(bh) * N + key) * D;
#pragma unroll 1
        for (int g = c * (D / 64); g < (c + 1) * (D / 64); ++g) {  // half the columns
            uint32_t a[32], b[32], pa[16], pb[16];
            tmem_ld32(tmem + lb + C::kTmAcc0 + 32 * g, a);
            tmem_ld32(tmem + lb + C::kTmAcc1 + 32 * g, b);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                pa[e] = pack_bf16x2(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
                pb[e] = pack_bf16x2(__uint_as_float(b[2 * e]) * p.scale,
                                    __uint_as_float(b[2 * e + 1]) * p.scale);
            }
            if (in && dbg_ok(row_ok && ((reinterpret_cast<uintptr_t>(dvp + 32 * g) |
                                         reinterpret_cast<uintptr_t>(dkp + 32 * g)) & 15u) == 0,
                             ctl, kChkStoreO)) {
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

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                const Params p) {
    using C = Cfg<D>;
    const View<D> v = view<D>();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) setup_barriers(v.once, v.full, v.empty, v.vfull, v.vempty, v.s_full, v.p_full,
                                         v.o_full, v.dp_free,
                                         v.abort_flag);
    if (warp == kMmaWarp) {
        tmem_alloc(v.tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // Each role runs inside the branch that set its register budget and
    // rebuilds what it needs, so little stays live across the switch.
    if (warp >= kMmaWarp) {
        regs_decrease<kRegsCtl>();  // warp 11: no role
        if (warp == kTmaWarp)
            dkdv_producer<D, CAUSAL>(&tmQ, &tmK, &tmV, &tmdO, p, lane);
        else if (warp == kMmaWarp)
            dkdv_issue_sdp<D, CAUSAL>(p);
        else if (warp == kMmaWarp + 2)
            dkdv_issue_acc<D, CAUSAL>(p);
        __syncwarp();
    } else {
        regs_increase<kRegsEw>();
        dkdv_elementwise<D, CAUSAL>(p, warp, lane);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(*view<D>().tmem_slot, kTmemCols);
    }
}

// ================================= dQ kernel =================================
template <int D, bool CAUSAL>
__device__ __forceinline__ void dq_producer(const CUtensorMap *tmQ, const CUtensorMap *tmK,
                                            const CUtensorMap *tmV, const CUtensorMap *tmdO,
                                            const Params &p, int lane) {
    using C = Cfg<D>;
    const View<D> v = view<D>();
    int bh, ib;  // ib: query block
    block_of<CAUSAL, false>(p, bh, ib);
    const int N = p.N;
    const int n_k = CAUSAL ? ib + 1 : p.n_blocks;  // key blocks at or below the diagonal
    const uint32_t tmem = *v.tmem_slot;
    const WaitCtl ctl{v.abort_flag, &g_fa_status_bwd, p.limit_ns};
    (void)N, (void)tmem, (void)bh;
    const int bk = kv_head(p, bh);  // this query head's K/V head
    if (lane == 0 &&
        dbg_ok(bh >= 0 && bh < p.grid_heads && ib >= 0 && ib < p.n_blocks &&
                   in_smem(v.a, 2 * C::kTile, C::kSmemBytes),
               ctl, kChkItem)) {
        const uint64_t pol_q = l2_policy_evict_first(), pol_kv = l2_policy_evict_last();
        mbar_arrive_expect_tx(v.once, 2 * C::kTile);
        load_tile<D>(v.a, tmQ, v.once, ib * kBlk, bh, pol_q);
        load_tile<D>(v.b, tmdO, v.once, ib * kBlk, bh, pol_q);
        int nk = 0, nv = 0;  // K and V tiles issued
        bool ok = true;
        for (int t = 0; t < n_k && ok; ++t) {
            const int sk = t % C::kStagesK, sv = t % C::kStagesV;
            if (t >= C::kStagesK)
                ok = mbar_wait(&v.empty[sk], ((t / C::kStagesK) & 1) ^ 1, ctl, kSiteEmpty);
            if (!ok) break;
            if (!dbg_ok(t * kBlk < p.n_blocks * kBlk && bk >= 0 && bk < p.BH / p.group, ctl,
                        kChkTmaKV) ||
                !dbg_ok(in_smem(v.ring + sk * C::kTile, C::kTile, C::kSmemBytes) &&
                            in_smem(v.vring + sv * C::kTile, C::kTile, C::kSmemBytes),
                        ctl, kChkSmem)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(&v.full[sk], C::kTile);
            load_tile<D>(v.ring + sk * C::kTile, tmK, &v.full[sk], t * kBlk, bk, pol_kv);
            ++nk;
            if (t >= C::kStagesV)
                ok = mbar_wait(&v.vempty[sv], ((t / C::kStagesV) & 1) ^ 1, ctl, kSiteEmpty);
            if (!ok) break;
            mbar_arrive_expect_tx(&v.vfull[sv], C::kTile);
            load_tile<D>(v.vring + sv * C::kTile, tmV, &v.vfull[sv], t * kBlk, bk, pol_kv);
            ++nv;
        }
        mbar_wait_drain(v.once, 0, p.limit_ns);
        for (int t = max(0, nk - C::kStagesK); t < nk; ++t)
            mbar_wait_drain(&v.full[t % C::kStagesK], (t / C::kStagesK) & 1, p.limit_ns);
        for (int t = max(0, nv - C::kStagesV); t < nv; ++t)
            mbar_wait_drain(&v.vfull[t % C::kStagesV], (t / C::kStagesV) & 1, p.limit_ns);
    }
    __syncwarp();
}

template <int D, bool CAUSAL>
__device__ __forceinline__ void dq_mma(const Params &p) {
    using C = Cfg<D>;
    const View<D> v = view<D>();
    int bh, ib;  // ib: query block
    block_of<CAUSAL, false>(p, bh, ib);
    const int N = p.N;
    const int n_k = CAUSAL ? ib + 1 : p.n_blocks;  // key blocks at or below the diagonal
    const uint32_t tmem = *v.tmem_slot;
    const WaitCtl ctl{v.abort_flag, &g_fa_status_bwd, p.limit_ns};
    (void)N, (void)tmem, (void)bh;
    const uint64_t dQ = sdesc_sw128(smem_u32(v.a), 16, 1024);
    const uint64_t ddO = sdesc_sw128(smem_u32(v.b), 16, 1024);
    const uint64_t kring = sdesc_sw128(smem_u32(v.ring), 16, 1024);          // K, K-major
    const uint64_t kring_mn = sdesc_sw128(smem_u32(v.ring), kBoxBytes, 1024);  // K, MN-major
    const uint64_t vring = sdesc_sw128(smem_u32(v.vring), 16, 1024);         // V, K-major
    const auto kofs = [](int t) {
        return static_cast<uint64_t>(((t % C::kStagesK) * C::kTile) >> 4);
    };
    const auto vofs = [](int t) {
        return static_cast<uint64_t>(((t % C::kStagesV) * C::kTile) >> 4);
    };
    const auto wait = [&](uint64_t *bar, uint32_t par, int site) {
        return __all_sync(0xffffffffu, mbar_wait(bar, par, ctl, site));
    };
    // S(t) goes to buffer t % 2, so S(t+1) and dP(t+1) run on the tensor
    // pipe while the elementwise warps work on block t: S(t+1) as soon as
    // K(t+1) is in (its buffer held dS(t-1), read by dQ(t-1) issued before),
    // dP(t+1) once the warps have read dP(t) (dp_free).
    bool ok = dbg_ok(whole_tmem(tmem), ctl, kChkTmem) && wait(v.once, 0, kSiteKV);
    if (ok) ok = wait(&v.full[0], 0, kSiteQ);
    if (ok) ok = wait(&v.vfull[0], 0, kSiteQ);
    if (ok) {
        tc_fence_after();
        mma_rows_rows<D>(tmem + kTmSq, dQ, kring);   // S(0) = Q K_0^T
        mma_rows_rows<D>(tmem + kTmPq, ddO, vring);  // dP(0) = dO V_0^T
        mma_commit_elect(&v.vempty[0]);              // V_0 read
        mma_commit_elect(&v.s_full[0]);
    }
    for (int t = 0; t < n_k && ok; ++t) {
        const int t1 = t + 1;
        const bool more = t1 < n_k;
        if (more) {
            ok = wait(&v.full[t1 % C::kStagesK], (t1 / C::kStagesK) & 1, kSiteQ);
            if (!ok) break;
            tc_fence_after();
            mma_rows_rows<D>(tmem + kTmSq + (t1 & 1) * kBlk, dQ, kring + kofs(t1));  // S(t+1)
        }
        ok = wait(v.dp_free, t & 1, kSiteP);
        if (ok && more) ok = wait(&v.vfull[t1 % C::kStagesV], (t1 / C::kStagesV) & 1, kSiteQ);
        if (!ok) break;
        tc_fence_after();
        if (more) {
            mma_rows_rows<D>(tmem + kTmPq, ddO, vring + vofs(t1));  // dP(t+1)
            mma_commit_elect(&v.vempty[t1 % C::kStagesV]);          // V(t+1) read
            mma_commit_elect(&v.s_full[t1 & 1]);
        }
        ok = wait(v.p_full, t & 1, kSiteP);
        if (!ok) break;
        tc_fence_after();
        mma_tmem_rows<D>(tmem + kTmAccq, tmem + kTmSq + (t & 1) * kBlk, kring_mn + kofs(t),
                         t > 0);  // dQ += dS(t) K(t)
        mma_commit_elect(&v.empty[t % C::kStagesK]);  // K(t) read by S(t) and dQ(t)
    }
    mma_commit_elect(v.o_full);
    mbar_wait_drain(v.o_full, 0, p.limit_ns);
}

template <int D, bool CAUSAL>
__device__ __forceinline__ void dq_elementwise(const Params &p, int warp, int lane) {
    using C = Cfg<D>;
    const View<D> v = view<D>();
    int bh, ib;  // ib: query block
    block_of<CAUSAL, false>(p, bh, ib);
    const int N = p.N;
    const int n_k = CAUSAL ? ib + 1 : p.n_blocks;  // key blocks at or below the diagonal
    const uint32_t tmem = *v.tmem_slot;
    const WaitCtl ctl{v.abort_flag, &g_fa_status_bwd, p.limit_ns};
    (void)N, (void)tmem, (void)bh;
    const int quarter = warp & 3, half = warp >> 2;  // half h: keys [64h, 64h + 64)
    const int row = quarter * 32 + lane;
    const int q = ib * kBlk + row;
    const uint32_t lb = static_cast<uint32_t>(quarter * 32) << 16;
    const int cb = half * 64;
    const bool qin = q < N;
    const size_t prow = static_cast<size_t>(bh) * p.n_blocks * kBlk + q;  // padded row
    const float my_nl2 = p.lse2[prow];  // -LSE log2 e (zero past N)
    const float my_nd = p.dd[prow];     // -D
    bool ok = dbg_ok(whole_tmem(tmem), ctl, kChkTmem);
    for (int t = 0; t < n_k && ok; ++t) {
        ok = __all_sync(0xffffffffu, mbar_wait(&v.s_full[t & 1], (t >> 1) & 1, ctl, kSiteS));
        if (!ok) break;
        tc_fence_after();
        const int k0 = t * kBlk;
        // key k kept iff k < N and, causal, k <= q
        const int lim_hi = CAUSAL ? min(N - k0, q - k0 + 1) : N - k0;
        uint32_t s0[32], s1[32], d0[32], d1[32], pp[16], pds[16];
        const uint32_t ts = tmem + lb + kTmSq + (t & 1) * kBlk + cb, tp = tmem + lb + kTmPq + cb;
        tmem_ld32x4(ts, ts + 32, tp, tp + 32, s0, s1, d0, d1);
        // dP(t) is in registers: the MMA warp may compute dP(t+1) over it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(v.dp_free);
        // masked only on the diagonal block (causal) and a ragged last block
        const bool masked = (CAUSAL && t == ib) || k0 + kBlk > N;
        if (masked)
            p_ds_masked(s0, d0, nullptr, nullptr, false, my_nl2, my_nd, p.scale_log2, 0,
                        lim_hi, cb, pp, pds);
        else
            p_ds_fast(s0, d0, nullptr, nullptr, false, my_nl2, my_nd, p.scale_log2, pp, pds);
        tmem_st16(ts, pds);
        if (masked)
            p_ds_masked(s1, d1, nullptr, nullptr, false, my_nl2, my_nd, p.scale_log2, 0,
                        lim_hi, cb + 32, pp, pds);
        else
            p_ds_fast(s1, d1, nullptr, nullptr, false, my_nl2, my_nd, p.scale_log2, pp, pds);
        tmem_st16(ts + 16, pds);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(v.p_full);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(v.o_full, 0, ctl, kSiteO));
    if (ok) {
        tc_fence_after();
        __nv_bfloat16 *dq = p.g0 + (static_cast<size_t>(bh) * N + q) * D;
#pragma unroll 1
        for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {  // half the columns
            uint32_t a[32], pa[16];
            tmem_ld32(tmem + lb + kTmAccq + 32 * c, a);
#pragma unroll
            for (int t = 0; t < 16; ++t)
                pa[t] = pack_bf16x2(__uint_as_float(a[2 * t]) * p.scale,
                                    __uint_as_float(a[2 * t + 1]) * p.scale);
            if (qin && dbg_ok(static_cast<size_t>(bh) * N + q < static_cast<size_t>(p.BH) * N &&
                                  (reinterpret_cast<uintptr_t>(dq + 32 * c) & 15u) == 0,
                              ctl, kChkStoreO)) {
                uint4 *o = reinterpret_cast<uint4 *>(dq + 32 * c);
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    o[t] = make_uint4(pa[4 * t], pa[4 * t + 1], pa[4 * t + 2], pa[4 * t + 3]);
            }
        }
    }
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
              const Params p) {
    using C = Cfg<D>;
    const View<D> v = view<D>();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) setup_barriers(v.once, v.full, v.empty, v.vfull, v.vempty, v.s_full, v.p_full,
                                         v.o_full, v.dp_free,
                                         v.abort_flag);
    if (warp == kMmaWarp) {
        tmem_alloc(v.tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // Each role runs inside the branch that set its register budget and
    // rebuilds what it needs, so little stays live across the switch.
    if (warp >= kMmaWarp) {
        regs_decrease<kRegsCtl>();  // warps 10, 11: no role
        if (warp == kTmaWarp)
            dq_producer<D, CAUSAL>(&tmQ, &tmK, &tmV, &tmdO, p, lane);
        else if (warp == kMmaWarp)
            dq_mma<D, CAUSAL>(p);
        __syncwarp();
    } else {
        regs_increase<kRegsEw>();
        dq_elementwise<D, CAUSAL>(p, warp, lane);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(*view<D>().tmem_slot, kTmemCols);
    }
}

// Per query row, into rows padded to Npad (a multiple of 128) per head, so
// that the other kernels fetch a block's rows with aligned bulk copies:
// -D = -rowsum(dO * O) (fp32) and -LSE * log2(e); zeros for rows past N.
// D/8 lanes per row, one 16-byte load of O and of dO each (32 / (D/8) rows
// per warp).
template <int D>
__global__ void pre_kernel(const __nv_bfloat16 *__restrict__ O,
                           const __nv_bfloat16 *__restrict__ dO, const float *__restrict__ LSE,
                           float *__restrict__ lse2, float *__restrict__ dd, int N, int Npad,
                           long long rows_pad) {
    constexpr int LPR = D / 8;        // lanes per row
    constexpr int RPW = 32 / LPR;     // rows per warp
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR, c = lane % LPR;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    for (long long wr = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         wr * RPW < rows_pad; wr += warps) {
        const long long prow = wr * RPW + sub;  // rows_pad is a multiple of 128: in range
        const long long bh = prow / Npad;
        const int q = static_cast<int>(prow - bh * Npad);
        float acc = 0.f;
        if (q < N) {
            const long long row = bh * N + q;
            const uint4 o4 = *reinterpret_cast<const uint4 *>(O + row * D + c * 8);
            const uint4 g4 = *reinterpret_cast<const uint4 *>(dO + row * D + c * 8);
            const uint32_t ow[4] = {o4.x, o4.y, o4.z, o4.w}, gw[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc = fmaf(__uint_as_float(ow[e] << 16), __uint_as_float(gw[e] << 16), acc);
                acc = fmaf(__uint_as_float(ow[e] & 0xFFFF0000u),
                           __uint_as_float(gw[e] & 0xFFFF0000u), acc);
            }
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (c == 0 && dbg_ok_word(prow < rows_pad && bh * Npad + q == prow, &g_fa_status_bwd,
                                  kChkStoreLse)) {
            dd[prow] = -acc;
            lse2[prow] = q < N ? -LSE[bh * N + q] * kLog2e : 0.f;
        }
    }
}

}  // namespace bwd

template <int D, bool CAUSAL>
static int launch_bwd_t(const BwdArgs &a) {
    using C = bwd::Cfg<D>;
    static std::atomic<int> configured1[kMaxDevices], configured2[kMaxDevices];
    int dev = 0;
    FA_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_ARCH;
    auto k1 = bwd::dkdv_kernel<D, CAUSAL>;
    auto k2 = bwd::dq_kernel<D, CAUSAL>;
    int rc = set_smem_once(configured1, dev, k1, C::kSmemBytes);
    if (rc == FA_OK) rc = set_smem_once(configured2, dev, k2, C::kSmemBytes);
    if (rc != FA_OK) return rc;
    const int n_blocks = (a.N + bwd::kBlk - 1) / bwd::kBlk;
    const int Npad = n_blocks * bwd::kBlk;
    const long long rows_pad = static_cast<long long>(a.BH) * Npad;
    float *lse2 = a.rows, *dd = a.rows + rows_pad;
    const long long pre_blocks = (rows_pad / (32 / (D / 8)) + 3) / 4;  // 4 warps per block
    bwd::pre_kernel<D><<<static_cast<unsigned>(pre_blocks < (1 << 20) ? pre_blocks : (1 << 20)),
                         128, 0, a.stream>>>(
        static_cast<const __nv_bfloat16 *>(a.O), static_cast<const __nv_bfloat16 *>(a.dO),
        a.LSE, lse2, dd, a.N, Npad, rows_pad);
    FA_CUDA_TRY(cudaGetLastError());
    bwd::Params p;
    p.lse2 = lse2;
    p.dd = dd;
    p.N = a.N;
    p.BH = a.BH;
    p.H = a.H;
    p.group = a.H / a.Hkv;
    p.n_blocks = n_blocks;
    p.scale = a.scale;
    p.scale_log2 = a.scale * bwd::kLog2e;
    p.limit_ns = a.limit_ns;
    // Causal CTA order: a group of heads holds enough work that its heaviest
    // CTAs (about 2 / (n_blocks + 1) of a head's work each) start well
    // before the end even when the group runs last: about 3 x SMs / (n_blocks
    // + 1) heads.
    const int sms = device_sm_count(dev);
    const long long hg = (3LL * (sms > 0 ? sms : 1) + n_blocks) / (n_blocks + 1);
    const auto set_heads = [&](long long heads) {
        p.grid_heads = static_cast<int>(heads);
        p.head_group = static_cast<int>(hg < 1 ? 1 : (hg > heads ? heads : hg));
        return static_cast<long long>(p.n_blocks) * heads;
    };
    const long long bh_kv = a.BH / p.group;
    if (static_cast<long long>(p.n_blocks) * a.BH > 0x7FFFFFFFLL) return FA_ERR_SHAPE;
    // dK / dV: one CTA per (K/V head, key block)
    const long long grid1 = set_heads(bh_kv);
    p.g0 = static_cast<__nv_bfloat16 *>(a.dK);
    p.g1 = static_cast<__nv_bfloat16 *>(a.dV);
    k1<<<static_cast<unsigned>(grid1), bwd::kThreads, C::kSmemBytes, a.stream>>>(
        *a.tmQ, *a.tmK, *a.tmV, *a.tmdO, p);
    FA_CUDA_TRY(cudaGetLastError());
    // dQ: one CTA per (query head, query block)
    const long long grid2 = set_heads(a.BH);
    p.g0 = static_cast<__nv_bfloat16 *>(a.dQ);
    p.g1 = nullptr;
    k2<<<static_cast<unsigned>(grid2), bwd::kThreads, C::kSmemBytes, a.stream>>>(
        *a.tmQ, *a.tmK, *a.tmV, *a.tmdO, p);
    FA_CUDA_TRY(cudaGetLastError());
    return FA_OK;
}

// d = 256: the pre-pass here, the dK/dV and dQ kernels in fa_bwd256_sm103.cu.
static int launch_bwd_256(const BwdArgs &a) {
    const int n_blocks = (a.N + bwd::kBlk - 1) / bwd::kBlk;
    const int Npad = n_blocks * bwd::kBlk;
    const long long rows_pad = static_cast<long long>(a.BH) * Npad;
    float *lse2 = a.rows, *dd = a.rows + rows_pad;
    const long long pre_blocks = (rows_pad + 3) / 4;  // one row per warp, 4 warps per block
    bwd::pre_kernel<256><<<static_cast<unsigned>(pre_blocks < (1 << 20) ? pre_blocks : (1 << 20)),
                           128, 0, a.stream>>>(
        static_cast<const __nv_bfloat16 *>(a.O), static_cast<const __nv_bfloat16 *>(a.dO),
        a.LSE, lse2, dd, a.N, Npad, rows_pad);
    FA_CUDA_TRY(cudaGetLastError());
    return launch_bwd256(a, lse2, dd, n_blocks);
}

int launch_bwd(const BwdArgs &a) {
    if (a.d == 64) return a.causal ? launch_bwd_t<64, true>(a) : launch_bwd_t<64, false>(a);
    if (a.d == 128) return a.causal ? launch_bwd_t<128, true>(a) : launch_bwd_t<128, false>(a);
    if (a.d == 256) return launch_bwd_256(a);
    return FA_ERR_HEADDIM;
}

int bwd_read_and_clear_status(int *status) {
    int v = 0;
    FA_CUDA_TRY(cudaMemcpyFromSymbol(&v, g_fa_status_bwd, sizeof v));
    if (v != 0) {
        const int zero = 0;
        FA_CUDA_TRY(cudaMemcpyToSymbol(g_fa_status_bwd, &zero, sizeof zero));
    }
    *status = v;
    return FA_OK;
}

}  // namespace fa
