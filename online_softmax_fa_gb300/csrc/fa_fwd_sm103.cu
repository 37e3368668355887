// fa_fwd_sm103.cu -- exact attention forward pass for sm_103a (GB300).
//
// Computes, per (batch b, head h) and query row i,
//   O_i   = sum_j softmax_j(scale * q_i . k_j  [j <= i if causal]) v_j
//   LSE_i = log sum_j exp(scale * q_i . k_j)
// with the online-softmax recurrence ("Understanding FlashAttention Pt 1",
// wpnews.pro, section 2.4): per row a running max m, a running sum l and an
// unnormalised accumulator a; a new key block with scores s rescales (l, a)
// by alpha = exp(m - m') when the max moves to m' and adds p = exp(s - m');
// o = a / l once at the end ("Fix 1" of "FlashAttention-2 -- Deeper Math",
// aicassindra.com) and L = m + log(l) is written beside it ("Fix 2").
//
// GB300 mapping.  A work item is one (b, h, 256-row query block): query
// blocks are the outer loop and own their output ("Fix 3"), and the grid
// covers batch x heads x query blocks ("Fix 4").  The grid has one CTA per
// work item, in priority order, but only one CTA fits on an SM and the CTAs
// that run steal the rest: before a CTA runs out of work it asks the
// hardware scheduler (cluster launch control) to cancel the launch of the
// next CTA of the grid and does that CTA's item itself.  So each SM keeps
// its CTA (and its warm pipeline) while the items are handed out greedily
// in grid order, which balances the causal costs ("the assignment of blocks
// to SMs must account for the imbalance").  Causal order: heads in groups
// (the partial group first), inside a group the heaviest query block first
// with the group's heads interleaved; a group's K/V stays in L2 while its
// items run, and every group holds enough heavy items that its last ones
// start early.  Consecutive items of a CTA overlap: the next item's query
// block loads and its first S tiles are computed while the softmax warps
// write the previous item's output.
//   * warp 9 (TMA and schedule): per item, the query block once, then
//     128-key K and V tiles through separate multi-stage shared-memory rings
//     that run on across items; a few tiles before an item's loads end it
//     claims the next item and passes it to the other warps through a
//     two-slot ring in shared memory.
//   * warp 8 (MMA): tcgen05 MMAs issued by one elected lane of a converged
//     warp.  The query block is two 128-row sub-tiles; S_k = Q_k K_j^T lands
//     in TMEM (fp32), and O_k += P_k V_j reads P_k from TMEM (bf16, written
//     over S_k) and V_j from shared memory, accumulating O_k in TMEM.  Issue
//     order S_0(j), PV_1(j-1), S_1(j), PV_0(j) keeps the tensor pipe busy
//     while the two softmax groups work on the other sub-tile.
//   * warps 0-3 / 4-7 (softmax, one group per sub-tile; thread = row):
//     TMEM -> registers, mask (diagonal / ragged tiles only), row max with
//     the scale folded into base-2 exponents, p = 2^(s*c - m), row sum in
//     fp32, P -> TMEM as bf16, and the rescale of O_k in TMEM only for
//     warps where some row's reference max moved.  After an item's last
//     tile: O = a / l in bf16 and LSE = (m + log2 l) ln 2.
//   * causal: key tiles entirely above the diagonal are never loaded or
//     computed; only diagonal tiles are masked ("Causal masking: skip the
//     blocks, do not mask them").
//
// TMEM columns (512 allocated): S_0 [0,128), S_1 [128,256),
// O_0 [256, 256+D), O_1 [256+D, 256+2D).  P_k occupies the first 64 columns
// of S_k (128 bf16 per row, two per column).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_internal.h"
#include "sm103_primitives.cuh"
#include "debug_checks.cuh"
#ifdef FA_DEBUG
#include <mutex>

#include "../../include/fa_debug.h"
#endif

namespace fa {

// Device status word read by fa_device_error(): 0 or the site of the first
// bounded wait that expired.
__device__ int g_fa_status;

constexpr int kBlockM = 256;  // query rows per work item (two 128-row sub-tiles)
constexpr int kSubM = 128;    // rows per sub-tile = TMEM lanes
constexpr int kBlockN = 128;  // keys per K/V tile
constexpr int kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 64 bf16
constexpr int kThreads = 384;         // 12 warps = 3 warpgroups
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;           // warps 10, 11: no role (warpgroup padding)
// Registers per thread after reallocation.  Launch: 384 threads x 168.
// Warpgroup 2 (MMA, TMA) gives back down to 72; the two softmax warpgroups
// take 216 each: 128 x (216 + 216 + 72) = 64512 = 384 x 168, and each SM
// sub-partition holds one warp of each: 32 x 504 <= 16384 registers.
constexpr uint32_t kRegsSoftmax = 216;
constexpr uint32_t kRegsControl = 72;
constexpr uint32_t kTmemCols = 512;
// The running reference max moves only when a row's max exceeds it by more
// than this many base-2 units (factor 256); probabilities then stay <= 256.
constexpr float kStaleMax = 8.0f;
// Causal: the next work item is claimed this many key tiles before the end
// of the current item's loads: late enough that the CTA is nearly free
// (greedy hand-out in grid order over items of unequal cost), early enough
// that the answer is back before the next query block is due.  Items of
// equal cost (no mask) are claimed as an item's loads begin.
constexpr int kClaimLead = 3;

// wait sites recorded in the status word on a timeout
enum : int {
    kSiteQ = 1, kSiteKFull, kSiteVFull, kSitePFull, kSiteKEmpty, kSiteVEmpty,
    kSiteSFull, kSiteOFull, kSiteQEmpty, kSiteOEmpty, kSiteSchedFull, kSiteSchedEmpty,
    kSiteClaim
};

template <int D>
struct Cfg {
    static constexpr int kChunks = D / 64;  // 64-column (128-byte) swizzle chunks
    static constexpr int kStages = (D == 128) ? 2 : 4;
    static constexpr int kQBytes = 2 * kChunks * kBoxBytes;
    static constexpr int kTileBytes = kChunks * kBoxBytes;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    static constexpr int kOffBar = kOffV + kStages * kTileBytes;
    // barriers: q_full, q_empty, k_full[S], k_empty[S], v_full[S],
    // v_empty[S], s_full[2], p_full[2], o_full[2], o_empty[2], mma_done,
    // sched_full[2], sched_empty[2], claim; then (16-byte aligned) the tmem
    // slot, the abort flag, the two item slots and the 16-byte claim answer
    static constexpr int kNumBars = 2 + 4 * kStages + 2 + 2 + 2 + 2 + 1 + 2 + 2 + 1;
    static constexpr int kOffMisc = (kOffBar + 8 * kNumBars + 15) / 16 * 16;
    static constexpr int kSmemBytes = kOffMisc + 32 + 1024;  // + alignment slack
    static constexpr uint32_t kTmS0 = 0, kTmS1 = 128, kTmO0 = 256, kTmO1 = 256 + D;
    static constexpr uint32_t kIdescS = idesc_bf16_f32(kSubM, kBlockN, false);
    static constexpr uint32_t kIdescPV = idesc_bf16_f32(kSubM, D, true);
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(256 + 2 * D <= (int)kTmemCols, "TMEM budget");
};

// S = Q_k K_j^T: D/16 MMAs of M128 x N128 x K16, both operands K-major in
// 64-column swizzled chunks; K-step kk sits in chunk kk/4 at byte 32*(kk%4).
// A descriptor's low bits hold (address >> 4), so byte offsets are added as
// (offset >> 4).
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tm, uint64_t dq, uint64_t dk) {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
        mma_ss_elect(d_tm, dq + off, dk + off, Cfg<D>::kIdescS, kk > 0 ? 1u : 0u);
    }
}

// O_k += P_k V_j: 8 MMAs of M128 x N(D) x K16; P_k from TMEM (16 keys = 8
// columns of packed bf16 pairs), V_j MN-major, 16 keys = 2048 bytes.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tm, uint32_t p_tm, uint64_t dv, bool acc) {
#pragma unroll
    for (int kk = 0; kk < kBlockN / 16; ++kk)
        mma_ts_elect(d_tm, p_tm + kk * 8, dv + static_cast<uint64_t>((kk * 16 * 128) >> 4),
                     Cfg<D>::kIdescPV, (acc || kk > 0) ? 1u : 0u);
}

struct Params {
    __nv_bfloat16 *O;
    float *LSE;
    int N;
    int BH;         // batch x query heads
    int H;          // query heads per batch
    int group;      // query heads per K/V head (grouped-query attention; 1 = MHA)
    int n_qblocks;  // ceil(N / 256)
    int n_ktiles;   // ceil(N / 128)
    int n_items;    // BH x n_qblocks = the grid
    int head_group;   // causal order: heads per group
    int first_group;  // heads in the first (partial) group
    float scale_log2;  // scale * log2(e)
    uint64_t limit_ns;
    int o_align32;     // O is 32-byte aligned: the epilogue stores 32 bytes at a time
    // debug build only: the extent (rows of O and LSE) the store checks
    // use, and an injected fault -- the producer of item lose_item skips the
    // load of key tile lose_tile and the arrival on its barrier (-1: none)
    long long o_rows;
    int lose_item, lose_tile;
};

// Shared-memory layout of one CTA (rebuilt where needed: it costs a few
// integer instructions and keeps nothing live across register reallocation).
template <int D>
struct SmemView {
    uint8_t *q, *k, *v;
    uint64_t *q_full, *q_empty, *k_full, *k_empty, *v_full, *v_empty;
    uint64_t *s_full, *p_full, *o_full, *o_empty, *mma_done;
    uint64_t *sched_full, *sched_empty, *claim;
    uint32_t *tmem_slot;
    volatile int *abort_flag;
    volatile int *sched_item;  // [2]: work item, or -1 = no more work
    void *claim_resp;          // 16 bytes, 16-byte aligned
};

template <int D>
__device__ __forceinline__ SmemView<D> smem_view() {
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    SmemView<D> v;
    v.q = smem + C::kOffQ;
    v.k = smem + C::kOffK;
    v.v = smem + C::kOffV;
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    v.q_full = b;
    v.q_empty = b + 1;
    v.k_full = b + 2;
    v.k_empty = v.k_full + C::kStages;
    v.v_full = v.k_empty + C::kStages;
    v.v_empty = v.v_full + C::kStages;
    v.s_full = v.v_empty + C::kStages;
    v.p_full = v.s_full + 2;
    v.o_full = v.p_full + 2;
    v.o_empty = v.o_full + 2;
    v.mma_done = v.o_empty + 2;
    v.sched_full = v.mma_done + 1;
    v.sched_empty = v.sched_full + 2;
    v.claim = v.sched_empty + 2;
    v.tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    v.abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    v.sched_item = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 8);
    v.claim_resp = smem + C::kOffMisc + 16;
    return v;
}

// Debug checks: a range inside this kernel's shared memory.
template <int D>
__device__ __forceinline__ bool in_smem_d(const void *ptr, int bytes) {
    return in_smem(ptr, bytes, Cfg<D>::kSmemBytes);
}

// ------------------------------------------------------------- schedule
// Work item x (the grid's CTA index, in priority order) -> (head, query
// block).  Causal: heads in groups of head_group, the partial group
// (first_group heads) first; inside a group the heaviest query block first
// (block qb needs 2*qb + 2 key tiles), the group's heads interleaved.
// Otherwise head-major (equal costs; consecutive items share K/V in L2).
struct Work {
    int bh, kvh, qb, n_sub0, n_sub1;  // kvh: K/V head row; n_sub1 >= n_sub0
};

template <bool CAUSAL>
__device__ __forceinline__ Work work_of(const Params &p, int x) {
    Work w;
    if (CAUSAL) {
        const int nq = p.n_qblocks;
        const int first = p.first_group * nq;  // items of the first group
        int h0, gs, in;
        if (x < first) {
            h0 = 0;
            gs = p.first_group;
            in = x;
        } else {
            const int y = x - first, per = p.head_group * nq;
            const int g = y / per;
            h0 = p.first_group + g * p.head_group;
            gs = p.head_group;
            in = y - g * per;
        }
        const int level = in / gs;
        w.qb = nq - 1 - level;
        w.bh = h0 + (in - level * gs);
    } else {
        w.bh = x / p.n_qblocks;
        w.qb = x - w.bh * p.n_qblocks;
    }
    // grouped-query attention: query head h of batch b reads K/V head
    // h / group of that batch (consecutive query heads share one K/V head,
    // and the order keeps them adjacent, so they share it in L2)
    const int b = w.bh / p.H, h = w.bh - b * p.H;
    w.kvh = b * (p.H / p.group) + h / p.group;
    const int T = p.n_ktiles, N = p.N;
    // key tiles each 128-row sub-tile needs (causal: up to its last row)
    w.n_sub0 = CAUSAL ? min(T, min(w.qb * kBlockM + kSubM - 1, N - 1) / kBlockN + 1) : T;
    w.n_sub1 = CAUSAL ? min(T, min(w.qb * kBlockM + 2 * kSubM - 1, N - 1) / kBlockN + 1) : T;
    return w;
}

// The r-th work item of this CTA as the producer published it (-1: no more
// work).  Called by every thread of a consumer warp; one lane then frees the
// slot.
template <int D>
__device__ __forceinline__ bool next_item(const SmemView<D> &v, const WaitCtl &ctl, int r,
                                          int lane, int n_items, int &x) {
    const int slot = r & 1;
    if (!__all_sync(0xffffffffu, mbar_wait(&v.sched_full[slot], (r >> 1) & 1, ctl,
                                           kSiteSchedFull)))
        return false;
    x = v.sched_item[slot];
    if (x >= 0 && !dbg_ok(x < n_items, ctl, kChkItem)) x = -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(&v.sched_empty[slot]);
    return true;
}

// ================================ TMA producer ================================
template <int D, bool CAUSAL>
__device__ __forceinline__ void role_producer(const CUtensorMap *tmQ, const CUtensorMap *tmK,
                                              const CUtensorMap *tmV, const Params &p,
                                              int lane) {
    using C = Cfg<D>;
    if (lane != 0) return;
    const SmemView<D> v = smem_view<D>();
    const WaitCtl ctl{v.abort_flag, &g_fa_status, p.limit_ns};
    int g = 0;       // K/V tiles issued so far, across items
    int items = 0;   // query blocks issued so far
    // claims: 2 x (claims answered so far) + (1 if one is on its way); -1
    // once a claim has failed (no further claim may be made)
    int claims = 0;
    bool ok = true;
    int x = static_cast<int>(blockIdx.x);  // this CTA's own item first
    for (int r = 0;; ++r) {
        // publish item x (or the end of the work) to the MMA and softmax
        // warps; slot r & 1 last held item r - 2
        const int slot = r & 1;
        if (r >= 2) {
            ok = mbar_wait(&v.sched_empty[slot], ((r >> 1) & 1) ^ 1, ctl, kSiteSchedEmpty);
            if (!ok) break;
        }
        if (x >= 0 && !dbg_ok(x < p.n_items, ctl, kChkItem)) x = -1;  // end the work
        v.sched_item[slot] = x;
        mbar_arrive(&v.sched_full[slot]);
        if (x < 0) break;
        const Work w = work_of<CAUSAL>(p, x);
        if (r > 0) {  // the previous item's last S MMA has read Q
            ok = mbar_wait(v.q_empty, (r - 1) & 1, ctl, kSiteQEmpty);
            if (!ok) break;
        }
        if (!dbg_ok(w.bh >= 0 && w.bh < p.BH && w.qb >= 0 && w.qb < p.n_qblocks, ctl,
                    kChkTmaQ) ||
            !dbg_ok(in_smem_d<D>(v.q, C::kQBytes), ctl, kChkSmem)) {
            ok = false;
            break;
        }
        mbar_arrive_expect_tx(v.q_full, C::kQBytes);
        {
            const uint64_t pol_q = l2_policy_evict_first();
            for (int k = 0; k < 2; ++k)
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(v.q + (k * C::kChunks + c) * kBoxBytes, tmQ, v.q_full, 64 * c,
                                w.qb * kBlockM + k * kSubM, w.bh, pol_q);
        }
        ++items;
        const int claim_at = CAUSAL ? max(0, w.n_sub1 - kClaimLead) : 0;
        for (int j = 0; j < w.n_sub1; ++j) {
            if (j == claim_at && claims >= 0) {  // ask for the next item
                mbar_arrive_expect_tx(v.claim, 16);
                clc_try_cancel(v.claim_resp, v.claim);
                claims |= 1;
            }
            const uint64_t pol_kv = l2_policy_evict_last();
            const int t = g + j, s = t % C::kStages;
            const uint32_t ph = (t / C::kStages) & 1;
            if (t >= C::kStages) ok = mbar_wait(&v.k_empty[s], ph ^ 1, ctl, kSiteKEmpty);
            if (!ok) {
                g = t;
                break;
            }
            if (!dbg_ok(j * kBlockN < p.N && w.kvh >= 0 && w.kvh < p.BH / p.group, ctl,
                        kChkTmaKV) ||
                !dbg_ok(in_smem_d<D>(v.k + s * C::kTileBytes, C::kTileBytes) &&
                            in_smem_d<D>(v.v + s * C::kTileBytes, C::kTileBytes),
                        ctl, kChkSmem)) {
                ok = false;
                g = t;
                break;
            }
            // debug build: an injected fault loses this tile's K load and
            // its arrival (the consumers' waits then run out)
            if (!(kDebug && x == p.lose_item && j == p.lose_tile)) {
                mbar_arrive_expect_tx(&v.k_full[s], C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(v.k + s * C::kTileBytes + c * kBoxBytes, tmK, &v.k_full[s],
                                64 * c, j * kBlockN, w.kvh, pol_kv);
            }
            if (t >= C::kStages) ok = mbar_wait(&v.v_empty[s], ph ^ 1, ctl, kSiteVEmpty);
            if (!ok) {  // K of tile t is in flight: count it for the drain
                g = t + 1;
                break;
            }
            mbar_arrive_expect_tx(&v.v_full[s], C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_3d(v.v + s * C::kTileBytes + c * kBoxBytes, tmV, &v.v_full[s], 64 * c,
                            j * kBlockN, w.kvh, pol_kv);
        }
        if (!ok) break;
        g += w.n_sub1;
        // the next item: the cancelled CTA's, if the claim succeeded; after
        // a failed claim none is made again
        x = -1;
        if (claims > 0 && (claims & 1)) {
            ok = mbar_wait(v.claim, (claims >> 1) & 1, ctl, kSiteClaim);
            if (!ok) break;
            claims += 1;  // answered: clear the pending bit, count it
            x = clc_cancelled_x(v.claim_resp);
            if (x < 0) claims = -1;
        }
    }
    // Drain: every asynchronous write into shared memory lands before the
    // CTA exits.  The last query block, the last load of each ring stage
    // (after an abort V may lag K by one tile; a wait on a phase that never
    // started times out after the limit, a wait on one that completed
    // returns at once), and a claim answer still on its way.
    if (items > 0) mbar_wait_drain(v.q_full, (items - 1) & 1, p.limit_ns);
    for (int t = max(0, g - C::kStages); t < g; ++t) {
        mbar_wait_drain(&v.k_full[t % C::kStages], (t / C::kStages) & 1, p.limit_ns);
        mbar_wait_drain(&v.v_full[t % C::kStages], (t / C::kStages) & 1, p.limit_ns);
    }
    if (claims > 0 && (claims & 1)) mbar_wait_drain(v.claim, (claims >> 1) & 1, p.limit_ns);
}

// ================================= MMA issuer =================================
// The whole warp runs this loop (converged, operands warp-uniform); elect.sync
// inside the issue helpers picks the issuing lane.  Every wait result is made
// warp-uniform (__all_sync), so the warp leaves the loops together and stays
// converged for elect.sync even when a wait gives up.
template <int D, bool CAUSAL>
__device__ __forceinline__ void role_mma(const Params &p) {
    using C = Cfg<D>;
    const SmemView<D> v = smem_view<D>();
    const WaitCtl ctl{v.abort_flag, &g_fa_status, p.limit_ns};
    const uint32_t tmem = *v.tmem_slot;
    const uint64_t dq0 = sdesc_sw128(smem_u32(v.q), 16, 1024);
    const uint64_t dq1 = dq0 + ((C::kChunks * kBoxBytes) >> 4);
    const uint64_t dk0 = sdesc_sw128(smem_u32(v.k), 16, 1024);
    const uint64_t dv0 = sdesc_sw128(smem_u32(v.v), kBoxBytes, 1024);
    const uint32_t tS0 = tmem + C::kTmS0, tS1 = tmem + C::kTmS1;
    const uint32_t tO0 = tmem + C::kTmO0, tO1 = tmem + C::kTmO1;
    const auto wait = [&](uint64_t *bar, uint32_t parity, int site) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl, site));
    };
    const int lane = static_cast<int>(threadIdx.x & 31);
    int g = 0;             // K/V tiles consumed, across items
    int pc0 = 0, pc1 = 0;  // P tiles consumed per sub-tile, across items
    bool ok = dbg_ok(whole_tmem(tmem), ctl, kChkTmem) &&
              dbg_ok(in_smem_d<D>(v.q, C::kQBytes) &&
                         in_smem_d<D>(v.k, C::kStages * C::kTileBytes) &&
                         in_smem_d<D>(v.v, C::kStages * C::kTileBytes),
                     ctl, kChkSmem);
    for (int r = 0; ok; ++r) {
        int x;
        ok = next_item(v, ctl, r, lane, p.n_items, x);
        if (!ok || x < 0) break;
        const Work w = work_of<CAUSAL>(p, x);
        const int n0 = w.n_sub0, n1 = w.n_sub1;
        ok = wait(v.q_full, r & 1, kSiteQ);
        if (!ok) break;
        tc_fence_after();
        for (int j = 0; j <= n1 && ok; ++j) {
            const int t = g + j, s = t % C::kStages;
            if (j < n1) {
                ok = wait(&v.k_full[s], (t / C::kStages) & 1, kSiteKFull);
                if (!ok) break;
                tc_fence_after();
            }
            const uint64_t dk = dk0 + static_cast<uint64_t>((s * C::kTileBytes) >> 4);
            // S_0(j)
            if (j < n0) {
                issue_qk<D>(tS0, dq0, dk);
                mma_commit_elect(&v.s_full[0]);
            }
            // PV_1(j-1)
            if (j >= 1) {
                const int jp = j - 1, tp = g + jp, sp = tp % C::kStages;
                if (jp >= n0) {  // V not yet waited for by PV_0
                    ok = wait(&v.v_full[sp], (tp / C::kStages) & 1, kSiteVFull);
                    if (!ok) break;
                }
                if (jp == 0 && r > 0) {  // O_1 read out by the previous item's epilogue
                    ok = wait(&v.o_empty[1], (r - 1) & 1, kSiteOEmpty);
                    if (!ok) break;
                }
                ok = wait(&v.p_full[1], pc1 & 1, kSitePFull);
                if (!ok) break;
                ++pc1;
                tc_fence_after();
                issue_pv<D>(tO1, tS1, dv0 + static_cast<uint64_t>((sp * C::kTileBytes) >> 4),
                            jp > 0);
                mma_commit_elect(&v.v_empty[sp]);
                if (jp == n1 - 1) mma_commit_elect(&v.o_full[1]);
            }
            if (j < n1) {
                // S_1(j)
                issue_qk<D>(tS1, dq1, dk);
                mma_commit_elect(&v.s_full[1]);
                if (j == n1 - 1) mma_commit_elect(v.q_empty);  // last read of Q
                mma_commit_elect(&v.k_empty[s]);
                // PV_0(j)
                if (j < n0) {
                    ok = wait(&v.v_full[s], (t / C::kStages) & 1, kSiteVFull);
                    if (!ok) break;
                    if (j == 0 && r > 0) {
                        ok = wait(&v.o_empty[0], (r - 1) & 1, kSiteOEmpty);
                        if (!ok) break;
                    }
                    ok = wait(&v.p_full[0], pc0 & 1, kSitePFull);
                    if (!ok) break;
                    ++pc0;
                    tc_fence_after();
                    issue_pv<D>(tO0, tS0, dv0 + static_cast<uint64_t>((s * C::kTileBytes) >> 4),
                                j > 0);
                    if (j == n0 - 1) mma_commit_elect(&v.o_full[0]);
                }
            }
        }
        g += n1;
    }
    // Every MMA issued completes before the CTA frees its tensor memory.
    mma_commit_elect(v.mma_done);
    mbar_wait_drain(v.mma_done, 0, p.limit_ns);
}

// ============================ softmax (sub-tile k) ============================
// p = 2^(s*c - m) for 32 consecutive scores: packed FMA, two MUFU ex2 per
// pair, row sum into four packed fp32 accumulators, P packed to bf16 pairs.
__device__ __forceinline__ void exp_chunk32(const float *sv, uint64_t cs2, uint64_t neg2,
                                            uint64_t (&rs2)[4], uint32_t (&pk)[16]) {
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(sv[2 * t], sv[2 * t + 1]), cs2, neg2), x0, x1);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        rs2[t & 3] = f2_add(rs2[t & 3], f2_pack(p0, p1));
        pk[t] = pack_bf16x2(p0, p1);
    }
}

__device__ __forceinline__ float sum_pairs(const uint64_t (&rs2)[4]) {
    float a, b, c, d;
    f2_unpack(f2_add(rs2[0], rs2[1]), a, b);
    f2_unpack(f2_add(rs2[2], rs2[3]), c, d);
    return (a + b) + (c + d);
}

template <int D, bool CAUSAL>
__device__ __forceinline__ void role_softmax(const Params &p, int warp, int lane) {
    using C = Cfg<D>;
    const SmemView<D> v = smem_view<D>();
    const WaitCtl ctl{v.abort_flag, &g_fa_status, p.limit_ns};
    const uint32_t tmem = *v.tmem_slot;
    const int N = p.N;
    const int k = warp >> 2;  // warps 0-3 -> sub-tile 0, 4-7 -> sub-tile 1
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    const int row = wq * 32 + lane;
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tm_s = tmem + lane_bits + (k ? C::kTmS1 : C::kTmS0);
    const uint32_t tm_o = tmem + lane_bits + (k ? C::kTmO1 : C::kTmO0);
    uint64_t *s_full = v.s_full + k, *p_ready = v.p_full + k;
    uint64_t *o_full = v.o_full + k, *o_empty = v.o_empty + k;
    const float cs = p.scale_log2;
    const uint64_t cs2 = f2_pack(cs, cs);

    int sc = 0;  // S tiles consumed, across items
    bool ok = dbg_ok(whole_tmem(tmem), ctl, kChkTmem);
    for (int r = 0; ok; ++r) {
        int x;
        ok = next_item(v, ctl, r, lane, p.n_items, x);
        if (!ok || x < 0) break;
        const Work w = work_of<CAUSAL>(p, x);
        const int sub_start = w.qb * kBlockM + k * kSubM;
        const int qrow = sub_start + row;
        const int n_k = k ? w.n_sub1 : w.n_sub0;

        // Per row: reference max m (of s * scale * log2 e) and running sum l
        // of 2^(s*c - m).  The reference moves only when a tile's row max
        // exceeds it by more than kStaleMax, so p <= 2^kStaleMax; (l, O) and
        // the final LSE use the same reference, which keeps the result exact
        // in real arithmetic.
        float m = -INFINITY;
        float l = 0.f;
        for (int j = 0; j < n_k; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(s_full, sc & 1, ctl, kSiteSFull));
            if (!ok) break;
            ++sc;
            tc_fence_after();
            // S row and its max over the tile in one TMEM load (the load's
            // max reduction)
            uint32_t raw[128];
            float mx;
            tmem_ld128_max(tm_s, raw, mx);
            float *sv = reinterpret_cast<float *>(raw);

            const int key0 = j * kBlockN;
            const bool ragged = key0 + kBlockN > N;
            const bool diag = CAUSAL && (key0 + kBlockN - 1 > sub_start);
            if (ragged || diag) {
                // keys past N or above the diagonal -> -inf, and the row max
                // over the remaining keys only: eight short chains of
                // three-input max over all kBlockN columns (0-15, then 16
                // more per step)
                int lim = N - key0;
                if (CAUSAL) lim = min(lim, qrow - key0 + 1);
#pragma unroll
                for (int c = 0; c < kBlockN; ++c)
                    if (c >= lim) sv[c] = -INFINITY;
                float pm[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) pm[t] = fmaxf(sv[t], sv[8 + t]);
#pragma unroll
                for (int c = 16; c + 16 <= kBlockN; c += 16)
#pragma unroll
                    for (int t = 0; t < 8; ++t) pm[t] = fmax3(pm[t], sv[c + t], sv[c + 8 + t]);
                mx = fmaxf(fmax3(pm[0], pm[1], pm[2]),
                           fmaxf(fmax3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7])));
            }
            const float cand = mx * cs;
            const float m_new = (cand > m + kStaleMax) ? cand : m;
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = (m == m_use) ? 1.f : ex2_approx(m - m_use);
            const uint64_t neg2 = f2_pack(-m_use, -m_use);
            uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
            for (int c = 0; c < kBlockN; c += 32) {
                uint32_t pk[16];
                exp_chunk32(sv + c, cs2, neg2, rs2, pk);
                tmem_st16(tm_s + c / 2, pk);
            }
            // Rescale O_k where the reference moved for some row of this
            // warp; the S_k(j) barrier also covered PV_k(j-1), so O_k is
            // settled.
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tm_o + 32 * c, o);
#pragma unroll
                    for (int t = 0; t < 32; t += 2) {
                        float x0, x1;
                        f2_unpack(f2_mul(f2_pack(__uint_as_float(o[t]), __uint_as_float(o[t + 1])),
                                         a2), x0, x1);
                        o[t] = __float_as_uint(x0);
                        o[t + 1] = __float_as_uint(x1);
                    }
                    tmem_st32(tm_o + 32 * c, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_ready);
            l = l * alpha + sum_pairs(rs2);
            m = m_new;
        }
        if (!ok) break;

        // ---- epilogue: O = a / l (bf16), LSE = (m + log2 l) ln 2
        ok = __all_sync(0xffffffffu, mbar_wait(o_full, r & 1, ctl, kSiteOFull));
        if (!ok) break;
        tc_fence_after();
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        const bool in_range = qrow < N;
        const long long row_flat = static_cast<long long>(w.bh) * N + qrow;
        __nv_bfloat16 *orow = p.O + (static_cast<size_t>(w.bh) * N + qrow) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tm_o + 32 * c, o);
            uint32_t pk[16];
#pragma unroll
            for (int t = 0; t < 16; ++t)
                pk[t] = pack_bf16x2(__uint_as_float(o[2 * t]) * inv_l,
                                    __uint_as_float(o[2 * t + 1]) * inv_l);
            if (in_range &&
                dbg_ok(row_flat < p.o_rows &&
                           (reinterpret_cast<uintptr_t>(orow + 32 * c) &
                            (p.o_align32 ? 31u : 15u)) == 0,
                       ctl, kChkStoreO)) {
                if (p.o_align32) {
                    st_global_v8(orow + 32 * c, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6],
                                 pk[7]);
                    st_global_v8(orow + 32 * c + 16, pk[8], pk[9], pk[10], pk[11], pk[12],
                                 pk[13], pk[14], pk[15]);
                } else {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        dst[t] = make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2],
                                            pk[4 * t + 3]);
                }
            }
        }
        // O_k is read out: the next item's first PV_k may overwrite it.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_empty);
        if (in_range && dbg_ok(row_flat < p.o_rows, ctl, kChkStoreLse)) {
            const float lse = (l > 0.f) ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
            p.LSE[static_cast<size_t>(w.bh) * N + qrow] = lse;
        }
    }
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const Params p) {
    using C = Cfg<D>;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    {
        const SmemView<D> v = smem_view<D>();
        if (threadIdx.x == 0) {
            mbar_init(v.q_full, 1);
            mbar_init(v.q_empty, 1);
            for (int s = 0; s < C::kStages; ++s) {
                mbar_init(&v.k_full[s], 1);
                mbar_init(&v.k_empty[s], 1);
                mbar_init(&v.v_full[s], 1);
                mbar_init(&v.v_empty[s], 1);
            }
            for (int k = 0; k < 2; ++k) {
                mbar_init(&v.s_full[k], 1);
                mbar_init(&v.p_full[k], 4);  // one arrive per softmax warp
                mbar_init(&v.o_full[k], 1);
                mbar_init(&v.o_empty[k], 4);
            }
            mbar_init(v.mma_done, 1);
            for (int k = 0; k < 2; ++k) {
                mbar_init(&v.sched_full[k], 1);
                mbar_init(&v.sched_empty[k], 9);  // the MMA warp and 8 softmax warps
            }
            mbar_init(v.claim, 1);
            *v.abort_flag = 0;
            fence_mbarrier_init();
        }
        if (warp == kTmaWarp && lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
        if (warp == kMmaWarp) {
            tmem_alloc(v.tmem_slot, kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // Each role runs inside the branch that set its register budget, and
    // rebuilds what it needs, so no value stays live across the switch.
    if (warp >= 8) {
        regs_decrease<kRegsControl>();
        if (warp == kTmaWarp)
            role_producer<D, CAUSAL>(&tmQ, &tmK, &tmV, p, lane);
        else if (warp == kMmaWarp)
            role_mma<D, CAUSAL>(p);
        __syncwarp();
    } else {
        regs_increase<kRegsSoftmax>();
        role_softmax<D, CAUSAL>(p, warp, lane);
    }

    // ---- teardown: every role has drained its own asynchronous work
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(*smem_view<D>().tmem_slot, kTmemCols);
    }
}

// Bounded-wait self test: one thread waits on a barrier nothing signals.
__global__ void fa_wait_selftest_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtl ctl{&abort_flag, &g_fa_status, limit_ns};
        mbar_wait(&bar, 0, ctl, 0x7F);
    }
}

#ifdef FA_DEBUG
// The fault fa_debug_arm armed for the next forward launch (debug build
// only), taken and disarmed by that launch.
static std::mutex g_arm_mu;
static int g_arm_fault = FA_DEBUG_NONE;
static long long g_arm_a = 0, g_arm_b = 0;
static uint64_t g_arm_limit_ns = 0;

bool take_debug_fault(DebugFault *f) {
    std::lock_guard<std::mutex> lock(g_arm_mu);
    if (g_arm_fault == FA_DEBUG_NONE) return false;
    f->fault = g_arm_fault;
    f->a = g_arm_a;
    f->b = g_arm_b;
    f->limit_ns = g_arm_limit_ns;
    g_arm_fault = FA_DEBUG_NONE;
    return true;
}

static void take_armed_fault(Params &p) {
    DebugFault f;
    if (!take_debug_fault(&f)) return;
    if (f.fault == FA_DEBUG_LOSE_K_ARRIVAL) {
        p.lose_item = f.a > 0x7FFFFFFFLL ? -1 : static_cast<int>(f.a);
        p.lose_tile = f.b > 0x7FFFFFFFLL ? -1 : static_cast<int>(f.b);
    } else if (f.fault == FA_DEBUG_SHRINK_OUTPUT) {
        p.o_rows = f.a < p.o_rows ? f.a : p.o_rows;
    }
    if (f.limit_ns) p.limit_ns = f.limit_ns;
}
#endif

template <int D, bool CAUSAL>
static int launch_t(const LaunchArgs &a) {
    using C = Cfg<D>;
    auto kern = fa_fwd_kernel<D, CAUSAL>;
    static std::atomic<int> configured[kMaxDevices];
    int dev = 0;
    FA_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_ARCH;
    const int rc = set_smem_once(configured, dev, kern, C::kSmemBytes);
    if (rc != FA_OK) return rc;
    const int sms = device_sm_count(dev);
    if (sms <= 0) return record_message(FA_ERR_LAUNCH, "cannot query the SM count");
    Params p;
    p.O = static_cast<__nv_bfloat16 *>(a.O);
    p.LSE = a.LSE;
    p.N = a.N;
    p.BH = a.BH;
    p.H = a.H;
    p.group = a.H / a.Hkv;
    p.n_qblocks = (a.N + kBlockM - 1) / kBlockM;
    p.n_ktiles = (a.N + kBlockN - 1) / kBlockN;
    const long long items = static_cast<long long>(p.n_qblocks) * a.BH;
    if (items > 0x7FFFFFFFLL) return FA_ERR_SHAPE;
    p.n_items = static_cast<int>(items);
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.limit_ns = a.limit_ns;
    p.o_align32 = (reinterpret_cast<uintptr_t>(a.O) & 31u) == 0 ? 1 : 0;
    p.o_rows = static_cast<long long>(a.BH) * a.N;
    p.lose_item = -1;
    p.lose_tile = -1;
#ifdef FA_DEBUG
    take_armed_fault(p);
#endif
    // Causal head groups: each group holds about two waves of its heaviest
    // items (a head brings n_qblocks items, the heaviest twice the average),
    // whole K/V groups of grouped-query heads, at most all heads.
    long long hg = (2LL * sms + p.n_qblocks) / (p.n_qblocks + 1);
    hg = (hg + p.group - 1) / p.group * p.group;
    if (hg > a.BH) hg = a.BH;
    if (hg < 1) hg = 1;
    p.head_group = static_cast<int>(hg);
    p.first_group = a.BH % p.head_group == 0 ? p.head_group : a.BH % p.head_group;
    // one CTA per work item; one fits on an SM (shared memory), and the
    // CTAs that run take over the others' items (cluster launch control)
    kern<<<p.n_items, kThreads, C::kSmemBytes, a.stream>>>(*a.tmQ, *a.tmK, *a.tmV, p);
    FA_CUDA_TRY(cudaGetLastError());
    return FA_OK;
}

int launch_fwd(const LaunchArgs &a) {
    if (a.d == 64) return a.causal ? launch_t<64, true>(a) : launch_t<64, false>(a);
    if (a.d == 128) return a.causal ? launch_t<128, true>(a) : launch_t<128, false>(a);
    if (a.d == 256) return launch_fwd256(a);
    return FA_ERR_HEADDIM;
}

int read_and_clear_status(cudaStream_t stream, int *status) {
    FA_CUDA_TRY(cudaStreamSynchronize(stream));
    int v = 0;
    FA_CUDA_TRY(cudaMemcpyFromSymbol(&v, g_fa_status, sizeof v));
    if (v != 0) {
        const int zero = 0;
        FA_CUDA_TRY(cudaMemcpyToSymbol(g_fa_status, &zero, sizeof zero));
    }
    *status = v;
    return FA_OK;
}

int launch_wait_selftest(uint64_t limit_ns, cudaStream_t stream) {
    fa_wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
    FA_CUDA_TRY(cudaGetLastError());
    return FA_OK;
}

}  // namespace fa

#ifdef FA_DEBUG
extern "C" int fa_debug_arm(int fault, long long a, long long b, int limit_us) {
    if (fault != FA_DEBUG_NONE && fault != FA_DEBUG_LOSE_K_ARRIVAL &&
        fault != FA_DEBUG_SHRINK_OUTPUT)
        return FA_ERR_UNSUPPORTED;
    if (a < 0 || b < 0 || limit_us < 0 || limit_us > 1000000) return FA_ERR_SHAPE;
    std::lock_guard<std::mutex> lock(fa::g_arm_mu);
    fa::g_arm_fault = fault;
    fa::g_arm_a = a;
    fa::g_arm_b = b;
    fa::g_arm_limit_ns = fault == FA_DEBUG_NONE ? 0 : static_cast<uint64_t>(limit_us) * 1000ull;
    return FA_OK;
}
#endif
