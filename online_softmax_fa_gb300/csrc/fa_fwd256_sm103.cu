// fa_fwd256_sm103.cu -- the exact attention forward pass at head dimension
// 256 for sm_103a (GB300).
//
// Same computation as fa_fwd_sm103.cu (the online-softmax recurrence of
// "Understanding FlashAttention Pt 1", wpnews.pro, section 2.4, with the
// final normalisation and LSE of "FlashAttention-2 -- Deeper Math",
// aicassindra.com, "Fix 1" and "Fix 2"), laid out for d = 256, which the
// pages list beside 64 and 128 among the supported head dimensions.
//
// At d = 256 one 128-row accumulator O takes 256 of the 512 TMEM columns,
// so a work item is one (b, h, 128-row query block), and the other 256
// columns hold S twice: S(j+1) = Q K_{j+1}^T is computed while the softmax
// warps turn S(j) into P(j), and O += P(j) V_j follows.  Per key tile the
// tensor pipe has 2 x 1024 cycles of work and the softmax of a 128 x 128
// tile takes less, so the pipe, not the softmax, sets the pace.
//   * warp 5 (TMA and schedule): per item the query block (4 boxes of 64
//     columns), then K tiles in halves of 128 columns (d) through a 3-stage
//     ring; it claims the next item (cluster launch control: the grid has a
//     CTA per item, and a running CTA cancels the launch of the next one and
//     does its item) and passes it on through a two-slot ring, exactly as
//     in the d <= 128 kernel, with the same order of items.
//   * warp 6 (TMA): V tiles in halves of 64 keys through a 2-stage ring.
//   * warp 4 (MMA): S(j) as 16 MMAs of M128 x N128 x K16 (K over d), P(j)V_j
//     as 8 MMAs of M128 x N256 x K16 (K over keys) with P read from TMEM.
//   * warps 0-3 (softmax, thread = query row): as in the d <= 128 kernel,
//     with the reference max moving only when a row's max passes it by more
//     than 2^8; when it moves, O is rescaled in TMEM after the previous
//     P V has completed (o_ready).  Epilogue O = a / l, LSE = (m + log2 l) ln 2.
//   * causal: key tiles above the diagonal are skipped, the diagonal masked.
// TMEM: O [0,256), S buffers [256,384) and [384,512); P(j) is bf16 over the
// first 64 columns of its S buffer.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_internal.h"
#include "sm103_primitives.cuh"
#include "debug_checks.cuh"
#ifdef FA_DEBUG
#include "../../include/fa_debug.h"
#endif

namespace fa {

__device__ int g_fa_status_256;  // bounded-wait timeouts of this kernel

namespace f256 {

constexpr int kD = 256;
constexpr int kBlockM = 128;  // query rows per item (TMEM lanes)
constexpr int kBlockN = 128;  // keys per tile
constexpr int kThreads = 256;
constexpr int kMmaWarp = 4, kTmaKWarp = 5, kTmaVWarp = 6;  // warp 7: no role
constexpr int kBox = 128 * 128;   // Q / K box: 128 rows x 64 bf16
constexpr int kVBox = 64 * 128;   // V box: 64 rows x 64 bf16
constexpr int kStagesK = 3, kStagesV = 2;
constexpr int kQBytes = 4 * kBox;    // 128 x 256
constexpr int kKStage = 2 * kBox;    // 128 keys x 128 d
constexpr int kVStage = 4 * kVBox;   // 64 keys x 256 d
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;
constexpr int kOffV = kOffK + kStagesK * kKStage;
constexpr int kOffBar = kOffV + kStagesV * kVStage;
// q_full, q_empty, k_full[3], k_empty[3], v_full[2], v_empty[2], s_full[2],
// p_full, o_ready, o_full, o_empty, mma_done, sched_full[2], sched_empty[2],
// claim; then (16-byte aligned) the tmem slot, the abort flag, the two item
// slots and the 16-byte claim answer
constexpr int kNumBars = 2 + 2 * kStagesK + 2 * kStagesV + 2 + 5 + 5;
constexpr int kOffMisc = (kOffBar + 8 * kNumBars + 15) / 16 * 16;
constexpr int kSmemBytes = kOffMisc + 32 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmO = 0, kTmS = 256;  // S buffer b at kTmS + 128 b
constexpr uint32_t kIdescS = idesc_bf16_f32(kBlockM, kBlockN, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBlockM, kD, true);
constexpr float kStaleMax = 8.0f;
// Causal: the next item is claimed this many key tiles before the end of the
// current item's K loads (see the d <= 128 kernel); without a mask at the
// start of an item.
constexpr int kClaimLead = 3;

enum : int {
    kSiteQ = 0x41, kSiteK, kSiteV, kSiteP, kSiteS, kSiteOReady, kSiteOFull, kSiteOEmpty,
    kSiteQEmpty, kSiteKEmpty, kSiteVEmpty, kSiteSchedFull, kSiteSchedEmpty, kSiteClaim
};

struct Params {
    __nv_bfloat16 *O;
    float *LSE;
    int N, BH, H, group;
    int n_qblocks;  // ceil(N / 128)
    int n_ktiles;   // ceil(N / 128)
    int n_items;    // BH x n_qblocks = the grid
    int head_group;   // causal order: heads per group
    int first_group;  // heads in the first (partial) group
    float scale_log2;
    uint64_t limit_ns;
    // debug build only: the extent (rows of O and LSE) the store checks
    // use, and an injected fault -- the producer of item lose_item skips the
    // load of the first K half of key tile lose_tile and the arrival on its
    // barrier (-1: none)
    long long o_rows;
    int lose_item, lose_tile;
};

struct View {
    uint8_t *q, *k, *v;
    uint64_t *q_full, *q_empty, *k_full, *k_empty, *v_full, *v_empty, *s_full, *p_full,
        *o_ready, *o_full, *o_empty, *mma_done, *sched_full, *sched_empty, *claim;
    uint32_t *tmem_slot;
    volatile int *abort_flag;
    volatile int *sched_item;  // [2]: work item, or -1 = no more work
    void *claim_resp;          // 16 bytes, 16-byte aligned
};

__device__ __forceinline__ View view() {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    View v;
    v.q = smem + kOffQ;
    v.k = smem + kOffK;
    v.v = smem + kOffV;
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + kOffBar);
    v.q_full = b;
    v.q_empty = b + 1;
    v.k_full = b + 2;
    v.k_empty = v.k_full + kStagesK;
    v.v_full = v.k_empty + kStagesK;
    v.v_empty = v.v_full + kStagesV;
    v.s_full = v.v_empty + kStagesV;
    v.p_full = v.s_full + 2;
    v.o_ready = v.p_full + 1;
    v.o_full = v.o_ready + 1;
    v.o_empty = v.o_full + 1;
    v.mma_done = v.o_empty + 1;
    v.sched_full = v.mma_done + 1;
    v.sched_empty = v.sched_full + 2;
    v.claim = v.sched_empty + 2;
    v.tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    v.abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    v.sched_item = reinterpret_cast<volatile int *>(smem + kOffMisc + 8);
    v.claim_resp = smem + kOffMisc + 16;
    return v;
}

struct Work {
    int bh, kvh, qb, n;  // n: key tiles this query block needs
};

// Debug checks: a range inside this kernel's shared memory.
__device__ __forceinline__ bool in_smem_256(const void *ptr, int bytes) {
    return in_smem(ptr, bytes, kSmemBytes);
}

// Work item x (the grid's CTA index, in priority order) -> (head, query
// block), as in the d <= 128 kernel: causal, heads in groups (the partial
// group first) and inside a group the heaviest query block first with the
// group's heads interleaved; otherwise head-major.
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
    const int b = w.bh / p.H, h = w.bh - b * p.H;
    w.kvh = b * (p.H / p.group) + h / p.group;
    w.n = CAUSAL ? min(p.n_ktiles, min(w.qb * kBlockM + kBlockM - 1, p.N - 1) / kBlockN + 1)
                 : p.n_ktiles;
    return w;
}

// The r-th work item of this CTA as the Q/K load warp published it (-1: no
// more work).  Called by every thread of a consumer warp; one lane then
// frees the slot.
__device__ __forceinline__ bool next_item(const View &v, const WaitCtl &ctl, int r, int lane,
                                          int n_items, int &x) {
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

// ---------------------------------------------------------------- producers
template <bool CAUSAL>
__device__ __forceinline__ void role_load_qk(const CUtensorMap *tmQ, const CUtensorMap *tmK,
                                             const Params &p, int lane) {
    if (lane != 0) return;
    const View v = view();
    const WaitCtl ctl{v.abort_flag, &g_fa_status_256, p.limit_ns};
    int u = 0;      // K halves issued, across items
    int items = 0;  // query blocks issued
    // claims: 2 x (claims answered so far) + (1 if one is on its way); -1
    // once a claim has failed (no further claim may be made)
    int claims = 0;
    bool ok = true;
    int x = static_cast<int>(blockIdx.x);  // this CTA's own item first
    for (int r = 0;; ++r) {
        // publish item x (or the end of the work); slot r & 1 last held
        // item r - 2
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
        if (r > 0) {  // the previous item's last S has read Q
            ok = mbar_wait(v.q_empty, (r - 1) & 1, ctl, kSiteQEmpty);
            if (!ok) break;
        }
        if (!dbg_ok(w.bh >= 0 && w.bh < p.BH && w.qb >= 0 && w.qb < p.n_qblocks, ctl,
                    kChkTmaQ) ||
            !dbg_ok(in_smem_256(v.q, kQBytes), ctl, kChkSmem)) {
            ok = false;
            break;
        }
        mbar_arrive_expect_tx(v.q_full, kQBytes);
        {
            const uint64_t pol_q = l2_policy_evict_first();
            for (int c = 0; c < 4; ++c)
                tma_load_3d(v.q + c * kBox, tmQ, v.q_full, 64 * c, w.qb * kBlockM, w.bh, pol_q);
        }
        ++items;
        const int claim_at = CAUSAL ? max(0, w.n - kClaimLead) : 0;
        for (int j = 0; j < w.n && ok; ++j) {
            if (j == claim_at && claims >= 0) {  // ask for the next item
                mbar_arrive_expect_tx(v.claim, 16);
                clc_try_cancel(v.claim_resp, v.claim);
                claims |= 1;
            }
            const uint64_t pol_kv = l2_policy_evict_last();
            for (int h = 0; h < 2; ++h) {  // d columns [128h, 128h + 128)
                const int s = u % kStagesK;
                if (u >= kStagesK)
                    ok = mbar_wait(&v.k_empty[s], ((u / kStagesK) & 1) ^ 1, ctl, kSiteKEmpty);
                if (!ok) break;
                if (!dbg_ok(j * kBlockN < p.N && w.kvh >= 0 && w.kvh < p.BH / p.group, ctl,
                            kChkTmaKV) ||
                    !dbg_ok(in_smem_256(v.k + s * kKStage, kKStage), ctl, kChkSmem)) {
                    ok = false;
                    break;
                }
                // debug build: an injected fault loses this K half's load and
                // its arrival (the consumers' waits then run out)
                if (!(kDebug && x == p.lose_item && j == p.lose_tile && h == 0)) {
                    mbar_arrive_expect_tx(&v.k_full[s], kKStage);
                    for (int c = 0; c < 2; ++c)
                        tma_load_3d(v.k + s * kKStage + c * kBox, tmK, &v.k_full[s],
                                    64 * (2 * h + c), j * kBlockN, w.kvh, pol_kv);
                }
                ++u;
            }
        }
        if (!ok) break;
        // the next item: the cancelled CTA's, if the claim succeeded
        x = -1;
        if (claims > 0 && (claims & 1)) {
            ok = mbar_wait(v.claim, (claims >> 1) & 1, ctl, kSiteClaim);
            if (!ok) break;
            claims += 1;  // answered: clear the pending bit, count it
            x = clc_cancelled_x(v.claim_resp);
            if (x < 0) claims = -1;
        }
    }
    // drain the query block, the K stages and a claim answer in flight
    if (items > 0) mbar_wait_drain(v.q_full, (items - 1) & 1, p.limit_ns);
    for (int t = max(0, u - kStagesK); t < u; ++t)
        mbar_wait_drain(&v.k_full[t % kStagesK], (t / kStagesK) & 1, p.limit_ns);
    if (claims > 0 && (claims & 1)) mbar_wait_drain(v.claim, (claims >> 1) & 1, p.limit_ns);
}

template <bool CAUSAL>
__device__ __forceinline__ void role_load_v(const CUtensorMap *tmV64, const Params &p, int lane) {
    // the whole warp walks the items (the item ring is read warp-wide);
    // lane 0 waits for ring stages and issues the loads
    const View v = view();
    const WaitCtl ctl{v.abort_flag, &g_fa_status_256, p.limit_ns};
    int u = 0;  // V halves issued, across items (lane 0)
    bool ok = true;
    for (int r = 0; ok; ++r) {
        int x;
        ok = next_item(v, ctl, r, lane, p.n_items, x);
        if (!ok || x < 0) break;
        const Work w = work_of<CAUSAL>(p, x);
        if (lane == 0) {
            const uint64_t pol_kv = l2_policy_evict_last();
            for (int j = 0; j < w.n && ok; ++j) {
                for (int h = 0; h < 2; ++h) {  // keys [64h, 64h + 64) of tile j
                    const int s = u % kStagesV;
                    if (u >= kStagesV)
                        ok = mbar_wait(&v.v_empty[s], ((u / kStagesV) & 1) ^ 1, ctl,
                                       kSiteVEmpty);
                    if (!ok) break;
                    if (!dbg_ok(j < p.n_ktiles && w.kvh >= 0 && w.kvh < p.BH / p.group, ctl,
                                kChkTmaKV) ||
                        !dbg_ok(in_smem_256(v.v + s * kVStage, kVStage), ctl, kChkSmem)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&v.v_full[s], kVStage);
                    for (int c = 0; c < 4; ++c)
                        tma_load_3d(v.v + s * kVStage + c * kVBox, tmV64, &v.v_full[s],
                                    64 * c, j * kBlockN + 64 * h, w.kvh, pol_kv);
                    ++u;
                }
            }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0)
        for (int t = max(0, u - kStagesV); t < u; ++t)
            mbar_wait_drain(&v.v_full[t % kStagesV], (t / kStagesV) & 1, p.limit_ns);
    __syncwarp();
}

// -------------------------------------------------------------- MMA issuer
// Whole warp converged; elect.sync inside the issue helpers picks the lane.
template <bool CAUSAL>
__device__ __forceinline__ void role_mma(const Params &p) {
    const View v = view();
    const WaitCtl ctl{v.abort_flag, &g_fa_status_256, p.limit_ns};
    const uint32_t tmem = *v.tmem_slot;
    const uint64_t dq0 = sdesc_sw128(smem_u32(v.q), 16, 1024);
    const uint64_t dk0 = sdesc_sw128(smem_u32(v.k), 16, 1024);
    const uint64_t dv0 = sdesc_sw128(smem_u32(v.v), kVBox, 1024);  // MN-major, 64-row boxes
    const auto wait = [&](uint64_t *bar, uint32_t parity, int site) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl, site));
    };
    int uk = 0, uv = 0;  // K / V halves consumed, across items
    int t = 0;           // key tiles processed, across items (S buffer t & 1)
    const bool layout_ok =
        dbg_ok(whole_tmem(tmem), ctl, kChkTmem) &&
        dbg_ok(in_smem_256(v.q, kQBytes) && in_smem_256(v.k, kStagesK * kKStage) &&
                   in_smem_256(v.v, kStagesV * kVStage),
               ctl, kChkSmem);
    // S(t) = Q K^T: 16 K-steps over d, two K halves of 8 steps each.
    const auto issue_s = [&](int tt) -> bool {
        const uint32_t d_tm = tmem + kTmS + (tt & 1) * kBlockN;
        for (int h = 0; h < 2; ++h) {
            const int s = uk % kStagesK;
            if (!wait(&v.k_full[s], (uk / kStagesK) & 1, kSiteK)) return false;
            tc_fence_after();
            const uint64_t dk = dk0 + static_cast<uint64_t>((s * kKStage) >> 4);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {  // d = 128h + 16kk
                const int c = kk >> 2;        // chunk within the half
                const uint64_t ok_ = static_cast<uint64_t>((c * kBox + (kk & 3) * 32) >> 4);
                const uint64_t oq = static_cast<uint64_t>(((2 * h + c) * kBox + (kk & 3) * 32) >> 4);
                mma_ss_elect(d_tm, dq0 + oq, dk + ok_, kIdescS, (h > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit_elect(&v.k_empty[s]);
            ++uk;
        }
        return true;
    };
    const int lane = static_cast<int>(threadIdx.x & 31);
    bool ok = layout_ok;
    for (int r = 0; ok; ++r) {
        int x;
        ok = next_item(v, ctl, r, lane, p.n_items, x);
        if (!ok || x < 0) break;
        const Work w = work_of<CAUSAL>(p, x);
        ok = wait(v.q_full, r & 1, kSiteQ);
        if (!ok) break;
        tc_fence_after();
        ok = issue_s(t);
        if (!ok) break;
        if (w.n == 1) mma_commit_elect(v.q_empty);  // last read of Q issued
        mma_commit_elect(&v.s_full[t & 1]);
        for (int j = 0; j < w.n && ok; ++j, ++t) {
            if (j + 1 < w.n) {  // S(t+1) into the buffer PV(t-1) has read
                ok = issue_s(t + 1);
                if (!ok) break;
                if (j + 2 == w.n) mma_commit_elect(v.q_empty);
                mma_commit_elect(&v.s_full[(t + 1) & 1]);
            }
            if (j == 0 && r > 0) {  // O read out by the previous item's epilogue
                ok = wait(v.o_empty, (r - 1) & 1, kSiteOEmpty);
                if (!ok) break;
            }
            ok = wait(v.p_full, t & 1, kSiteP);
            if (!ok) break;
            tc_fence_after();
            // O += P(t) V_t: 8 K-steps over keys, two V halves of 4 steps each
            const uint32_t p_tm = tmem + kTmS + (t & 1) * kBlockN;
            for (int h = 0; h < 2 && ok; ++h) {
                const int s = uv % kStagesV;
                ok = wait(&v.v_full[s], (uv / kStagesV) & 1, kSiteV);
                if (!ok) break;
                tc_fence_after();
                const uint64_t dv = dv0 + static_cast<uint64_t>((s * kVStage) >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ts_elect(tmem + kTmO, p_tm + (4 * h + kk) * 8,
                                 dv + static_cast<uint64_t>((kk * 16 * 128) >> 4), kIdescPV,
                                 (j > 0 || h > 0 || kk > 0) ? 1u : 0u);
                mma_commit_elect(&v.v_empty[s]);
                ++uv;
            }
            if (!ok) break;
            mma_commit_elect(v.o_ready);
            if (j + 1 == w.n) mma_commit_elect(v.o_full);
        }
    }
    // every MMA issued completes before the CTA frees its tensor memory
    mma_commit_elect(v.mma_done);
    mbar_wait_drain(v.mma_done, 0, p.limit_ns);
}

// ------------------------------------------------------------------ softmax
// p = 2^(s*c - m) for 32 consecutive scores, row sum into rs2, bf16 pairs.
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

template <bool CAUSAL>
__device__ __forceinline__ void role_softmax(const Params &p, int warp, int lane) {
    const View v = view();
    const WaitCtl ctl{v.abort_flag, &g_fa_status_256, p.limit_ns};
    const uint32_t tmem = *v.tmem_slot;
    const int N = p.N;
    const int row = warp * 32 + lane;
    const uint32_t lane_bits = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tm_o = tmem + lane_bits + kTmO;
    const float cs = p.scale_log2;
    const uint64_t cs2 = f2_pack(cs, cs);
    int t = 0;  // key tiles consumed, across items
    bool ok = dbg_ok(whole_tmem(tmem), ctl, kChkTmem);
    for (int r = 0; ok; ++r) {
        int x;
        ok = next_item(v, ctl, r, lane, p.n_items, x);
        if (!ok || x < 0) break;
        const Work w = work_of<CAUSAL>(p, x);
        const int qrow = w.qb * kBlockM + row;
        // reference max m (base 2, scale folded in) and running sum l; the
        // reference moves only when a row's max passes it by more than
        // kStaleMax, so p <= 2^kStaleMax
        float m = -INFINITY, l = 0.f;
        for (int j = 0; j < w.n; ++j, ++t) {
            ok = __all_sync(0xffffffffu, mbar_wait(&v.s_full[t & 1], (t >> 1) & 1, ctl, kSiteS));
            if (!ok) break;
            tc_fence_after();
            const uint32_t tm_s = tmem + lane_bits + kTmS + (t & 1) * kBlockN;
            // S row and its max over the tile in one TMEM load (the load's
            // max reduction)
            uint32_t raw[128];
            float mx;
            tmem_ld128_max(tm_s, raw, mx);
            float *sv = reinterpret_cast<float *>(raw);
            const int key0 = j * kBlockN;
            const bool ragged = key0 + kBlockN > N;
            const bool diag = CAUSAL && (key0 + kBlockN - 1 > w.qb * kBlockM);
            if (ragged || diag) {
                // keys past N or above the diagonal -> -inf, and the row max
                // over the remaining keys only (columns 0-15, then 16 more
                // per step)
                int lim = N - key0;
                if (CAUSAL) lim = min(lim, qrow - key0 + 1);
#pragma unroll
                for (int c = 0; c < kBlockN; ++c)
                    if (c >= lim) sv[c] = -INFINITY;
                float pm[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) pm[e] = fmaxf(sv[e], sv[8 + e]);
#pragma unroll
                for (int c = 16; c + 16 <= kBlockN; c += 16)
#pragma unroll
                    for (int e = 0; e < 8; ++e) pm[e] = fmax3(pm[e], sv[c + e], sv[c + 8 + e]);
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
            // rescale O where the reference moved for some row of this warp,
            // once the previous tile's P V has landed in O
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                ok = __all_sync(0xffffffffu,
                                mbar_wait(v.o_ready, (t - 1) & 1, ctl, kSiteOReady));
                if (!ok) break;
                tc_fence_after();
                const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
                for (int c = 0; c < kD / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tm_o + 32 * c, o);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float x0, x1;
                        f2_unpack(f2_mul(f2_pack(__uint_as_float(o[e]), __uint_as_float(o[e + 1])),
                                         a2), x0, x1);
                        o[e] = __float_as_uint(x0);
                        o[e + 1] = __float_as_uint(x1);
                    }
                    tmem_st32(tm_o + 32 * c, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(v.p_full);
            float a, b, c2, d2;
            f2_unpack(f2_add(rs2[0], rs2[1]), a, b);
            f2_unpack(f2_add(rs2[2], rs2[3]), c2, d2);
            l = l * alpha + ((a + b) + (c2 + d2));
            m = m_new;
        }
        if (!ok) break;
        // ---- epilogue: O = a / l (bf16), LSE = (m + log2 l) ln 2
        ok = __all_sync(0xffffffffu, mbar_wait(v.o_full, r & 1, ctl, kSiteOFull));
        if (!ok) break;
        tc_fence_after();
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        const bool in_range = qrow < N;
        const long long row_flat = static_cast<long long>(w.bh) * N + qrow;
        __nv_bfloat16 *orow = p.O + (static_cast<size_t>(w.bh) * N + qrow) * kD;
#pragma unroll 1
        for (int c = 0; c < kD / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tm_o + 32 * c, o);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
                pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l,
                                    __uint_as_float(o[2 * e + 1]) * inv_l);
            if (in_range &&
                dbg_ok(row_flat < p.o_rows &&
                           (reinterpret_cast<uintptr_t>(orow + 32 * c) & 15u) == 0,
                       ctl, kChkStoreO)) {
                uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(v.o_empty);  // O may be overwritten by the next item
        if (in_range && dbg_ok(row_flat < p.o_rows, ctl, kChkStoreLse)) {
            const float lse = (l > 0.f) ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
            p.LSE[static_cast<size_t>(w.bh) * N + qrow] = lse;
        }
    }
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd256_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV64, const Params p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    {
        const View v = view();
        if (threadIdx.x == 0) {
            mbar_init(v.q_full, 1);
            mbar_init(v.q_empty, 1);
            for (int s = 0; s < kStagesK; ++s) {
                mbar_init(&v.k_full[s], 1);
                mbar_init(&v.k_empty[s], 1);
            }
            for (int s = 0; s < kStagesV; ++s) {
                mbar_init(&v.v_full[s], 1);
                mbar_init(&v.v_empty[s], 1);
            }
            mbar_init(&v.s_full[0], 1);
            mbar_init(&v.s_full[1], 1);
            mbar_init(v.p_full, 4);
            mbar_init(v.o_ready, 1);
            mbar_init(v.o_full, 1);
            mbar_init(v.o_empty, 4);
            mbar_init(v.mma_done, 1);
            for (int k = 0; k < 2; ++k) {
                mbar_init(&v.sched_full[k], 1);
                mbar_init(&v.sched_empty[k], 6);  // V load, MMA and 4 softmax warps
            }
            mbar_init(v.claim, 1);
            *v.abort_flag = 0;
            fence_mbarrier_init();
        }
        if (warp == kTmaKWarp && lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV64);
        }
        if (warp == kMmaWarp) {
            tmem_alloc(v.tmem_slot, kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp < 4)
        role_softmax<CAUSAL>(p, warp, lane);
    else if (warp == kMmaWarp)
        role_mma<CAUSAL>(p);
    else if (warp == kTmaKWarp)
        role_load_qk<CAUSAL>(&tmQ, &tmK, p, lane);
    else if (warp == kTmaVWarp)
        role_load_v<CAUSAL>(&tmV64, p, lane);
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(*view().tmem_slot, kTmemCols);
    }
}

}  // namespace f256

template <bool CAUSAL>
static int launch_256_t(const LaunchArgs &a) {
    auto kern = f256::fa_fwd256_kernel<CAUSAL>;
    static std::atomic<int> configured[kMaxDevices];
    int dev = 0;
    FA_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_ARCH;
    const int rc = set_smem_once(configured, dev, kern, f256::kSmemBytes);
    if (rc != FA_OK) return rc;
    const int sms = device_sm_count(dev);
    if (sms <= 0) return record_message(FA_ERR_LAUNCH, "cannot query the SM count");
    f256::Params p;
    p.O = static_cast<__nv_bfloat16 *>(a.O);
    p.LSE = a.LSE;
    p.N = a.N;
    p.BH = a.BH;
    p.H = a.H;
    p.group = a.H / a.Hkv;
    p.n_qblocks = (a.N + f256::kBlockM - 1) / f256::kBlockM;
    p.n_ktiles = (a.N + f256::kBlockN - 1) / f256::kBlockN;
    const long long items = static_cast<long long>(p.n_qblocks) * a.BH;
    if (items > 0x7FFFFFFFLL) return FA_ERR_SHAPE;
    p.n_items = static_cast<int>(items);
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.limit_ns = a.limit_ns;
    p.o_rows = static_cast<long long>(a.BH) * a.N;
    p.lose_item = -1;
    p.lose_tile = -1;
#ifdef FA_DEBUG
    DebugFault f;
    if (take_debug_fault(&f)) {
        if (f.fault == FA_DEBUG_LOSE_K_ARRIVAL) {
            p.lose_item = f.a > 0x7FFFFFFFLL ? -1 : static_cast<int>(f.a);
            p.lose_tile = f.b > 0x7FFFFFFFLL ? -1 : static_cast<int>(f.b);
        } else if (f.fault == FA_DEBUG_SHRINK_OUTPUT) {
            p.o_rows = f.a < p.o_rows ? f.a : p.o_rows;
        }
        if (f.limit_ns) p.limit_ns = f.limit_ns;
    }
#endif
    // causal head groups of about two waves of their heaviest items, whole
    // K/V groups, at most all heads (as in the d <= 128 kernel)
    long long hg = (2LL * sms + p.n_qblocks) / (p.n_qblocks + 1);
    hg = (hg + p.group - 1) / p.group * p.group;
    if (hg > a.BH) hg = a.BH;
    if (hg < 1) hg = 1;
    p.head_group = static_cast<int>(hg);
    p.first_group = a.BH % p.head_group == 0 ? p.head_group : a.BH % p.head_group;
    // one CTA per work item; the CTAs that run take over the others' items
    kern<<<p.n_items, f256::kThreads, f256::kSmemBytes, a.stream>>>(*a.tmQ, *a.tmK, *a.tmV64,
                                                                     p);
    FA_CUDA_TRY(cudaGetLastError());
    return FA_OK;
}

int launch_fwd256(const LaunchArgs &a) {
    return a.causal ? launch_256_t<true>(a) : launch_256_t<false>(a);
}

int fwd256_read_and_clear_status(int *status) {
    int v = 0;
    FA_CUDA_TRY(cudaMemcpyFromSymbol(&v, g_fa_status_256, sizeof v));
    if (v != 0) {
        const int zero = 0;
        FA_CUDA_TRY(cudaMemcpyToSymbol(g_fa_status_256, &zero, sizeof zero));
    }
    *status = v;
    return FA_OK;
}

}  // namespace fa
