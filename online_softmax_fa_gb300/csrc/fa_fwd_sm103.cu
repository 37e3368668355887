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
// GB300 mapping (one CTA per (b, h, 256-row query block), "Fix 3"/"Fix 4"):
//   * warp 9 (TMA): loads the query block once, then streams 128-key K and
//     V tiles through separate multi-stage shared-memory rings.
//   * warp 8 (MMA): one thread issues tcgen05 MMAs.  The query block is two
//     128-row sub-tiles; S_k = Q_k K_j^T lands in TMEM (fp32), and
//     O_k += P_k V_j reads P_k from TMEM (bf16, written over S_k) and V_j
//     from shared memory, accumulating O_k in TMEM.  The issue order
//     S_0(j), PV_1(j-1), S_1(j), PV_0(j) keeps the tensor pipe busy while
//     the two softmax groups work on the other sub-tile.
//   * warps 0-3 / 4-7 (softmax, one group per sub-tile; thread = row):
//     TMEM -> registers, mask (diagonal / ragged tiles only), row max with
//     the scale folded into base-2 exponents, p = 2^(s*c - m), row sum in
//     fp32, P -> TMEM as bf16, and the rescale of O_k in TMEM only for
//     warps where some row's max moved.  After the last tile: O = a / l in
//     bf16 and LSE = (m + log2 l) ln 2.
//   * causal: key tiles entirely above the diagonal are never loaded or
//     computed; only diagonal tiles are masked ("Causal masking: skip the
//     blocks, do not mask them"), and CTAs start heaviest query block first.
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

namespace fa {

// Device status word read by fa_device_error(): 0 or the site of the first
// bounded wait that expired.
__device__ int g_fa_status;

constexpr int kBlockM = 256;  // query rows per CTA (two 128-row sub-tiles)
constexpr int kSubM = 128;    // rows per sub-tile = TMEM lanes
constexpr int kBlockN = 128;  // keys per K/V tile
constexpr int kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 64 bf16
constexpr int kThreads = 320;         // 10 warps
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr uint32_t kTmemCols = 512;

// wait sites recorded in the status word on a timeout
enum : int {
    kSiteQ = 1, kSiteKFull, kSiteVFull, kSitePFull, kSiteKEmpty, kSiteVEmpty,
    kSiteSFull, kSiteOFull
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
    // barriers: q_full, k_full[S], k_empty[S], v_full[S], v_empty[S],
    // s_full[2], p_full[2], o_full, then tmem slot + abort flag
    static constexpr int kNumBars = 1 + 4 * kStages + 2 + 2 + 1;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
    static constexpr uint32_t kTmS0 = 0, kTmS1 = 128, kTmO0 = 256, kTmO1 = 256 + D;
    static constexpr uint32_t kIdescS = idesc_bf16_f32(kSubM, kBlockN, false);
    static constexpr uint32_t kIdescPV = idesc_bf16_f32(kSubM, D, true);
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(256 + 2 * D <= (int)kTmemCols, "TMEM budget");
};

struct Params {
    __nv_bfloat16 *O;
    float *LSE;
    int N;
    int n_qblocks;  // ceil(N / 256)
    int n_ktiles;   // ceil(N / 128)
    float scale_log2;  // scale * log2(e)
    uint64_t limit_ns;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const Params p) {
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem + C::kOffQ;
    uint8_t *sK = smem + C::kOffK;
    uint8_t *sV = smem + C::kOffV;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *q_full = bars;
    uint64_t *k_full = bars + 1;
    uint64_t *k_empty = k_full + C::kStages;
    uint64_t *v_full = k_empty + C::kStages;
    uint64_t *v_empty = v_full + C::kStages;
    uint64_t *s_full = v_empty + C::kStages;
    uint64_t *p_full = s_full + 2;
    uint64_t *o_full = p_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work item: head-major, heaviest query block first when causal
    const int bh = blockIdx.x / p.n_qblocks;
    const int qi = blockIdx.x % p.n_qblocks;
    const int qb = CAUSAL ? (p.n_qblocks - 1 - qi) : qi;
    const int N = p.N;
    const int T = p.n_ktiles;
    // key tiles each sub-tile needs (causal: up to its last row's diagonal)
    const int n_sub0 = CAUSAL ? min(T, min(qb * kBlockM + kSubM - 1, N - 1) / kBlockN + 1) : T;
    const int n_sub1 =
        CAUSAL ? min(T, min(qb * kBlockM + 2 * kSubM - 1, N - 1) / kBlockN + 1) : T;
    const int n_tiles = n_sub1;  // n_sub1 >= n_sub0

    // ---- setup
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&s_full[k], 1);
            mbar_init(&p_full[k], 4);  // one arrive per softmax warp
        }
        mbar_init(o_full, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == kTmaWarp && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const WaitCtl ctl{abort_flag, &g_fa_status, p.limit_ns};

    if (warp == kTmaWarp) {
        // =========================== TMA producer ===========================
        if (lane == 0) {
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            int issued_k = 0, issued_v = 0;
            mbar_arrive_expect_tx(q_full, C::kQBytes);
            for (int k = 0; k < 2; ++k)
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sQ + (k * C::kChunks + c) * kBoxBytes, &tmQ, q_full, 64 * c,
                                qb * kBlockM + k * kSubM, bh, pol_q);
            bool ok = true;
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int s = j % C::kStages;
                const uint32_t ph = (j / C::kStages) & 1;
                if (j >= C::kStages) ok = mbar_wait(&k_empty[s], ph ^ 1, ctl, kSiteKEmpty);
                if (!ok) break;
                mbar_arrive_expect_tx(&k_full[s], C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sK + s * C::kTileBytes + c * kBoxBytes, &tmK, &k_full[s], 64 * c,
                                j * kBlockN, bh, pol_kv);
                ++issued_k;
                if (j >= C::kStages) ok = mbar_wait(&v_empty[s], ph ^ 1, ctl, kSiteVEmpty);
                if (!ok) break;
                mbar_arrive_expect_tx(&v_full[s], C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sV + s * C::kTileBytes + c * kBoxBytes, &tmV, &v_full[s], 64 * c,
                                j * kBlockN, bh, pol_kv);
                ++issued_v;
            }
            // Drain: every load issued must land before the CTA exits.
            mbar_wait_drain(q_full, 0, p.limit_ns);
            for (int t = max(0, issued_k - C::kStages); t < issued_k; ++t)
                mbar_wait_drain(&k_full[t % C::kStages], (t / C::kStages) & 1, p.limit_ns);
            for (int t = max(0, issued_v - C::kStages); t < issued_v; ++t)
                mbar_wait_drain(&v_full[t % C::kStages], (t / C::kStages) & 1, p.limit_ns);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ============================ MMA issuer ============================
        if (lane == 0) {
            const uint32_t q_base = smem_u32(sQ);
            const uint32_t k_base = smem_u32(sK);
            const uint32_t v_base = smem_u32(sV);
            auto issue_S = [&](int k, int s) {
                const uint32_t d_tm = tmem + (k ? C::kTmS1 : C::kTmS0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                    const uint64_t a = sdesc_sw128(q_base + k * C::kChunks * kBoxBytes + off, 16, 1024);
                    const uint64_t b = sdesc_sw128(k_base + s * C::kTileBytes + off, 16, 1024);
                    mma_ss(d_tm, a, b, C::kIdescS, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_PV = [&](int k, int s, bool acc) {
                const uint32_t d_tm = tmem + (k ? C::kTmO1 : C::kTmO0);
                const uint32_t p_tm = tmem + (k ? C::kTmS1 : C::kTmS0);
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk) {
                    const uint64_t b = sdesc_sw128(v_base + s * C::kTileBytes + kk * 16 * 128,
                                                   kBoxBytes, 1024);
                    mma_ts(d_tm, p_tm + kk * 8, b, C::kIdescPV, (acc || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = mbar_wait(q_full, 0, ctl, kSiteQ);
            tc_fence_after();
            for (int j = 0; j <= n_tiles && ok; ++j) {
                const int s = j % C::kStages;
                if (j < n_tiles) {
                    ok = mbar_wait(&k_full[s], (j / C::kStages) & 1, ctl, kSiteKFull);
                    if (!ok) break;
                    tc_fence_after();
                }
                // S_0(j)
                if (j < n_sub0) {
                    issue_S(0, s);
                    mma_commit(&s_full[0]);
                }
                // PV_1(j-1)
                if (j >= 1 && j - 1 < n_sub1) {
                    const int jp = j - 1, sp = jp % C::kStages;
                    if (jp >= n_sub0) {  // V_{j-1} not yet waited for by PV_0
                        ok = mbar_wait(&v_full[sp], (jp / C::kStages) & 1, ctl, kSiteVFull);
                        if (!ok) break;
                    }
                    ok = mbar_wait(&p_full[1], jp & 1, ctl, kSitePFull);
                    if (!ok) break;
                    tc_fence_after();
                    issue_PV(1, sp, jp > 0);
                    mma_commit(&v_empty[sp]);
                }
                if (j < n_tiles) {
                    // S_1(j)
                    if (j < n_sub1) {
                        issue_S(1, s);
                        mma_commit(&s_full[1]);
                    }
                    mma_commit(&k_empty[s]);
                    // PV_0(j)
                    if (j < n_sub0) {
                        ok = mbar_wait(&v_full[s], (j / C::kStages) & 1, ctl, kSiteVFull);
                        if (!ok) break;
                        ok = mbar_wait(&p_full[0], j & 1, ctl, kSitePFull);
                        if (!ok) break;
                        tc_fence_after();
                        issue_PV(0, s, j > 0);
                    }
                }
            }
            // All MMAs (or, after an abort, all issued ones) complete before
            // o_full fires; the drain below makes the exit safe either way.
            mma_commit(o_full);
            mbar_wait_drain(o_full, 0, p.limit_ns);
        }
        __syncwarp();
    } else {
        // ======================= softmax (sub-tile k) =======================
        const int k = warp >> 2;  // warps 0-3 -> 0, 4-7 -> 1
        const int wq = warp & 3;  // TMEM lane quarter this warp may access
        const int row = wq * 32 + lane;
        const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tm_s = tmem + lane_bits + (k ? C::kTmS1 : C::kTmS0);
        const uint32_t tm_o = tmem + lane_bits + (k ? C::kTmO1 : C::kTmO0);
        const int sub_start = qb * kBlockM + k * kSubM;
        const int qrow = sub_start + row;
        const float cs = p.scale_log2;
        const int n_k = k ? n_sub1 : n_sub0;

        float m = -INFINITY;  // running max of s * scale * log2(e)
        float l = 0.f;        // running sum of 2^(s*c - m)
        bool ok = true;
        for (int j = 0; j < n_k; ++j) {
            ok = mbar_wait(&s_full[k], j & 1, ctl, kSiteSFull);
            if (!ok) break;
            tc_fence_after();
            uint32_t raw[128];
            tmem_ld128(tm_s, raw);
            float *sv = reinterpret_cast<float *>(raw);

            const int key0 = j * kBlockN;
            const bool ragged = key0 + kBlockN > N;
            const bool diag = CAUSAL && (key0 + kBlockN - 1 > sub_start);
            if (ragged || diag) {
                int lim = N - key0;
                if (CAUSAL) lim = min(lim, qrow - key0 + 1);
#pragma unroll
                for (int c = 0; c < kBlockN; ++c)
                    if (c >= lim) sv[c] = -INFINITY;
            }
            float mx = sv[0];
#pragma unroll
            for (int c = 1; c < kBlockN; ++c) mx = fmaxf(mx, sv[c]);
            const float m_new = fmaxf(m, mx * cs);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = (m == m_use) ? 1.f : ex2_approx(m - m_use);
            const float neg = -m_use;

            float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int c16 = 0; c16 < kBlockN / 32; ++c16) {
                uint32_t pk[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const float p0 = ex2_approx(fmaf(sv[32 * c16 + 2 * t], cs, neg));
                    const float p1 = ex2_approx(fmaf(sv[32 * c16 + 2 * t + 1], cs, neg));
                    rs0 += p0;
                    rs1 += p1;
                    pk[t] = pack_bf16x2(p0, p1);
                }
                tmem_st16(tm_s + 16 * c16, pk);
            }
            // rescale O_k when the max moved for some row of this warp; the
            // S_k(j) barrier also covered PV_k(j-1), so O_k is settled
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tm_o + 32 * c, o);
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
                    tmem_st32(tm_o + 32 * c, o);
                }
            }
            tmem_wait_st();
            l = l * alpha + (rs0 + rs1);
            m = m_new;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[k]);
        }

        // ---- epilogue: O = a / l (bf16), LSE = (m + log2 l) ln 2
        if (ok) ok = mbar_wait(o_full, 0, ctl, kSiteOFull);
        if (ok) {
            tc_fence_after();
            const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
            const bool in_range = qrow < N;
            __nv_bfloat16 *orow = p.O + (static_cast<size_t>(bh) * N + qrow) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tm_o + 32 * c, o);
                uint32_t pk[16];
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    pk[t] = pack_bf16x2(__uint_as_float(o[2 * t]) * inv_l,
                                        __uint_as_float(o[2 * t + 1]) * inv_l);
                if (in_range) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        dst[t] = make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
                }
            }
            if (in_range) {
                const float lse = (l > 0.f) ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
                p.LSE[static_cast<size_t>(bh) * N + qrow] = lse;
            }
        }
    }

    // ---- teardown: every role has drained its own asynchronous work
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
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

template <int D, bool CAUSAL>
static int launch_t(const LaunchArgs &a) {
    using C = Cfg<D>;
    auto kern = fa_fwd_kernel<D, CAUSAL>;
    static int configured_device = -1;  // attribute set once per process
    int dev = 0;
    FA_CUDA_TRY(cudaGetDevice(&dev));
    if (configured_device != dev) {
        FA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes));
        configured_device = dev;
    }
    Params p;
    p.O = static_cast<__nv_bfloat16 *>(a.O);
    p.LSE = a.LSE;
    p.N = a.N;
    p.n_qblocks = (a.N + kBlockM - 1) / kBlockM;
    p.n_ktiles = (a.N + kBlockN - 1) / kBlockN;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.limit_ns = a.limit_ns;
    const long long grid = static_cast<long long>(p.n_qblocks) * a.BH;
    if (grid > 0x7FFFFFFFLL) return FA_ERR_SHAPE;
    kern<<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, a.stream>>>(*a.tmQ, *a.tmK,
                                                                             *a.tmV, p);
    FA_CUDA_TRY(cudaGetLastError());
    return FA_OK;
}

int launch_fwd(const LaunchArgs &a) {
    if (a.d == 64) return a.causal ? launch_t<64, true>(a) : launch_t<64, false>(a);
    if (a.d == 128) return a.causal ? launch_t<128, true>(a) : launch_t<128, false>(a);
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
