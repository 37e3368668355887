// fa_decode_sm103.cu -- split-KV attention decoding for sm_103a (GB300).
//
// One new query row per (batch, query head) against a key/value cache of N
// positions: O = softmax(scale * q K^T) V and LSE.  With a single query row
// the FA-2 query-block parallelism collapses and the work is bound by
// reading K and V from HBM ("FlashAttention-2 -- Deeper Math",
// aicassindra.com, "What FA-2 does not fix": parallelise over keys and merge
// the partial softmaxes).  So:
//   * split kernel: one persistent CTA per SM streams an equal, contiguous
//     run of 128-key K/V tiles (of all (batch, K/V head) pairs in turn)
//     through a ring of shared-memory stages filled by TMA.  Eight warps
//     each take 16 keys of every tile and use each K and V row for every
//     query head of the group (grouped-query attention), keeping the online
//     state (m, l, a) per query head ("Understanding FlashAttention Pt 1",
//     wpnews.pro, section 2.4).  At a head boundary and at the end of the
//     run the warps merge their states and the CTA writes one state per
//     (query head, run) to the caller's workspace.
//   * merge kernel: one warp per (batch, query head) combines the runs'
//     states with the same merge rule -- m = max m_s, l = sum l_s 2^(m_s-m),
//     a = sum a_s 2^(m_s-m) -- and writes O = a / l (bf16) and LSE.
// The contraction is matrix-vector (a handful of query rows), so it runs on
// the CUDA cores, not the tensor cores: 16 lanes share one 256-byte key row
// (8 elements each, one 16-byte load), bf16 pairs are widened to fp32 pairs
// once and multiplied with packed fp32x2 FMAs, and a transposed butterfly of
// shuffles leaves each lane with the whole score of one query head.  Base-2
// exponentials with the scale folded in, as in the forward kernel; the
// reference max of a head moves only when a score passes it by more than
// 2^8 (as in the forward kernel), p is rounded to bf16 for the P.V products
// (as the tensor-core path does) and l sums the fp32 p.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fa_internal.h"
#include "sm103_primitives.cuh"
#include "debug_checks.cuh"

namespace fa {

constexpr int kDecWarps = 4;       // warps per CTA of the merge kernel
// keys per K/V tile of the split kernel: 128, or 64 at d = 256 (stage size)
template <int D>
constexpr int dec_tile_keys() { return D == 256 ? 64 : 128; }
constexpr int kDecConsumers = 8;   // consumer warps per split CTA
constexpr int kDecThreads = (kDecConsumers + 1) * 32;  // + one producer warp
constexpr int kDecMaxGrid = 1024;
// A head's reference max moves only when a score passes it by more than this
// (base-2 units), so p = 2^(s - m) <= 256 and the common path skips the
// per-head update.
constexpr float kDecStaleMax = 8.f;  // split CTAs at most (>= the SM count)

// A packed bf16 pair (low half = element 2i) widened to an fp32 pair, exactly:
// bf16 is the upper half of an fp32.  Two integer operations per pair, shared
// by every query head, then packed fp32x2 FMAs do two products at a time.
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t w) {
    return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint4 lds128(const uint8_t *p) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(smem_u32(p)));
    return r;
}

__device__ __forceinline__ uint32_t bf16_bits(float x) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

__device__ int g_fa_status_dec;  // bounded-wait timeouts of the decoding kernels

// ------------------------------------------------------------ work partition
// The K/V cache is cut into tiles of dec_tile_keys<D>() keys; the tiles of all
// (batch, K/V head) pairs form one sequence of T = heads * T_h tiles, and
// CTA c of `grid` takes the contiguous run [c*T/grid, (c+1)*T/grid).  Every
// CTA streams the same number of bytes (to one tile), and a run crosses at
// most a few head boundaries: the CTA writes one partial softmax state per
// (head, run) it touches, in slot (CTA - first CTA of the head) of the head.
__host__ __device__ __forceinline__ long long dec_run_begin(long long c, long long T, int grid) {
    return c * T / grid;
}
// The CTA whose run holds tile t.
__host__ __device__ __forceinline__ int dec_cta_of(long long t, long long T, int grid) {
    return static_cast<int>(((t + 1) * grid - 1) / T);
}
// Slots per head: a head's T_h tiles meet at most floor(grid / heads) + 2 runs.
__host__ __device__ __forceinline__ int dec_slots(int heads, int grid) {
    return grid / heads + 2;
}

template <int D, int G>
struct DecCfg {
    static constexpr int kLanesPerKey = D / 8;         // 16-byte chunks per row
    static constexpr int kKeysPerStep = 32 / kLanesPerKey;
    // A warp keeps the state of at most 4 query heads; for G = 8 the heads
    // split into kHeadGroups groups, each served by its own set of warps
    // that sees every key of the tile.
    static constexpr int kHeadsPerWarp = G < 4 ? G : 4;
    static constexpr int kHeadGroups = G / kHeadsPerWarp;
    static constexpr int kWarpsPerGroup = kDecConsumers / kHeadGroups;
    static constexpr int kTileKeys = dec_tile_keys<D>();
    static constexpr int kKeysPerWarp = kTileKeys / kWarpsPerGroup;  // per tile
    static constexpr int kSteps = kKeysPerWarp / kKeysPerStep;
    static constexpr int kTileBytes = kTileKeys * D * 2;  // one K or V tile
    static constexpr int kStages = (D == 64) ? 6 : 3;
    static constexpr int kOffRing = 0;                       // [S][K tile, V tile]
    static constexpr int kOffRed = kStages * 2 * kTileBytes;  // merge scratch
    static constexpr int kRedFloats = kDecConsumers * kHeadsPerWarp * (D + 2);
    static constexpr int kOffBar = kOffRed + kRedFloats * 4;
    // full[S], empty[S], the consumers' flush barrier; then the abort flag
    static constexpr int kSmemBytes = kOffBar + 8 * (2 * kStages + 1) + 16 + 128;
    static_assert(kKeysPerWarp % kKeysPerStep == 0, "tile split");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Split kernel: one persistent CTA per SM.  Warp kDecConsumers (one thread)
// streams the run's K and V tiles into a ring of shared-memory stages with
// TMA; the kDecConsumers consumer warps each take kKeysPerWarp keys of every
// tile (16-byte chunks, D/8 lanes per key) and keep the online-softmax state
// (m, l, a) of each of the G query heads of the tile's K/V head.  At a head
// boundary and at the end of the run the warps merge their states through
// shared memory and the CTA writes one state per query head.
template <int D, int G>
__global__ void __launch_bounds__(kDecThreads, 1)
    fa_decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV,
                           const __nv_bfloat16 *__restrict__ Q, float *__restrict__ part_ml,
                           float *__restrict__ part_acc, int H, int H_kv, int N, int n_heads,
                           int T_h, int stride, float scale_log2, uint64_t limit_ns) {
    using C = DecCfg<D, G>;
    constexpr int LPK = C::kLanesPerKey, KPS = C::kKeysPerStep, ST = C::kSteps;
    constexpr int SG = G >= 8 ? 2 : (ST < 4 ? ST : 4);  // steps per group (bounds the registers)
    constexpr int GW = C::kHeadsPerWarp, WPG = C::kWarpsPerGroup;
    constexpr int S = C::kStages;
    extern __shared__ __align__(128) uint8_t dsm_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(dsm_raw) + 127) & ~static_cast<uintptr_t>(127));
    float *red = reinterpret_cast<float *>(smem + C::kOffRed);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *empty = full + S;
    uint64_t *fbar = empty + S;  // consumer warps meet here (bounded, unlike bar.sync)
    volatile int *abort_flag = reinterpret_cast<volatile int *>(fbar + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kDecConsumers);
        }
        mbar_init(fbar, kDecConsumers);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    const WaitCtl ctl{abort_flag, &g_fa_status_dec, limit_ns};
    const long long T = static_cast<long long>(n_heads) * T_h;
    const int grid = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    const long long t0 = dec_run_begin(c, T, grid), t1 = dec_run_begin(c + 1, T, grid);

    if (warp == kDecConsumers) {
        // ---- producer
        if (lane != 0) return;
        const uint64_t pol = l2_policy_evict_first();
        int h = static_cast<int>(t0 / T_h), j = static_cast<int>(t0 - static_cast<long long>(h) * T_h);
        const int n_run = static_cast<int>(t1 - t0);
        int i = 0;
        bool ok = true;
        for (; i < n_run; ++i, ++j) {
            if (j == T_h) {
                j = 0;
                ++h;
            }
            const int s = i % S;
            if (i >= S) ok = mbar_wait(&empty[s], static_cast<uint32_t>((i / S) & 1) ^ 1u, ctl, 1);
            if (!ok) break;
            uint8_t *dst = smem + C::kOffRing + s * 2 * C::kTileBytes;
            if (!dbg_ok(h >= 0 && h < n_heads && j >= 0 && j < T_h, ctl, kChkTmaKV) ||
                !dbg_ok(in_smem_at(smem, dst, 2 * C::kTileBytes, C::kSmemBytes - 128), ctl,
                        kChkSmem)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(&full[s], 2 * C::kTileBytes);
            for (int r = 0; r < C::kTileKeys; r += 64) {  // 64-row boxes
                tma_load_3d(dst + r * D * 2, &tmK, &full[s], 0, j * C::kTileKeys + r, h, pol);
                tma_load_3d(dst + C::kTileBytes + r * D * 2, &tmV, &full[s], 0,
                            j * C::kTileKeys + r, h, pol);
            }
        }
        // every copy issued lands before the CTA exits (bounded)
        for (int k = (i > S ? i - S : 0); k < i; ++k)
            mbar_wait_drain(&full[k % S], static_cast<uint32_t>((k / S) & 1), limit_ns);
        return;
    }

    // ---- consumers
    const int cw = lane % LPK;  // this lane's 16-byte chunk of a row
    const int sub = lane / LPK;  // which key of a step this lane's group reads
    const int ctid = threadIdx.x;  // 0 .. kDecConsumers*32-1
    // After the transposed reduction (below) a lane holds the dot of head hl
    // of its key: round r sends the lower or upper half of the heads across
    // lane bit LPK >> (r+1).  head_lane(g) is the first lane holding head g.
    constexpr int KB = GW == 4 ? 2 : (GW == 2 ? 1 : 0);  // log2(GW)
    int hl = 0;
#pragma unroll
    for (int r = 0; r < KB; ++r)
        if (lane & (LPK >> (r + 1))) hl += GW >> (r + 1);
    const auto head_lane = [](int g) {
        int src = 0;
#pragma unroll
        for (int r = 0; r < KB; ++r)
            if (g & (GW >> (r + 1))) src += LPK >> (r + 1);
        return src;
    };
    const int key_base = lane & ~(LPK - 1);  // first lane of this lane's key
    const int hg = warp / WPG;      // this warp's head group
    const int wg = warp - hg * WPG;  // and its rank in the group
    uint64_t q2[GW][4];    // this lane's 8 query elements per head, fp32 pairs
    float m[GW];      // reference max per head (every lane)
    float m_own = 0.f;  // m of head hl
    float l_own = 0.f;  // sum of p of head hl over this lane's keys (fp32)
    uint64_t acc2[GW][4];  // this lane's 8 accumulator elements per head
    int cur = -1;  // head of the state being accumulated
    uint32_t fphase = 0;  // completed phases of fbar
    const auto meet = [&]() {  // all consumer warps; false on timeout or abort
        __syncwarp();
        if (lane == 0) mbar_arrive(fbar);
        const bool met = __all_sync(0xffffffffu, mbar_wait(fbar, fphase & 1u, ctl, 3));
        ++fphase;
        return met;
    };

    // merges the consumer warps' states for head `h` and writes them
    const auto flush = [&](int h) -> bool {
        // l of each head: the lanes of a key that hold head hl carry the
        // same sum, so add over the keys, then fetch it from a holder
        float lt = l_own;
#pragma unroll
        for (int off = LPK; off < 32; off <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
#pragma unroll
        for (int g = 0; g < GW; ++g) {
            const float lg = __shfl_sync(0xffffffffu, lt, head_lane(g));
            float acc[8];
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) f2_unpack(acc2[g][w4], acc[2 * w4], acc[2 * w4 + 1]);
#pragma unroll
            for (int off = LPK; off < 32; off <<= 1) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
            }
            if (sub == 0) {
                float *ra = red + (warp * GW + g) * (D + 2);
#pragma unroll
                for (int e = 0; e < 8; ++e) ra[cw * 8 + e] = acc[e];
                if (cw == 0) {
                    ra[D] = m[g];
                    ra[D + 1] = lg;
                }
            }
        }
        if (!meet()) return false;
        const long long hT = static_cast<long long>(h) * T_h;
        const int slot = c - dec_cta_of(hT, T, grid);
        if (!dbg_ok(h >= 0 && h < n_heads && slot >= 0 && slot < stride, ctl, kChkStoreO))
            return false;
        for (int q = ctid; q < G * D; q += kDecConsumers * 32) {
            const int g = q / D, dim = q - g * D;  // query head g of the group
            const int gw = g / GW, gl = g - gw * GW;  // its head group, index there
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < WPG; ++w)
                M = fmaxf(M, red[((gw * WPG + w) * GW + gl) * (D + 2) + D]);
            float a = 0.f, lsum = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < WPG; ++w) {
                    const float *ra = red + ((gw * WPG + w) * GW + gl) * (D + 2);
                    const float wt = ex2f(ra[D] - M);
                    a += wt * ra[dim];
                    lsum += wt * ra[D + 1];
                }
            }
            const size_t idx = (static_cast<size_t>(h) * stride + slot) * G + g;
            part_acc[idx * D + dim] = a;
            if (dim == 0) {
                part_ml[idx * 2] = M;
                part_ml[idx * 2 + 1] = lsum;
            }
        }
        return meet();  // the scratch is free again
    };

    // (head, tile in head) of the run's tiles, advanced without division
    int h = static_cast<int>(t0 / T_h), j = static_cast<int>(t0 - static_cast<long long>(h) * T_h);
    const int n_run = static_cast<int>(t1 - t0);
    bool ok = true;
    for (int i = 0; i < n_run; ++i, ++j) {
        if (j == T_h) {
            j = 0;
            ++h;
        }
        if (h != cur) {
            if (cur >= 0 && !flush(cur)) {
                ok = false;
                break;
            }
            cur = h;
            const int b = h / H_kv, kvh = h - b * H_kv;
            if (!dbg_ok(h < n_heads && kvh * G + hg * GW + GW <= H, ctl, kChkTmaQ)) {
                ok = false;
                break;
            }
#pragma unroll
            for (int g = 0; g < GW; ++g) {
                const uint4 qq = *reinterpret_cast<const uint4 *>(
                    Q + (static_cast<size_t>(b) * H + kvh * G + hg * GW + g) * D + cw * 8);
                q2[g][0] = bf16x2_to_f2(qq.x);
                q2[g][1] = bf16x2_to_f2(qq.y);
                q2[g][2] = bf16x2_to_f2(qq.z);
                q2[g][3] = bf16x2_to_f2(qq.w);
                m[g] = -INFINITY;
#pragma unroll
                for (int w4 = 0; w4 < 4; ++w4) acc2[g][w4] = 0ull;
            }
            m_own = -INFINITY;
            l_own = 0.f;
        }
        const int s = i % S;
        ok = __all_sync(0xffffffffu, mbar_wait(&full[s], static_cast<uint32_t>((i / S) & 1), ctl, 2));
        if (!ok) break;
        const uint8_t *kt_s = smem + C::kOffRing + s * 2 * C::kTileBytes;
        const uint8_t *vt_s = kt_s + C::kTileBytes;
        // the warp's keys in groups of SG steps (one step at a time for G = 8, to
        // bound the registers the scores and V chunks hold)
#pragma unroll
        for (int st0 = 0; st0 < ST; st0 += SG) {
            uint4 kt[SG], vt[SG];
            bool valid[SG];
#pragma unroll
            for (int st = 0; st < SG; ++st) {
                const int kk = wg * C::kKeysPerWarp + (st0 + st) * KPS + sub;  // key in tile
                valid[st] = j * C::kTileKeys + kk < N;
                kt[st] = lds128(kt_s + kk * (D * 2) + cw * 16);
                vt[st] = lds128(vt_s + kk * (D * 2) + cw * 16);
            }
            if (st0 + SG == ST) {  // this warp's last reads of the stage are issued
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            // Scores (base 2).  Each lane holds partial dots of the GW heads
            // over its 8 elements.  A transposed butterfly halves the heads
            // a lane carries each round, then plain rounds finish the sum:
            // every lane ends with the whole dot of head `hl` for its key,
            // after log2(LPK) + GW - 1 shuffles instead of GW log2(LPK).
            float sc[SG];  // score of (this lane's key, head hl)
#pragma unroll
            for (int st = 0; st < SG; ++st) {
                const uint64_t k2[4] = {bf16x2_to_f2(kt[st].x), bf16x2_to_f2(kt[st].y),
                                        bf16x2_to_f2(kt[st].z), bf16x2_to_f2(kt[st].w)};
                float dv[GW];
#pragma unroll
                for (int g = 0; g < GW; ++g) {
                    uint64_t d2 = f2_mul(k2[0], q2[g][0]);
#pragma unroll
                    for (int w4 = 1; w4 < 4; ++w4) d2 = f2_fma(k2[w4], q2[g][w4], d2);
                    float d0, d1;
                    f2_unpack(d2, d0, d1);
                    dv[g] = d0 + d1;
                }
#pragma unroll
                for (int r = 0; r < KB; ++r) {
                    const int half = GW >> (r + 1), off = LPK >> (r + 1);
                    const bool up = (lane & off) != 0;
#pragma unroll
                    for (int i = 0; i < half; ++i) {
                        const float send = up ? dv[i] : dv[i + half];
                        const float keep = up ? dv[i + half] : dv[i];
                        dv[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                    }
                }
#pragma unroll
                for (int off = LPK >> (KB + 1); off > 0; off >>= 1)
                    dv[0] += __shfl_xor_sync(0xffffffffu, dv[0], off);
                sc[st] = valid[st] ? dv[0] * scale_log2 : -INFINITY;
            }
            // tile max of head hl over this warp's keys; a head's reference
            // moves (rescaling its l and a by 2^(m - m')) only when the max
            // passes it by more than kDecStaleMax, which a vote detects
            float mt = sc[0];
#pragma unroll
            for (int st = 1; st < SG; ++st) mt = fmaxf(mt, sc[st]);
#pragma unroll
            for (int off = LPK; off < 32; off <<= 1)
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
            if (__any_sync(0xffffffffu, mt > m_own + kDecStaleMax)) {
#pragma unroll
                for (int g = 0; g < GW; ++g) {
                    const float mg = __shfl_sync(0xffffffffu, mt, head_lane(g));
                    if (mg > m[g] + kDecStaleMax) {  // warp-uniform
                        const float alpha = ex2f(m[g] - mg);  // m = -inf gives 0
                        const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
                        for (int w4 = 0; w4 < 4; ++w4) acc2[g][w4] = f2_mul(acc2[g][w4], a2);
                        if (hl == g) l_own *= alpha;
                        m[g] = mg;
                    }
                    if (hl == g) m_own = m[g];
                }
            }
            // p = 2^(s - m) for (key, head hl), l += p (fp32); every lane of
            // the key then fetches bf16(p) of each head: a += bf16(p) * V
#pragma unroll
            for (int st = 0; st < SG; ++st) {
                // a key past N has s = -inf; its p is forced to 0 (m may
                // still be -inf, and -inf - -inf is NaN)
                const float pown = valid[st] ? ex2f(sc[st] - m_own) : 0.f;
                l_own += pown;
                // P.V takes p rounded to bf16, as the tensor-core path does
                const float prown = __uint_as_float(bf16_bits(pown) << 16);
                const uint64_t v2[4] = {bf16x2_to_f2(vt[st].x), bf16x2_to_f2(vt[st].y),
                                        bf16x2_to_f2(vt[st].z), bf16x2_to_f2(vt[st].w)};
#pragma unroll
                for (int g = 0; g < GW; ++g) {
                    const float pr = __shfl_sync(0xffffffffu, prown, key_base + head_lane(g));
                    const uint64_t p2 = f2_pack(pr, pr);
#pragma unroll
                    for (int w4 = 0; w4 < 4; ++w4) acc2[g][w4] = f2_fma(v2[w4], p2, acc2[g][w4]);
                }
            }
        }
    }
    if (ok && cur >= 0) flush(cur);  // a failed flush has recorded its status
}

// Merge kernel: one warp per (batch, query head) combines the states of the
// runs that touched its K/V head: m = max m_s, l = sum l_s 2^(m_s - m),
// a = sum a_s 2^(m_s - m); O = a / l (bf16), LSE = (m + log2 l) ln 2.
template <int D, int G>
__global__ void __launch_bounds__(kDecWarps * 32)
    fa_decode_merge_kernel(const float *__restrict__ part_ml, const float *__restrict__ part_acc,
                           __nv_bfloat16 *__restrict__ O, float *__restrict__ LSE, int rows,
                           int H, int H_kv, int T_h, int grid, int stride) {
    constexpr int E = D / 32;  // output elements per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kDecWarps + warp;  // b * H + h
    if (row >= rows) return;
    const int b = row / H, h = row - b * H;
    const int kvh = h / G, g = h - kvh * G;
    const int bkv = b * H_kv + kvh;
    const long long T = static_cast<long long>(rows / H) * H_kv * T_h;
    const long long first = static_cast<long long>(bkv) * T_h;
    int n_slots = dec_cta_of(first + T_h - 1, T, grid) - dec_cta_of(first, T, grid) + 1;
    if (!dbg_ok_word(n_slots >= 1 && n_slots <= stride, &g_fa_status_dec, kChkItem)) n_slots = 0;
    const size_t base = static_cast<size_t>(bkv) * stride;
    float M = -INFINITY;
    for (int s = lane; s < n_slots; s += 32) M = fmaxf(M, part_ml[((base + s) * G + g) * 2]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float l = 0.f, o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < n_slots; ++s) {
            const size_t idx = (base + s) * G + g;
            const float w = ex2f(part_ml[idx * 2] - M);
            l += w * part_ml[idx * 2 + 1];
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] += w * part_acc[idx * D + lane * E + e];
        }
    }
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e)
        O[static_cast<size_t>(row) * D + lane * E + e] = __float2bfloat16_rn(o[e] * inv);
    if (lane == 0) LSE[row] = (l > 0.f) ? (M + log2f(l)) * 0.6931471805599453f : -INFINITY;
}

// ------------------------------------------------------------------ host side
// Partial states the workspace holds: every (batch, K/V head) gets the slots
// of the largest grid the kernels ever launch, so the size does not depend on
// the device.
size_t decode_state_count(int B, int H, int H_kv) {
    const int heads = B * H_kv;
    return static_cast<size_t>(heads) * dec_slots(heads, kDecMaxGrid) * (H / H_kv);
}

template <int D, int G>
static int launch_decode_t(const DecodeArgs &a) {
    using C = DecCfg<D, G>;
    auto kern = fa_decode_split_kernel<D, G>;
    static std::atomic<int> configured[kMaxDevices];
    int dev = 0;
    FA_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_ARCH;
    const int rc = set_smem_once(configured, dev, kern, C::kSmemBytes);
    if (rc != FA_OK) return rc;
    const int sms = device_sm_count(dev);
    if (sms <= 0) return record_message(FA_ERR_LAUNCH, "cannot query the SM count");
    const int heads = a.B * a.H_kv;
    const int T_h = (a.N + C::kTileKeys - 1) / C::kTileKeys;
    const long long T = static_cast<long long>(heads) * T_h;
    int grid = sms < kDecMaxGrid ? sms : kDecMaxGrid;
    if (T < grid) grid = static_cast<int>(T);
    const int stride = dec_slots(heads, grid);
    kern<<<grid, kDecThreads, C::kSmemBytes, a.stream>>>(
        *a.tmK, *a.tmV, static_cast<const __nv_bfloat16 *>(a.Q), a.part_ml, a.part_acc, a.H,
        a.H_kv, a.N, heads, T_h, stride, a.scale * 1.4426950408889634f, a.limit_ns);
    FA_CUDA_TRY(cudaGetLastError());
    const int rows = a.B * a.H;
    fa_decode_merge_kernel<D, G><<<(rows + kDecWarps - 1) / kDecWarps, kDecWarps * 32, 0,
                                   a.stream>>>(a.part_ml, a.part_acc,
                                               static_cast<__nv_bfloat16 *>(a.O), a.LSE, rows,
                                               a.H, a.H_kv, T_h, grid, stride);
    FA_CUDA_TRY(cudaGetLastError());
    return FA_OK;
}

template <int D>
static int launch_decode_d(const DecodeArgs &a) {
    switch (a.H / a.H_kv) {
        case 1: return launch_decode_t<D, 1>(a);
        case 2: return launch_decode_t<D, 2>(a);
        case 4: return launch_decode_t<D, 4>(a);
        case 8: return launch_decode_t<D, 8>(a);
        default: return FA_ERR_UNSUPPORTED;
    }
}

int launch_decode(const DecodeArgs &a) {
    if (a.d == 64) return launch_decode_d<64>(a);
    if (a.d == 256) return launch_decode_d<256>(a);
    if (a.d == 128) return launch_decode_d<128>(a);
    return FA_ERR_HEADDIM;
}

int dec_read_and_clear_status(int *status) {
    int v = 0;
    FA_CUDA_TRY(cudaMemcpyFromSymbol(&v, g_fa_status_dec, sizeof v));
    if (v != 0) {
        const int zero = 0;
        FA_CUDA_TRY(cudaMemcpyToSymbol(g_fa_status_dec, &zero, sizeof zero));
    }
    *status = v;
    return FA_OK;
}

}  // namespace fa

// ----------------------------------------------------- no-allocation decoding
// fa_decode_noalloc() runs the same two kernels as fa_decode() but keeps the
// split states in a fixed area of device memory that the library itself
// owns, so the caller never has to allocate.  That is for callers that
// cannot call cudaMalloc at the point where they decode: an allocation can
// block on, or synchronise with, work already queued on the device, it can
// fail once a host framework's memory pool has claimed the free memory, and
// some plugin hosts hand a component only the buffers of its inputs and
// outputs.
//
// The area is 16 MiB; every GPU that loads this library keeps it reserved
// until the process exits.  Requests whose states need more are rejected.
namespace fa {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(16) << 20;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

namespace {
// The device address of g_decode_scratch belongs to a CUDA context: a
// device reset, or another context made current on the same device, gives
// the module a new copy.  Each cached address is therefore kept with the
// unique id of the context it was looked up in (ids are never reused within
// a process), and looked up again when the current context differs.
struct ScratchAddr {
    unsigned long long ctx_id = 0;  // 0: none cached
    void *ptr = nullptr;
};
std::mutex g_scratch_mu;
ScratchAddr g_scratch_addr[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

template <class Fn>
Fn driver_fn(const char *name) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(p);
}

// Unique id of the current context; 0 if none is current or it cannot be
// read.
unsigned long long current_ctx_id() {
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}
}  // namespace

// Device address of g_decode_scratch in the current context.  In host code
// the symbol names a host-side stand-in, not device memory, so the address
// is asked for with the device current, once per context, and cached.
int decode_static_scratch(void **ptr, size_t *bytes) {
    int dev = 0;
    FA_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices)
        return record_message(FA_ERR_ARCH, "device ordinal out of range");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    unsigned long long id = current_ctx_id();
    ScratchAddr &e = g_scratch_addr[dev];
    if (id == 0 || e.ctx_id != id) {
        // the lookup also makes the runtime's context current if none was
        void *p = nullptr;
        FA_CUDA_TRY(cudaGetSymbolAddress(&p, g_decode_scratch));
        if (id == 0) id = current_ctx_id();
        e.ptr = p;
        e.ctx_id = id;  // 0 if the id cannot be read: looked up again next call
    }
    *ptr = e.ptr;
    *bytes = kNoAllocScratchBytes;
    return FA_OK;
}

}  // namespace fa
