// fa_decode_sm103.cu -- split-KV attention decoding for sm_103a (GB300).
//
// One new query row per (batch, query head) against a key/value cache of N
// positions: O = softmax(scale * q K^T) V and LSE.  With a single query row
// the FA-2 query-block parallelism collapses and the work is bound by
// reading K and V from HBM ("FlashAttention-2 -- Deeper Math",
// aicassindra.com, "What FA-2 does not fix": parallelise over keys and merge
// the partial softmaxes).  So:
//   * split kernel: one warp per (batch, K/V head, key split).  The warp
//     reads each K and V row of its split once and uses it for every query
//     head of the group (grouped-query attention), keeping the online state
//     (m, l, a) per query head ("Understanding FlashAttention Pt 1",
//     wpnews.pro, section 2.4), and writes (m, l, a) of the split to the
//     caller's workspace.
//   * merge kernel: one warp per (batch, query head) combines the splits'
//     states with the same merge rule -- m = max m_s, l = sum l_s 2^(m_s-m),
//     a = sum a_s 2^(m_s-m) -- and writes O = a / l (bf16) and LSE.
// The contraction is matrix-vector (a handful of query rows), so it runs on
// the CUDA cores, not the tensor cores: 16 lanes share one 256-byte key row
// (8 bf16 each, one 16-byte load), dot products use mixed-precision FMAs on
// the bf16 operands with fp32 accumulation, and shuffles sum the 16 lanes.
// Base-2 exponentials with the scale folded in, as in the forward kernel;
// p is rounded to bf16 for the P.V products (as the tensor-core path does)
// and l sums the fp32 p.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fa_internal.h"

namespace fa {

constexpr int kDecWarps = 4;  // warps per CTA (both kernels)

// d += a * b with a, b the low (HI = false) or high halves of packed bf16
// pairs, fp32 accumulation (sm_100+ mixed-precision FMA).
template <bool HI>
__device__ __forceinline__ void fma_bf16(float &d, uint32_t a, uint32_t b) {
    if (HI)
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"
            "mov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
            "fma.rn.f32.bf16 %0, a1, b1, %0;\n\t}"
            : "+f"(d)
            : "r"(a), "r"(b));
    else
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"
            "mov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
            "fma.rn.f32.bf16 %0, a0, b0, %0;\n\t}"
            : "+f"(d)
            : "r"(a), "r"(b));
}

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t bf16_bits(float x) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

template <int D, int G>
struct DecCfg {
    static constexpr int kLanesPerKey = D / 8;          // 16-byte chunks per row
    static constexpr int kKeysPerStep = 32 / kLanesPerKey;
    static constexpr int kSteps = (G <= 4) ? 8 : 4;     // register budget
    static constexpr int kTileKeys = kKeysPerStep * kSteps;
};

template <int D, int G>
__global__ void __launch_bounds__(kDecWarps * 32)
    fa_decode_split_kernel(const __nv_bfloat16 *__restrict__ Q,
                           const __nv_bfloat16 *__restrict__ K,
                           const __nv_bfloat16 *__restrict__ V, float *__restrict__ part_ml,
                           float *__restrict__ part_acc, int H, int H_kv, int N, int split_len,
                           int n_splits, float scale_log2) {
    using C = DecCfg<D, G>;
    constexpr int LPK = C::kLanesPerKey, KPS = C::kKeysPerStep, ST = C::kSteps;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x * kDecWarps + warp;
    if (split >= n_splits) return;
    const int bkv = blockIdx.y;  // b * H_kv + K/V head
    const int b = bkv / H_kv, kvh = bkv - b * H_kv;
    const int c = lane % LPK;    // this lane's 8-element chunk of a row
    const int sub = lane / LPK;  // which key of a step this lane's group reads

    // the group's query rows, chunk c (8 bf16 = 4 packed pairs per row)
    uint32_t qv[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const uint4 t = *reinterpret_cast<const uint4 *>(
            Q + (static_cast<size_t>(b) * H + kvh * G + g) * D + c * 8);
        qv[g][0] = t.x;
        qv[g][1] = t.y;
        qv[g][2] = t.z;
        qv[g][3] = t.w;
    }
    const __nv_bfloat16 *Kh = K + static_cast<size_t>(bkv) * N * D + c * 8;
    const __nv_bfloat16 *Vh = V + static_cast<size_t>(bkv) * N * D + c * 8;
    const int key_begin = split * split_len;
    const int key_end = min(key_begin + split_len, N);

    float m[G], l[G], acc[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
    }

    for (int k0 = key_begin; k0 < key_end; k0 += C::kTileKeys) {
        uint4 kt[ST], vt[ST];
        bool valid[ST];
#pragma unroll
        for (int st = 0; st < ST; ++st) {
            const int key = k0 + st * KPS + sub;
            valid[st] = key < key_end;
            const int kk = valid[st] ? key : key_begin;  // in-bounds address either way
            kt[st] = ldg_stream(Kh + static_cast<size_t>(kk) * D);
            vt[st] = ldg_stream(Vh + static_cast<size_t>(kk) * D);
        }
        // scores (base 2): the LPK lanes of a key each hold a partial dot
        float s[ST][G];
#pragma unroll
        for (int st = 0; st < ST; ++st) {
            const uint32_t kw[4] = {kt[st].x, kt[st].y, kt[st].z, kt[st].w};
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float dot = 0.f;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    fma_bf16<false>(dot, kw[w], qv[g][w]);
                    fma_bf16<true>(dot, kw[w], qv[g][w]);
                }
#pragma unroll
                for (int off = LPK / 2; off > 0; off >>= 1)
                    dot += __shfl_xor_sync(0xffffffffu, dot, off);
                s[st][g] = valid[st] ? dot * scale_log2 : -INFINITY;
            }
        }
        // tile max per query row over the warp's keys, then the reference
        // update: rescale (l, a) by 2^(m - m') when the max moves
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float mt = s[0][g];
#pragma unroll
            for (int st = 1; st < ST; ++st) mt = fmaxf(mt, s[st][g]);
#pragma unroll
            for (int off = LPK; off < 32; off <<= 1)
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
            if (mt > m[g]) {  // warp-uniform: every lane holds the same values
                const float alpha = ex2f(m[g] - mt);  // m = -inf gives 0
                l[g] *= alpha;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[g][e] *= alpha;
                m[g] = mt;
            }
        }
        // p = 2^(s - m); l += p (fp32); a += bf16(p) * V
#pragma unroll
        for (int st = 0; st < ST; ++st) {
            const uint32_t vw[4] = {vt[st].x, vt[st].y, vt[st].z, vt[st].w};
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float p = ex2f(s[st][g] - m[g]);
                l[g] += p;
                const uint32_t pb = bf16_bits(p);
                const uint32_t pp = pb | (pb << 16);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    fma_bf16<false>(acc[g][2 * w], vw[w], pp);
                    fma_bf16<true>(acc[g][2 * w + 1], vw[w], pp);
                }
            }
        }
    }
    // Lanes with the same chunk c hold different keys: sum them.  (m is
    // already the same on every lane; each of the LPK lanes of a key added
    // that key's p to l once, so l needs only the cross-key sum.)
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int off = LPK; off < 32; off <<= 1) {
            l[g] += __shfl_xor_sync(0xffffffffu, l[g], off);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], off);
        }
    }
    if (sub == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const size_t idx = (static_cast<size_t>(bkv) * n_splits + split) * G + g;
            float4 *dst = reinterpret_cast<float4 *>(part_acc + idx * D + c * 8);
            dst[0] = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
            dst[1] = make_float4(acc[g][4], acc[g][5], acc[g][6], acc[g][7]);
            if (c == 0) {
                part_ml[idx * 2] = m[g];
                part_ml[idx * 2 + 1] = l[g];
            }
        }
    }
}

template <int D, int G>
__global__ void __launch_bounds__(kDecWarps * 32)
    fa_decode_merge_kernel(const float *__restrict__ part_ml, const float *__restrict__ part_acc,
                           __nv_bfloat16 *__restrict__ O, float *__restrict__ LSE, int rows,
                           int H, int H_kv, int n_splits) {
    constexpr int E = D / 32;  // output elements per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kDecWarps + warp;  // b * H + h
    if (row >= rows) return;
    const int b = row / H, h = row - b * H;
    const int kvh = h / G, g = h - kvh * G;
    const size_t base = (static_cast<size_t>(b) * H_kv + kvh) * n_splits;
    float M = -INFINITY;
    for (int s = lane; s < n_splits; s += 32) M = fmaxf(M, part_ml[((base + s) * G + g) * 2]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float l = 0.f, o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;
    for (int s = 0; s < n_splits; ++s) {
        const size_t idx = (base + s) * G + g;
        const float w = ex2f(part_ml[idx * 2] - M);
        l += w * part_ml[idx * 2 + 1];
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] += w * part_acc[idx * D + lane * E + e];
    }
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e)
        O[static_cast<size_t>(row) * D + lane * E + e] = __float2bfloat16_rn(o[e] * inv);
    if (lane == 0) LSE[row] = (l > 0.f) ? (M + log2f(l)) * 0.6931471805599453f : -INFINITY;
}

// ------------------------------------------------------------------ host side
// Key-split length: enough warps to fill the GPU with loads in flight
// (about 2432 = 16 per SM on 152 SMs), in multiples of 64 keys.
int decode_split_len(int B, int H_kv, int N) {
    const long long work = static_cast<long long>(N) * B * H_kv;
    long long len = (work + 2432LL * 64 - 1) / (2432LL * 64) * 64;
    if (len < 64) len = 64;
    if (len > N) len = ((N + 63) / 64) * 64;
    return static_cast<int>(len);
}

int decode_n_splits(int B, int H_kv, int N) {
    const int len = decode_split_len(B, H_kv, N);
    return (N + len - 1) / len;
}

template <int D, int G>
static int launch_decode_t(const DecodeArgs &a) {
    const int len = decode_split_len(a.B, a.H_kv, a.N);
    const int ns = (a.N + len - 1) / len;
    const dim3 grid1((ns + kDecWarps - 1) / kDecWarps, a.B * a.H_kv);
    fa_decode_split_kernel<D, G><<<grid1, kDecWarps * 32, 0, a.stream>>>(
        static_cast<const __nv_bfloat16 *>(a.Q), static_cast<const __nv_bfloat16 *>(a.K),
        static_cast<const __nv_bfloat16 *>(a.V), a.part_ml, a.part_acc, a.H, a.H_kv, a.N, len,
        ns, a.scale * 1.4426950408889634f);
    FA_CUDA_TRY(cudaGetLastError());
    const int rows = a.B * a.H;
    fa_decode_merge_kernel<D, G><<<(rows + kDecWarps - 1) / kDecWarps, kDecWarps * 32, 0,
                                   a.stream>>>(a.part_ml, a.part_acc,
                                               static_cast<__nv_bfloat16 *>(a.O), a.LSE, rows,
                                               a.H, a.H_kv, ns);
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
    if (a.d == 128) return launch_decode_d<128>(a);
    return FA_ERR_HEADDIM;
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
std::mutex g_scratch_mu;
void *g_scratch_addr[64] = {nullptr};
}  // namespace

// Device address of g_decode_scratch on the current device.  In host code
// the symbol names a host-side stand-in, not device memory, so the address
// is asked for once per device, with that device current, and cached.
int decode_static_scratch(void **ptr, size_t *bytes) {
    int dev = 0;
    FA_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return record_message(FA_ERR_ARCH, "device ordinal out of range");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        FA_CUDA_TRY(cudaGetSymbolAddress(&p, g_decode_scratch));
        g_scratch_addr[dev] = p;
    }
    *ptr = g_scratch_addr[dev];
    *bytes = kNoAllocScratchBytes;
    return FA_OK;
}

}  // namespace fa
