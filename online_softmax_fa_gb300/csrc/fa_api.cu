// fa_api.cu -- the C ABI declared in include/fa.h: argument checks, the
// device-architecture check, TMA tensor-map encoding, and the host-buffer
// wrapper.  Every check runs on the host before the first CUDA call, so a
// rejected request enqueues nothing.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <cstdio>
#include <mutex>

#include "fa_internal.h"
#include "host_pipe.h"

namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per in-kernel wait
using fa::kMaxDevices;

std::atomic<int> g_arch_ok[kMaxDevices];  // 0 unknown, 1 sm_103, -1 other

int check_arch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_ARCH;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_ARCH;
    int state = g_arch_ok[dev].load(std::memory_order_relaxed);
    if (state == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) !=
                cudaSuccess)
            return FA_ERR_ARCH;
        state = (major == 10 && minor == 3) ? 1 : -1;
        g_arch_ok[dev].store(state, std::memory_order_relaxed);
    }
    return state == 1 ? FA_OK : FA_ERR_ARCH;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [B*H, N, d] bf16 viewed as a 3-D tensor (d innermost).  Box = 64 columns
// (128 bytes, the 128-byte swizzle span) x 128 rows x 1 head.  Rows past N
// inside a head read as zero, so a ragged tail never touches the next head.
bool encode_qkv_map(CUtensorMap *m, const void *base, int BH, int N, int d, int rows = 128) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                   static_cast<cuuint64_t>(N) * d * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K/V cache [B*H_kv, N, d] bf16 for decoding: box = all d columns x 64 rows
// x 1 head, no swizzle (rows land contiguously in shared memory), rows past N
// read as zero.
bool encode_cache_map(CUtensorMap *m, const void *base, int BH, int N, int d) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                   static_cast<cuuint64_t>(N) * d * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(d), 64, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Shape and scalar checks shared by the forward and backward entry points.
int check_shape(int B, int H, int N, int d, float scale) {
    if (B < 1 || H < 1 || N < 1) return FA_ERR_SHAPE;
    if (d != 64 && d != 128 && d != 256) return FA_ERR_HEADDIM;
    if (static_cast<long long>(B) * H > 0x7FFFFFFFLL) return FA_ERR_SHAPE;
    const long long qblocks = (static_cast<long long>(N) + 255) / 256;
    if (qblocks * B * H > 0x7FFFFFFFLL) return FA_ERR_SHAPE;  // grid size
    if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_SCALE;
    return FA_OK;
}

thread_local char g_detail[256] = "";
thread_local int g_last_status = 0;  // raw status behind the last fa_device_error

}  // namespace

namespace fa {
int device_sm_count(int dev) {
    static std::atomic<int> counts[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices) return 0;
    int n = counts[dev].load(std::memory_order_acquire);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        counts[dev].store(n, std::memory_order_release);
    }
    return n;
}

int record_cuda_error(cudaError_t e, const char *what) {
    std::snprintf(g_detail, sizeof g_detail, "%s: %s (%s)", what, cudaGetErrorName(e),
                  cudaGetErrorString(e));
    return FA_ERR_LAUNCH;
}
int record_message(int status, const char *what) {
    std::snprintf(g_detail, sizeof g_detail, "%s", what);
    return status;
}
}  // namespace fa

extern "C" {

int fa_fwd_gqa(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
               int H, int H_kv, int N, int d, int causal, float scale, fa_stream_t stream) {
    if (!Q || !K || !V || !O || !LSE) return FA_ERR_NULL;
    int rc = check_shape(B, H, N, d, scale);
    if (rc != FA_OK) return rc;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_SHAPE;
    const auto mis16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (mis16(Q) || mis16(K) || mis16(V) || mis16(O) ||
        (reinterpret_cast<uintptr_t>(LSE) & 3u) != 0)
        return FA_ERR_ALIGN;
    const size_t q_bytes = static_cast<size_t>(B) * H * N * d * 2;
    const size_t kv_bytes = static_cast<size_t>(B) * H_kv * N * d * 2;
    const size_t l_bytes = static_cast<size_t>(B) * H * N * 4;
    if (overlaps(O, q_bytes, Q, q_bytes) || overlaps(LSE, l_bytes, Q, q_bytes)) return FA_ERR_ALIAS;
    for (const void *in : {K, V})
        if (overlaps(O, q_bytes, in, kv_bytes) || overlaps(LSE, l_bytes, in, kv_bytes))
            return FA_ERR_ALIAS;
    if (overlaps(O, q_bytes, LSE, l_bytes)) return FA_ERR_ALIAS;

    rc = check_arch();
    if (rc != FA_OK) return rc;
    CUtensorMap tmQ, tmK, tmV, tmV64;
    if (!encode_qkv_map(&tmQ, Q, B * H, N, d) || !encode_qkv_map(&tmK, K, B * H_kv, N, d) ||
        !encode_qkv_map(&tmV, V, B * H_kv, N, d) ||
        (d == 256 && !encode_qkv_map(&tmV64, V, B * H_kv, N, d, 64)))
        return fa::record_message(FA_ERR_LAUNCH, "cuTensorMapEncodeTiled failed");
    fa::LaunchArgs a;
    a.tmQ = &tmQ;
    a.tmK = &tmK;
    a.tmV = &tmV;
    a.tmV64 = d == 256 ? &tmV64 : nullptr;
    a.O = O;
    a.LSE = LSE;
    a.BH = B * H;
    a.N = N;
    a.d = d;
    a.H = H;
    a.Hkv = H_kv;
    a.causal = causal != 0;
    a.scale = scale;
    a.limit_ns = kWaitLimitNs;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    return fa::launch_fwd(a);
}

int fa_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
           int N, int d, int causal, float scale, fa_stream_t stream) {
    return fa_fwd_gqa(Q, K, V, O, LSE, B, H, H, N, d, causal, scale, stream);
}

size_t fa_fwd_host_gqa_workspace_bytes(int B, int H, int H_kv, int N, int d) {
    if (check_shape(B, H, N, d, 1.f) != FA_OK) return 0;
    if (H_kv < 1 || H % H_kv != 0) return 0;
    const size_t q_bytes = static_cast<size_t>(B) * H * N * d * 2;
    const size_t kv_bytes = static_cast<size_t>(B) * H_kv * N * d * 2;
    const size_t l_bytes = static_cast<size_t>(B) * H * N * 4;
    return 2 * align256(q_bytes) + 2 * align256(kv_bytes) + align256(l_bytes);
}

size_t fa_fwd_host_workspace_bytes(int B, int H, int N, int d) {
    return fa_fwd_host_gqa_workspace_bytes(B, H, H, N, d);
}

namespace {
// Streams and events of the host-buffer path, created once per device and
// kept for the life of the process; `mu` serialises the enqueueing of calls
// that share them.
struct HostPipe {
    static constexpr int kMaxChunks = 16;
    std::mutex mu;
    bool ready = false;
    cudaStream_t in = nullptr, comp[2] = {nullptr, nullptr}, out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t loaded[kMaxChunks] = {}, computed[kMaxChunks] = {};
};
HostPipe g_pipes[kMaxDevices];

// Creates the device's streams and events on first use; call with h.mu held.
int host_pipe_init(HostPipe &h) {
    if (h.ready) return FA_OK;
    const unsigned fl = cudaStreamNonBlocking;
    FA_CUDA_TRY(cudaStreamCreateWithFlags(&h.in, fl));
    FA_CUDA_TRY(cudaStreamCreateWithFlags(&h.comp[0], fl));
    FA_CUDA_TRY(cudaStreamCreateWithFlags(&h.comp[1], fl));
    FA_CUDA_TRY(cudaStreamCreateWithFlags(&h.out, fl));
    FA_CUDA_TRY(cudaEventCreateWithFlags(&h.start, cudaEventDisableTiming));
    FA_CUDA_TRY(cudaEventCreateWithFlags(&h.done, cudaEventDisableTiming));
    for (int c = 0; c < HostPipe::kMaxChunks; ++c) {
        FA_CUDA_TRY(cudaEventCreateWithFlags(&h.loaded[c], cudaEventDisableTiming));
        FA_CUDA_TRY(cudaEventCreateWithFlags(&h.computed[c], cudaEventDisableTiming));
    }
    h.ready = true;
    return FA_OK;
}

// Chunk boundaries (in heads) for the host-buffer pipeline: chunks of
// `size` heads, except that the last chunks shrink by halves down to one
// head (..., 4, 2, 1, 1), so that little work waits for the last copy-in
// and little output for the last kernel.  Falls back to equal chunks when
// that would take more than kMaxChunks.  Returns the chunk count; chunk c
// covers heads [bounds[c], bounds[c + 1]).
int plan_chunks(long long BH, long long equal_chunks, long long *bounds) {
    const long long size = (BH + equal_chunks - 1) / equal_chunks;
    long long tail[HostPipe::kMaxChunks];
    int nt = 0;
    long long used = 0;
    for (long long sz = 1; sz < size && used + sz <= BH && nt < HostPipe::kMaxChunks; sz *= 2) {
        tail[nt++] = sz;
        used += sz;
        if (sz == 1 && used + 1 <= BH && nt < HostPipe::kMaxChunks) {  // two chunks of one head
            tail[nt++] = 1;
            used += 1;
        }
    }
    const long long full = (BH - used + size - 1) / size;
    if (size <= 1 || full + nt > HostPipe::kMaxChunks) {  // equal chunks
        for (long long c = 0; c <= equal_chunks; ++c) bounds[c] = c * BH / equal_chunks;
        return static_cast<int>(equal_chunks);
    }
    int n = 0;
    bounds[0] = 0;
    // the first chunk takes the remainder, the others `size` heads each
    long long h = BH - used - (full - 1) * size;
    for (long long c = 0; c < full; ++c) {
        bounds[n + 1] = bounds[n] + (c == 0 ? h : size);
        ++n;
    }
    for (int i = nt - 1; i >= 0; --i) {
        bounds[n + 1] = bounds[n] + tail[i];
        ++n;
    }
    return n;
}
}  // namespace

int fa_fwd_host_gqa(const void *Q_host, const void *K_host, const void *V_host,
                    void *O_host, float *LSE_host, void *workspace, size_t workspace_bytes,
                    int B, int H, int H_kv, int N, int d, int causal, float scale,
                    fa_stream_t stream) {
    if (!Q_host || !K_host || !V_host || !O_host || !LSE_host) return FA_ERR_NULL;
    int rc = check_shape(B, H, N, d, scale);
    if (rc != FA_OK) return rc;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_SHAPE;
    const size_t need = fa_fwd_host_gqa_workspace_bytes(B, H, H_kv, N, d);
    if (!workspace || workspace_bytes < need ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return FA_ERR_WORKSPACE;
    rc = check_arch();
    if (rc != FA_OK) return rc;
    const size_t q_bytes = static_cast<size_t>(B) * H * N * d * 2;
    const size_t kv_bytes = static_cast<size_t>(B) * H_kv * N * d * 2;
    uint8_t *w = static_cast<uint8_t *>(workspace);
    uint8_t *dQ = w, *dO = dQ + align256(q_bytes), *dK = dO + align256(q_bytes);
    uint8_t *dV = dK + align256(kv_bytes);
    float *dL = reinterpret_cast<float *>(dV + align256(kv_bytes));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int G = H / H_kv;  // query heads per K/V head

    // The heads are independent, so the work is cut into chunks of heads:
    // the copy-in of chunk c+1, the kernel on chunk c and the copy-out of
    // chunk c-1 overlap (one copy-in stream, two kernel streams taken in
    // turn, one copy-out stream).  Most chunks keep at least about one query
    // block per SM, so the kernel stays reasonably efficient while the
    // copies (the longer part) hide it; the last chunks shrink (plan_chunks)
    // and their kernels overlap each other on the two kernel streams.  The
    // results are those of one fa_fwd call (each head is computed the same
    // way).
    int dev = 0;
    FA_CUDA_TRY(cudaGetDevice(&dev));
    int sms = 0;
    FA_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    // chunks are whole groups of query heads sharing a K/V head (bounds in
    // K/V heads; a flattened query head x uses flattened K/V head x / G)
    const long long BH = static_cast<long long>(B) * H, BHkv = BH / G;
    const long long rows_per_item = d == 256 ? 128 : 256;
    const long long qblocks = (static_cast<long long>(N) + rows_per_item - 1) / rows_per_item;
    long long equal = BH * qblocks / (sms > 0 ? sms : 1);
    if (equal > 8) equal = 8;
    if (equal > BHkv) equal = BHkv;
    if (equal < 1) equal = 1;
    long long bounds[HostPipe::kMaxChunks + 1];
    const int chunks = plan_chunks(BHkv, equal, bounds);
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_ARCH;
    HostPipe *hp = &g_pipes[dev];
    std::lock_guard<std::mutex> lock(hp->mu);
    rc = host_pipe_init(*hp);
    if (rc != FA_OK) return rc;
    const size_t head_t = static_cast<size_t>(N) * d * 2, head_l = static_cast<size_t>(N) * 4;
    // The stream operations of the pipeline (host_pipe.h holds its order).
    // Chunk c covers K/V heads [bounds[c], bounds[c+1]) and their query
    // heads [G bounds[c], G bounds[c+1]).
    struct Ops {
        HostPipe *hp;
        cudaStream_t caller;
        const long long *bounds;
        long long G;
        size_t head_t, head_l;
        const uint8_t *Qh, *Kh, *Vh;
        uint8_t *Oh, *Lh, *dQ, *dK, *dV, *dO, *dL;
        int N, d, causal;
        float scale;
        cudaStream_t stream(fa::pipe::Stream s) const {
            switch (s) {
                case fa::pipe::kIn: return hp->in;
                case fa::pipe::kComp0: return hp->comp[0];
                case fa::pipe::kComp1: return hp->comp[1];
                case fa::pipe::kOut: return hp->out;
                default: return caller;
            }
        }
        cudaEvent_t event(fa::pipe::Event e) const {
            switch (e.kind) {
                case fa::pipe::kStart: return hp->start;
                case fa::pipe::kLoaded: return hp->loaded[e.chunk];
                case fa::pipe::kComputed: return hp->computed[e.chunk];
                default: return hp->done;
            }
        }
        int record(fa::pipe::Event e, fa::pipe::Stream s) {
            FA_CUDA_TRY(cudaEventRecord(event(e), stream(s)));
            return FA_OK;
        }
        int wait(fa::pipe::Stream s, fa::pipe::Event e) {
            FA_CUDA_TRY(cudaStreamWaitEvent(stream(s), event(e), 0));
            return FA_OK;
        }
        int copy_in(int c) {
            const size_t kv_off = bounds[c] * head_t, kv_n = (bounds[c + 1] - bounds[c]) * head_t;
            FA_CUDA_TRY(cudaMemcpyAsync(dQ + G * kv_off, Qh + G * kv_off, G * kv_n,
                                        cudaMemcpyHostToDevice, hp->in));
            FA_CUDA_TRY(cudaMemcpyAsync(dK + kv_off, Kh + kv_off, kv_n, cudaMemcpyHostToDevice,
                                        hp->in));
            FA_CUDA_TRY(cudaMemcpyAsync(dV + kv_off, Vh + kv_off, kv_n, cudaMemcpyHostToDevice,
                                        hp->in));
            return FA_OK;
        }
        int launch(int c, fa::pipe::Stream s) {
            // one batch of the chunk's heads (B = 1): query head i of the
            // chunk uses its K/V head i / G, as in the whole problem
            const long long hkv = bounds[c + 1] - bounds[c];
            const size_t kv_off = bounds[c] * head_t, l_off = G * bounds[c] * head_l;
            return fa_fwd_gqa(dQ + G * kv_off, dK + kv_off, dV + kv_off, dO + G * kv_off,
                              reinterpret_cast<float *>(dL + l_off), 1,
                              static_cast<int>(G * hkv), static_cast<int>(hkv), N, d, causal,
                              scale, reinterpret_cast<fa_stream_t>(stream(s)));
        }
        int copy_out(int c) {
            const long long hq = G * (bounds[c + 1] - bounds[c]);
            const size_t q_off = G * bounds[c] * head_t, l_off = G * bounds[c] * head_l;
            FA_CUDA_TRY(cudaMemcpyAsync(Oh + q_off, dO + q_off, hq * head_t,
                                        cudaMemcpyDeviceToHost, hp->out));
            FA_CUDA_TRY(cudaMemcpyAsync(Lh + l_off, dL + l_off, hq * head_l,
                                        cudaMemcpyDeviceToHost, hp->out));
            return FA_OK;
        }
    } ops{hp, s, bounds, G, head_t, head_l,
          static_cast<const uint8_t *>(Q_host), static_cast<const uint8_t *>(K_host),
          static_cast<const uint8_t *>(V_host), static_cast<uint8_t *>(O_host),
          reinterpret_cast<uint8_t *>(LSE_host), dQ, dK, dV, dO,
          reinterpret_cast<uint8_t *>(dL), N, d, causal, scale};
    return fa::pipe::run(ops, chunks);
}

int fa_fwd_host(const void *Q_host, const void *K_host, const void *V_host, void *O_host,
                float *LSE_host, void *workspace, size_t workspace_bytes, int B, int H, int N,
                int d, int causal, float scale, fa_stream_t stream) {
    return fa_fwd_host_gqa(Q_host, K_host, V_host, O_host, LSE_host, workspace,
                           workspace_bytes, B, H, H, N, d, causal, scale, stream);
}

// ----------------------------------------------------------- decoding
namespace {
int check_decode_shape(int B, int H, int H_kv, int N, int d, float scale) {
    if (B < 1 || H < 1 || H_kv < 1 || N < 1) return FA_ERR_SHAPE;
    if (d != 64 && d != 128 && d != 256) return FA_ERR_HEADDIM;
    if (H % H_kv != 0) return FA_ERR_SHAPE;
    const int G = H / H_kv;
    if (G != 1 && G != 2 && G != 4 && G != 8) return FA_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * H_kv > 65535) return FA_ERR_SHAPE;  // bounds the tile arithmetic
    if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_SCALE;
    return FA_OK;
}

// workspace layout: partial accumulators, then partial (m, l) pairs
void decode_layout(int B, int H, int H_kv, int N, int d, size_t *acc_bytes, size_t *ml_bytes) {
    (void)N;  // the state count depends on the heads only
    const size_t states = fa::decode_state_count(B, H, H_kv);
    *acc_bytes = align256(states * d * sizeof(float));
    *ml_bytes = align256(states * 2 * sizeof(float));
}
}  // namespace

size_t fa_decode_workspace_bytes(int B, int H, int H_kv, int N, int d) {
    if (check_decode_shape(B, H, H_kv, N, d, 1.f) != FA_OK) return 0;
    size_t a = 0, m = 0;
    decode_layout(B, H, H_kv, N, d, &a, &m);
    return a + m;
}

int fa_decode(const void *Q, const void *K, const void *V, void *O, float *LSE,
              void *workspace, size_t workspace_bytes, int B, int H, int H_kv, int N, int d,
              float scale, fa_stream_t stream) {
    if (!Q || !K || !V || !O || !LSE) return FA_ERR_NULL;
    int rc = check_decode_shape(B, H, H_kv, N, d, scale);
    if (rc != FA_OK) return rc;
    const auto mis16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (mis16(Q) || mis16(K) || mis16(V) || mis16(O) ||
        (reinterpret_cast<uintptr_t>(LSE) & 3u) != 0)
        return FA_ERR_ALIGN;
    size_t acc_bytes = 0, ml_bytes = 0;
    decode_layout(B, H, H_kv, N, d, &acc_bytes, &ml_bytes);
    if (!workspace || workspace_bytes < acc_bytes + ml_bytes ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return FA_ERR_WORKSPACE;
    const size_t q_bytes = static_cast<size_t>(B) * H * d * 2;
    const size_t kv_bytes = static_cast<size_t>(B) * H_kv * N * d * 2;
    const size_t l_bytes = static_cast<size_t>(B) * H * 4;
    const size_t w_bytes = acc_bytes + ml_bytes;
    const struct { const void *p; size_t n; } ins[] = {{Q, q_bytes}, {K, kv_bytes},
                                                       {V, kv_bytes}};
    for (const auto &in : ins)
        if (overlaps(O, q_bytes, in.p, in.n) || overlaps(LSE, l_bytes, in.p, in.n) ||
            overlaps(workspace, w_bytes, in.p, in.n))
            return FA_ERR_ALIAS;
    if (overlaps(O, q_bytes, LSE, l_bytes) || overlaps(O, q_bytes, workspace, w_bytes) ||
        overlaps(LSE, l_bytes, workspace, w_bytes))
        return FA_ERR_ALIAS;
    rc = check_arch();
    if (rc != FA_OK) return rc;
    CUtensorMap tmK, tmV;
    if (!encode_cache_map(&tmK, K, B * H_kv, N, d) || !encode_cache_map(&tmV, V, B * H_kv, N, d))
        return fa::record_message(FA_ERR_LAUNCH, "cuTensorMapEncodeTiled failed for K/V");
    fa::DecodeArgs a;
    a.tmK = &tmK;
    a.tmV = &tmV;
    a.Q = Q;
    a.O = O;
    a.LSE = LSE;
    a.part_acc = static_cast<float *>(workspace);
    a.part_ml = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + acc_bytes);
    a.B = B;
    a.H = H;
    a.H_kv = H_kv;
    a.N = N;
    a.d = d;
    a.scale = scale;
    a.limit_ns = kWaitLimitNs;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    return fa::launch_decode(a);
}

int fa_decode_noalloc(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                      int H, int H_kv, int N, int d, float scale, fa_stream_t stream) {
    if (!Q || !K || !V || !O || !LSE) return FA_ERR_NULL;
    int rc = check_decode_shape(B, H, H_kv, N, d, scale);
    if (rc != FA_OK) return rc;
    rc = check_arch();
    if (rc != FA_OK) return rc;
    // the area's device address in the current context (looked up, without
    // allocating, on the first call in each context) and its size
    void *scratch = nullptr;
    size_t scratch_bytes = 0;
    rc = fa::decode_static_scratch(&scratch, &scratch_bytes);
    if (rc != FA_OK) return rc;
    size_t acc_bytes = 0, ml_bytes = 0;
    decode_layout(B, H, H_kv, N, d, &acc_bytes, &ml_bytes);
    if (acc_bytes + ml_bytes > scratch_bytes) {
        char msg[200];
        std::snprintf(msg, sizeof msg,
                      "request needs %zu bytes of decoding scratch, more than the %zu MiB "
                      "the library owns; use fa_decode with a workspace",
                      acc_bytes + ml_bytes, scratch_bytes >> 20);
        return fa::record_message(FA_ERR_WORKSPACE, msg);
    }
    // Same checks and kernels as the caller-workspace entry point.
    return fa_decode(Q, K, V, O, LSE, scratch, scratch_bytes, B, H, H_kv, N, d, scale, stream);
}

// ------------------------------------------------------------ backward
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
    if (check_shape(B, H, N, d, 1.f) != FA_OK) return 0;
    // two fp32 values per query row, rows padded to a multiple of 128 per head
    const size_t npad = (static_cast<size_t>(N) + 127) / 128 * 128;
    return align256(2 * static_cast<size_t>(B) * H * npad * sizeof(float));
}

int fa_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
           const float *LSE, void *dQ, void *dK, void *dV, void *workspace,
           size_t workspace_bytes, int B, int H, int N, int d, int causal, float scale,
           fa_stream_t stream) {
    return fa_bwd_gqa(Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B, H, H, N,
                      d, causal, scale, stream);
}

int fa_bwd_gqa(const void *Q, const void *K, const void *V, const void *O, const void *dO,
               const float *LSE, void *dQ, void *dK, void *dV, void *workspace,
               size_t workspace_bytes, int B, int H, int H_kv, int N, int d, int causal,
               float scale, fa_stream_t stream) {
    if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV) return FA_ERR_NULL;
    int rc = check_shape(B, H, N, d, scale);
    if (rc != FA_OK) return rc;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_SHAPE;
    const auto mis16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (mis16(Q) || mis16(K) || mis16(V) || mis16(O) || mis16(dO) || mis16(dQ) || mis16(dK) ||
        mis16(dV) || (reinterpret_cast<uintptr_t>(LSE) & 3u) != 0)
        return FA_ERR_ALIGN;
    const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
    if (!workspace || workspace_bytes < need ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return FA_ERR_WORKSPACE;
    const size_t t_bytes = static_cast<size_t>(B) * H * N * d * 2;
    const size_t kv_bytes = static_cast<size_t>(B) * H_kv * N * d * 2;
    const size_t l_bytes = static_cast<size_t>(B) * H * N * 4;
    const struct { const void *p; size_t n; } ins[] = {
        {Q, t_bytes}, {K, kv_bytes}, {V, kv_bytes}, {O, t_bytes}, {dO, t_bytes}, {LSE, l_bytes}};
    const struct { const void *p; size_t n; } outs[] = {
        {dQ, t_bytes}, {dK, kv_bytes}, {dV, kv_bytes}, {workspace, need}};
    for (const auto &o : outs) {
        for (const auto &in : ins)
            if (overlaps(o.p, o.n, in.p, in.n)) return FA_ERR_ALIAS;
        for (const auto &o2 : outs)
            if (&o2 != &o && overlaps(o.p, o.n, o2.p, o2.n)) return FA_ERR_ALIAS;
    }
    rc = check_arch();
    if (rc != FA_OK) return rc;
    CUtensorMap tmQ, tmK, tmV, tmdO, tmQ64, tmK64, tmV64, tmdO64;
    const int BH = B * H;
    if (!encode_qkv_map(&tmQ, Q, BH, N, d) || !encode_qkv_map(&tmK, K, B * H_kv, N, d) ||
        !encode_qkv_map(&tmV, V, B * H_kv, N, d) || !encode_qkv_map(&tmdO, dO, BH, N, d))
        return fa::record_message(FA_ERR_LAUNCH, "cuTensorMapEncodeTiled failed");
    // d = 256 streams 64-row halves (Q, dO in the dK/dV kernel; K, V in dQ)
    if (d == 256 && (!encode_qkv_map(&tmQ64, Q, BH, N, d, 64) ||
                     !encode_qkv_map(&tmK64, K, B * H_kv, N, d, 64) ||
                     !encode_qkv_map(&tmV64, V, B * H_kv, N, d, 64) ||
                     !encode_qkv_map(&tmdO64, dO, BH, N, d, 64)))
        return fa::record_message(FA_ERR_LAUNCH, "cuTensorMapEncodeTiled failed");
    fa::BwdArgs a;
    a.tmQ = &tmQ;
    a.tmK = &tmK;
    a.tmV = &tmV;
    a.tmdO = &tmdO;
    const bool d256 = d == 256;
    a.tmQ64 = d256 ? &tmQ64 : nullptr;
    a.tmK64 = d256 ? &tmK64 : nullptr;
    a.tmV64 = d256 ? &tmV64 : nullptr;
    a.tmdO64 = d256 ? &tmdO64 : nullptr;
    a.O = O;
    a.dO = dO;
    a.LSE = LSE;
    a.rows = static_cast<float *>(workspace);
    a.dQ = dQ;
    a.dK = dK;
    a.dV = dV;
    a.BH = BH;
    a.N = N;
    a.d = d;
    a.H = H;
    a.Hkv = H_kv;
    a.causal = causal != 0;
    a.scale = scale;
    a.limit_ns = kWaitLimitNs;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    return fa::launch_bwd(a);
}

int fa_device_error(fa_stream_t stream) {
    g_last_status = 0;
    // status words in the order of fa_last_device_status's kernel numbers
    int w[5] = {0, 0, 0, 0, 0};
    int rc = fa::read_and_clear_status(reinterpret_cast<cudaStream_t>(stream), &w[0]);
    if (rc != FA_OK) return rc;
    rc = fa::fwd256_read_and_clear_status(&w[1]);
    if (rc != FA_OK) return rc;
    rc = fa::bwd_read_and_clear_status(&w[2]);
    if (rc != FA_OK) return rc;
    rc = fa::bwd256_read_and_clear_status(&w[3]);
    if (rc != FA_OK) return rc;
    rc = fa::dec_read_and_clear_status(&w[4]);
    if (rc != FA_OK) return rc;
    for (int k = 0; k < 5; ++k) {
        if (w[k] == 0) continue;
        g_last_status = ((k + 1) << 8) | (w[k] & 0xFF);
        return (w[k] & 0x80) ? FA_ERR_CHECK : FA_ERR_TIMEOUT;
    }
    return FA_OK;
}

int fa_last_device_status(void) { return g_last_status; }

int fa_selftest_bounded_wait(int limit_us, fa_stream_t stream) {
    if (limit_us < 1 || limit_us > 1000000) return FA_ERR_SHAPE;
    int rc = check_arch();
    if (rc != FA_OK) return rc;
    rc = fa::launch_wait_selftest(static_cast<uint64_t>(limit_us) * 1000ull,
                                  reinterpret_cast<cudaStream_t>(stream));
    if (rc != FA_OK) return rc;
    return fa_device_error(stream);
}

const char *fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "ok";
        case FA_ERR_NULL: return "a required pointer is NULL";
        case FA_ERR_SHAPE: return "invalid shape (B, H, N must be >= 1 and fit the indexing)";
        case FA_ERR_HEADDIM:
            return "head dimension not supported (64, 128 or 256)";
        case FA_ERR_ALIGN: return "Q, K, V, O must be 16-byte aligned and LSE 4-byte aligned";
        case FA_ERR_ARCH: return "current device is not compute capability 10.3 (sm_103)";
        case FA_ERR_LAUNCH: return "a CUDA call failed";
        case FA_ERR_TIMEOUT: return "a kernel wait exceeded its time limit";
        case FA_ERR_UNSUPPORTED: return "request not supported by this library";
        case FA_ERR_SCALE: return "scale must be a finite number > 0";
        case FA_ERR_ALIAS: return "an output buffer overlaps an input buffer";
        case FA_ERR_WORKSPACE: return "workspace NULL, too small or not 256-byte aligned";
        case FA_ERR_CHECK: return "a device index check failed (debug build)";
        default: return "unknown status";
    }
}

int fa_version(void) { return 100; }

const char *fa_last_error_detail(void) { return g_detail; }

}  // extern "C"
