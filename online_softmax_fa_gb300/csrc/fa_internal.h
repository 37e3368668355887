// fa_internal.h -- declarations shared by the C-ABI layer (fa_api.cu) and the
// kernel translation unit (fa_fwd_sm103.cu).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/fa.h"

namespace fa {

struct LaunchArgs {
    const CUtensorMap *tmQ, *tmK, *tmV;
    const CUtensorMap *tmV64;  // d = 256: V with 64-row boxes
    void *O;
    float *LSE;
    int BH, N, d;
    int H, Hkv;  // query heads and K/V heads per batch (H % Hkv == 0)
    bool causal;
    float scale;
    uint64_t limit_ns;  // bound on every in-kernel wait
    cudaStream_t stream;
};

int launch_fwd(const LaunchArgs &a);
// d = 256 forward (fa_fwd256_sm103.cu).
int launch_fwd256(const LaunchArgs &a);

#ifdef FA_DEBUG
// The fault fa_debug_arm (fa_debug.h) armed, if any: taken, and disarmed,
// by the next forward launch (debug build only).
struct DebugFault {
    int fault;
    long long a, b;
    uint64_t limit_ns;  // 0: the launch's own limit
};
bool take_debug_fault(DebugFault *f);
#endif
int fwd256_read_and_clear_status(int *status);

// Backward pass (fa_bwd_sm103.cu).
struct BwdArgs {
    const CUtensorMap *tmQ, *tmK, *tmV, *tmdO;
    const CUtensorMap *tmQ64, *tmK64, *tmV64, *tmdO64;  // d = 256: 64-row boxes (else null)
    const void *O, *dO;          // bf16 [BH, N, d]
    const float *LSE;            // fp32 [BH, N] (natural log)
    float *rows;                 // fp32 scratch [2][BH][Npad]: LSE*log2(e), rowsum(dO*O)
    void *dQ;                    // bf16 [BH, N, d]
    void *dK, *dV;               // bf16 [BH / (H / Hkv), N, d]
    int BH, N, d;
    int H, Hkv;                  // query and K/V heads per batch (Hkv divides H)
    bool causal;
    float scale;
    uint64_t limit_ns;
    cudaStream_t stream;
};
int launch_bwd(const BwdArgs &a);
int bwd_read_and_clear_status(int *status);
// d = 256 dK/dV and dQ kernels (fa_bwd256_sm103.cu), after the pre-pass
// has written the padded -LSE*log2(e) and -D rows.
int launch_bwd256(const BwdArgs &a, const float *lse2, const float *dd, int n_blocks);
int bwd256_read_and_clear_status(int *status);

// Split-KV decoding (fa_decode_sm103.cu).
struct DecodeArgs {
    const CUtensorMap *tmK, *tmV;  // K, V as [B*H_kv, N, d], 64-row boxes
    const void *Q;          // bf16 [B,H,d]
    void *O;                // bf16 [B,H,d]
    float *LSE;             // fp32 [B,H]
    float *part_acc;        // fp32 [B*H_kv, slots, G, d]
    float *part_ml;         // fp32 [B*H_kv, slots, G, 2]
    int B, H, H_kv, N, d;
    float scale;
    uint64_t limit_ns;      // bound on every in-kernel wait
    cudaStream_t stream;
};
int launch_decode(const DecodeArgs &a);
// Partial softmax states a decoding workspace holds (device-independent).
size_t decode_state_count(int B, int H, int H_kv);
int dec_read_and_clear_status(int *status);
// Device address and size of the library-owned scratch area that
// fa_decode_noalloc uses (resolved once per device).
int decode_static_scratch(void **ptr, size_t *bytes);

// Records the CUDA error of a failed call (thread-local) for
// fa_last_error_detail(); returns FA_ERR_LAUNCH.
int record_cuda_error(cudaError_t e, const char *what);
int record_message(int status, const char *what);
#define FA_CUDA_TRY(call)                                              \
    do {                                                               \
        cudaError_t fa_e_ = (call);                                    \
        if (fa_e_ != cudaSuccess) return ::fa::record_cuda_error(fa_e_, #call); \
    } while (0)
int read_and_clear_status(cudaStream_t stream, int *status);

// Per-device facts kept for the life of the process, for device ordinals
// 0 .. kMaxDevices - 1.  Several host threads may fill an entry at the same
// time: they store the same value, and the entries are atomics, so the
// first launch on a device needs no lock.
constexpr int kMaxDevices = 64;
// SM count of device `dev` (queried once), or 0 if the query fails.
int device_sm_count(int dev);
// Sets `kern`'s dynamic shared-memory limit to `bytes` the first time it is
// launched on device `dev` (`flags`: one per device, zero-initialised).
template <class Kern>
int set_smem_once(std::atomic<int> *flags, int dev, Kern kern, int bytes) {
    if (flags[dev].load(std::memory_order_acquire)) return FA_OK;
    FA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
    flags[dev].store(1, std::memory_order_release);
    return FA_OK;
}
int launch_wait_selftest(uint64_t limit_ns, cudaStream_t stream);

}  // namespace fa
