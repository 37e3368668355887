// debug_checks.cuh -- device checks of the debug build (compiled with
// FA_DEBUG) of the attention kernels.  Every index a kernel computes is
// checked before use; a failed check records 0x80 | its number in the
// kernel's status word (first error wins), raises the CTA's abort flag and
// skips the access, so the CTA's other warps stop at their next wait that
// does not complete at once.  No check traps.  Release builds compile every
// check to `true`.
#pragma once

#include "sm103_primitives.cuh"

namespace fa {

enum : int {
    kChkItem = 1,  // work item id outside [0, n_items)
    kChkTmaQ,      // Q box rows outside the padded query rows, or head >= B*H
    kChkTmaKV,     // K/V box starting past the keys, or K/V head >= B*H_kv
    kChkSmem,      // a shared-memory range outside the CTA's allocation
    kChkTmem,      // tensor memory not the whole 512-column allocation
    kChkStoreO,    // an O store outside the output, or misaligned for its width
    kChkStoreLse   // an LSE store outside the output
};

#ifdef FA_DEBUG
constexpr bool kDebug = true;
__device__ __forceinline__ bool dbg_ok(bool cond, const WaitCtl &c, int check) {
    if (cond) return true;
    raise_abort(c, 0x80 | check);
    return false;
}
// The same for a kernel without bounded waits: records the failure in
// `status` only.
__device__ __forceinline__ bool dbg_ok_word(bool cond, int *status, int check) {
    if (cond) return true;
    atomicCAS(status, 0, 0x80 | check);
    return false;
}
#else
constexpr bool kDebug = false;
__device__ __forceinline__ bool dbg_ok(bool, const WaitCtl &, int) { return true; }
__device__ __forceinline__ bool dbg_ok_word(bool, int *, int) { return true; }
#endif

// [ptr, ptr + bytes) lies inside the CTA's dynamic shared memory of
// `smem_bytes` bytes, below the 256 KB a matrix descriptor's 14-bit address
// field reaches.
__device__ __forceinline__ bool in_smem(const void *ptr, int bytes, int smem_bytes) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw), a = smem_u32(ptr);
    const uint32_t end = base + static_cast<uint32_t>(smem_bytes);
    return a >= base && a + static_cast<uint32_t>(bytes) <= end && a + bytes <= (1u << 18);
}

// The same against a kernel's own aligned dynamic shared-memory base.
__device__ __forceinline__ bool in_smem_at(const void *base, const void *ptr, int bytes,
                                           int smem_bytes) {
    const uint32_t b = smem_u32(base), a = smem_u32(ptr);
    return a >= b && a + static_cast<uint32_t>(bytes) <= b + static_cast<uint32_t>(smem_bytes);
}

// The TMEM address of a whole 512-column allocation starts at lane 0,
// column 0.
__device__ __forceinline__ bool whole_tmem(uint32_t tmem) { return tmem == 0u; }

}  // namespace fa
