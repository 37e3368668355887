/*
 * fa_debug.h -- extra entry points of the debug build of the library
 * (_build/libfa_gb300_debug.so, the attention kernels compiled with FA_DEBUG).
 *
 * The debug build exports everything fa.h declares and behaves like the
 * release build, with one difference: the forward, backward and decoding
 * kernels (head dimensions 64, 128 and 256) check each index they compute
 * before using it:
 *   - the work item id (from the grid or a cancelled CTA) or the CTA's
 *     (head, block);
 *   - the head and row coordinates of every Q, K, V and dO tensor-map load
 *     and of every bulk copy of the backward's row statistics, and the query
 *     rows decoding reads;
 *   - the shared-memory ranges that the loads write and the MMAs read;
 *   - the tensor-memory allocation;
 *   - the element range and alignment of every O, dQ, dK and dV store, the
 *     index of every LSE (and backward statistics) store, and the slot of
 *     every partial decoding state written and merged.
 * A failed check writes 0x80 | its number to the kernel's device status
 * word; the first error wins.  The access is skipped, and the CTA's abort
 * flag is raised so the CTA's other warps stop at their next wait.  No
 * check traps.  fa_device_error then returns FA_ERR_CHECK, and
 * fa_last_device_status returns (k << 8) | 0x80 | n, with k the kernel
 * number of fa.h (1 forward d 64/128, 2 forward d 256, 3 backward d 64/128,
 * 4 backward d 256, 5 decoding), and n:
 *   1 item id, 2 Q (dO) load, 3 K/V load, 4 shared memory, 5 tensor
 *   memory, 6 O (dQ, dK, dV) store, 7 LSE (statistics) store.
 * The fault knobs below apply to the forward kernels.
 * The checks follow the kernel's own design: one CTA per
 * (batch, head, query block) work item, tiled over key blocks
 * ("Understanding FlashAttention Pt 1" (wpnews.pro), section 2.4, and
 * "FlashAttention-2 -- Deeper Math" (aicassindra.com), "Fix 3" and "Fix 4").
 *
 * The release library does not export the functions below.
 */
#ifndef FA_GB300_FA_DEBUG_H
#define FA_GB300_FA_DEBUG_H

#include "fa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_DEBUG_NONE = 0,           /* disarm */
    /* The producer of work item `a` (a CTA's first item is its grid index)
     * skips the load of key tile `b` (0-based; at d = 256 the tile's first
     * half of K columns) and the arrival on that tile's barrier, as if the
     * arrival had been lost.  The waits that
     * depend on the tile run out after the launch's limit: the kernel
     * drains its copies, frees its tensor memory and exits, and
     * fa_device_error returns FA_ERR_TIMEOUT. */
    FA_DEBUG_LOSE_K_ARRIVAL = 1,
    /* The O and LSE store checks take the output to hold only `a` rows
     * (of the B*H*N rows it really holds).  Every store to a row >= a fails
     * its check and is skipped, although it lies inside the real buffer.
     * `b` is unused. */
    FA_DEBUG_SHRINK_OUTPUT = 2
} fa_debug_fault;

/*
 * fa_debug_arm -- arms one fault for the next launch of a forward kernel
 * (any head dimension) made by this process (fa_fwd, fa_fwd_gqa, or the
 * host-buffer variants).  That launch disarms it.  While a fault is
 * armed, `limit_us` (1 .. 1000000) replaces that launch's time limit per
 * wait (2 s); 0 keeps the default.  Host-only: it enqueues nothing and
 * needs no GPU.
 *   fault       one of fa_debug_fault; FA_DEBUG_NONE disarms
 *   a, b        the fault's arguments (see fa_debug_fault), >= 0
 * Returns FA_OK; FA_ERR_UNSUPPORTED for an unknown fault; FA_ERR_SHAPE for
 * a negative argument or a limit out of range.  Thread-safe.
 */
int fa_debug_arm(int fault, long long a, long long b, int limit_us);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_DEBUG_H */
