/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact attention forward pass.
 *
 *   O   = softmax(scale * Q K^T [+ causal mask]) V
 *   LSE = m + log(l)          (per query row, natural log)
 *
 * The operation: "Chapter 26 Online Softmax & FlashAttention" (gowda.ai),
 * section 26.2 and Listing 26.2 (scores q k^T / sqrt(d), causal keeps key j
 * for query i iff j <= i, stable row softmax, weights @ v); the logsumexp
 * statistic L = m + log(l) is "Fix 2" of "FlashAttention-2 -- Deeper Math"
 * (aicassindra.com).  The kernel computes it exactly (no approximation)
 * with the online-softmax recurrence of "Understanding FlashAttention Pt 1"
 * (wpnews.pro), section 2.4, query blocks outermost ("Fix 3"), one CTA per
 * (batch, head, query block) ("Fix 4"), and causal tiles above the diagonal
 * skipped ("Causal masking: skip the blocks, do not mask them").
 *
 * Every entry point returns an fa_status (0 = success, negative = error).
 * No entry point falls back to another implementation: an unsupported
 * argument is an error code.  Nothing here is thread-hostile; concurrent
 * calls on different streams are independent.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle; identical to cudaStream_t / CUstream.  NULL is the
 * legacy default stream. */
typedef struct CUstream_st *fa_stream_t;

typedef enum {
    FA_OK = 0,
    FA_ERR_NULL = -1,        /* a required pointer is NULL */
    FA_ERR_SHAPE = -2,       /* B, H or N < 1, or a size overflows the indexing */
    FA_ERR_HEADDIM = -3,     /* d not supported by the entry point (see each) */
    FA_ERR_ALIGN = -4,       /* Q, K, V, O not 16-byte aligned, or LSE not 4-byte */
    FA_ERR_ARCH = -5,        /* current device is not compute capability 10.3 */
    FA_ERR_LAUNCH = -6,      /* a CUDA call failed (launch, copy, tensor map) */
    FA_ERR_TIMEOUT = -7,     /* a kernel wait exceeded its limit (see fa_device_error) */
    FA_ERR_UNSUPPORTED = -8, /* valid request this library does not implement */
    FA_ERR_SCALE = -9,       /* scale is not a finite number > 0 */
    FA_ERR_ALIAS = -10,      /* an output buffer overlaps an input buffer */
    FA_ERR_WORKSPACE = -11,  /* workspace too small or misaligned */
    FA_ERR_CHECK = -12       /* a device index check failed (debug build, fa_debug.h) */
} fa_status;

/*
 * fa_fwd -- attention forward on device buffers, enqueued on `stream`.
 *
 *   Q, K, V  bf16 [B, H, N, d], contiguous, device memory; element
 *            (b, h, n, k) at ((b*H + h)*N + n)*d + k.  Read only.
 *   O        bf16 [B, H, N, d], same layout, device memory, written.
 *   LSE      fp32 [B, H, N], device memory, written: log(sum_j exp(s_ij))
 *            over the scaled, masked scores s_ij = scale * q_i . k_j.
 *   B, H, N  >= 1.  B*H < 2^31, N < 2^31.
 *   d        64, 128 or 256 (head dimension; values have the same width;
 *            the pages list all three).  At 256 a separate kernel runs:
 *            128 query rows per work item, with S double-buffered in TMEM.
 *   causal   0: every key; nonzero: key j is used for query i iff j <= i.
 *   scale    finite, > 0; the pages' choice is 1/sqrt(d).
 *
 * All buffers are owned by the caller; the library keeps no pointer after
 * the call and allocates no device memory.  Q, K, V, O must be 16-byte
 * aligned, LSE 4-byte aligned, and O / LSE must not overlap Q, K or V.
 * Arguments are checked on the host before any CUDA call; on error nothing
 * is enqueued.  The kernel runs asynchronously: a FA_OK return means it was
 * enqueued, and fa_device_error() reports a failure found while it ran.
 * Results are deterministic: the same inputs give bit-identical outputs.
 */
int fa_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
           int B, int H, int N, int d, int causal, float scale,
           fa_stream_t stream);

/*
 * fa_fwd_gqa -- grouped-query (and multi-query) attention: H query heads
 * share H_kv key/value heads, query head h of batch b using K/V head
 * h / (H / H_kv) ("Understanding FlashAttention Pt 1", section 4.1: the
 * number of query heads is a multiple of the number of K/V heads).
 *
 *   Q, O     bf16 [B, H, N, d];  LSE fp32 [B, H, N]
 *   K, V     bf16 [B, H_kv, N, d]
 *   H_kv     >= 1 and divides H (H_kv = 1: multi-query; H_kv = H: fa_fwd)
 * Everything else, including errors (FA_ERR_SHAPE when H_kv does not divide
 * H), as fa_fwd.  Consecutive query heads of a group run next to each other
 * so they share the group's K/V through L2.
 */
int fa_fwd_gqa(const void *Q, const void *K, const void *V, void *O, float *LSE,
               int B, int H, int H_kv, int N, int d, int causal, float scale,
               fa_stream_t stream);

/*
 * fa_fwd_host_workspace_bytes -- device workspace fa_fwd_host needs for this
 * shape: room for Q, K, V, O (bf16) and LSE (fp32), each 256-byte aligned.
 * Returns 0 for an invalid shape.
 */
size_t fa_fwd_host_workspace_bytes(int B, int H, int N, int d);

/*
 * fa_fwd_host -- the same operation on HOST buffers: copies Q, K, V from
 * host to the device workspace, runs fa_fwd, and copies O and LSE back,
 * asynchronously with respect to the host and ordered after the earlier work
 * on `stream` (synchronise `stream` before reading O_host / LSE_host).  The
 * heads are cut into chunks whose copy-in, kernel and copy-out overlap on
 * four streams the library creates once per device (and keeps); calls that
 * use them are enqueued one at a time.  The results equal those of one
 * fa_fwd call.  Host buffers should be pinned for the copies to overlap;
 * pageable memory works but the copies then block the host.
 *
 *   Q_host, K_host, V_host  bf16 [B, H, N, d] in host memory (read).
 *   O_host                  bf16 [B, H, N, d] in host memory (written).
 *   LSE_host                fp32 [B, H, N] in host memory (written).
 *   workspace               caller-owned device memory of at least
 *                           fa_fwd_host_workspace_bytes(B, H, N, d) bytes,
 *                           256-byte aligned; contents are scratch.
 * Other arguments and errors as fa_fwd; FA_ERR_WORKSPACE if the workspace
 * is NULL, too small or misaligned.  Argument errors are found before
 * anything is enqueued.  A CUDA failure found part-way (a copy or launch the
 * runtime refuses after earlier chunks were enqueued) returns its error
 * with `stream` made to wait for everything already enqueued, so the host
 * and device buffers may be released once `stream` is synchronised; the
 * outputs are then undefined.
 */
int fa_fwd_host(const void *Q_host, const void *K_host, const void *V_host,
                void *O_host, float *LSE_host, void *workspace,
                size_t workspace_bytes, int B, int H, int N, int d,
                int causal, float scale, fa_stream_t stream);

/*
 * fa_fwd_host_gqa_workspace_bytes -- device workspace fa_fwd_host_gqa needs:
 * Q and O ([B, H, N, d] bf16), K and V ([B, H_kv, N, d] bf16) and LSE
 * ([B, H, N] fp32), each 256-byte aligned.  0 for an invalid shape or an
 * H_kv that does not divide H.
 */
size_t fa_fwd_host_gqa_workspace_bytes(int B, int H, int H_kv, int N, int d);

/*
 * fa_fwd_host_gqa -- fa_fwd_gqa on host buffers ("Understanding
 * FlashAttention Pt 1", section 4.1: H query heads share H_kv K/V heads):
 *   Q_host, O_host  bf16 [B, H, N, d];  LSE_host fp32 [B, H, N]
 *   K_host, V_host  bf16 [B, H_kv, N, d] (each K/V head copied in once for
 *                   its whole group of query heads)
 *   workspace       at least fa_fwd_host_gqa_workspace_bytes(B, H, H_kv, N, d)
 *                   bytes of device memory, 256-byte aligned
 * A chunk holds whole groups (a K/V head with all its query heads).  The
 * results equal those of one fa_fwd_gqa call.  Everything else, including
 * errors and the part-way failure rule, as fa_fwd_host; fa_fwd_host is this
 * call with H_kv = H.
 */
int fa_fwd_host_gqa(const void *Q_host, const void *K_host, const void *V_host,
                    void *O_host, float *LSE_host, void *workspace,
                    size_t workspace_bytes, int B, int H, int H_kv, int N, int d,
                    int causal, float scale, fa_stream_t stream);

/*
 * fa_bwd_workspace_bytes -- device workspace fa_bwd needs: two fp32 per
 * query row (D_i = sum_r dO_ir O_ir and LSE_i log2 e), rows padded to a
 * multiple of 128 per head, 256-byte aligned.  0 if invalid.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * fa_bwd -- gradients of fa_fwd by recomputation ("Understanding
 * FlashAttention Pt 1", section 3.6): the probability tiles are rebuilt from
 * the forward's LSE (P_ij = exp(S_ij - LSE_i), "Fix 2" of "FlashAttention-2
 * -- Deeper Math") instead of being stored, and
 *   dV = P^T dO,  dP = dO V^T,  D_i = sum_r dO_ir O_ir,
 *   dS = P * (dP - D_i),  dQ = scale * dS K,  dK = scale * dS^T Q.
 *
 *   Q, K, V, O, dO  bf16 [B, H, N, d] (O and LSE as fa_fwd wrote them for
 *                   the same Q, K, V, causal and scale), device, read
 *   LSE             fp32 [B, H, N], device, read
 *   dQ, dK, dV      bf16 [B, H, N, d], device, written
 *   d               64, 128 or 256 (at 256 other kernels run: dK / dV by two
 *                   CTAs per key block, one per half of d, and the query or
 *                   key rows streamed in 64-row halves; correct and
 *                   deterministic, about a third of the d <= 128 rate)
 *   workspace       caller-owned device scratch of at least
 *                   fa_bwd_workspace_bytes(B, H, N, d) bytes, 256-byte aligned
 * Three kernels on `stream` (D, then dK/dV with key blocks outermost, then
 * dQ with query blocks outermost); no atomics, so the result is
 * deterministic.  Checks and errors as fa_fwd (outputs and workspace must
 * not overlap any input or each other; FA_ERR_WORKSPACE for a missing,
 * small or misaligned workspace).
 */
int fa_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
           const float *LSE, void *dQ, void *dK, void *dV, void *workspace,
           size_t workspace_bytes, int B, int H, int N, int d, int causal, float scale,
           fa_stream_t stream);

/*
 * fa_bwd_gqa -- fa_bwd for grouped-query (and multi-query) attention, the
 * gradients of fa_fwd_gqa: H query heads share H_kv K/V heads, query head h
 * of a batch reading K/V head h / (H / H_kv) ("Understanding FlashAttention
 * Pt 1", section 4.1).  The forward pass is the dense one on K/V heads
 * repeated for their group, so a K/V head's gradient is the sum of the
 * dense gradients of its repeats; dQ is the dense one.
 *
 *   Q, O, dO        bf16 [B, H, N, d], device, read
 *   K, V            bf16 [B, H_kv, N, d], device, read
 *   LSE             fp32 [B, H, N], device, read
 *   dQ              bf16 [B, H, N, d], device, written
 *   dK, dV          bf16 [B, H_kv, N, d], device, written
 *   H_kv            >= 1 and dividing H (FA_ERR_SHAPE otherwise)
 *   workspace       as fa_bwd: fa_bwd_workspace_bytes(B, H, N, d) bytes
 * The dK/dV kernel runs one CTA per (K/V head, key block) and walks the
 * query blocks of every query head of the group in turn, so the group sum
 * is accumulated in TMEM in a fixed order: deterministic, no atomics.
 * fa_bwd(...) is fa_bwd_gqa with H_kv = H.  Other checks and errors as
 * fa_bwd.
 */
int fa_bwd_gqa(const void *Q, const void *K, const void *V, const void *O, const void *dO,
               const float *LSE, void *dQ, void *dK, void *dV, void *workspace,
               size_t workspace_bytes, int B, int H, int H_kv, int N, int d, int causal,
               float scale, fa_stream_t stream);

/*
 * fa_decode_workspace_bytes -- device workspace fa_decode needs: the
 * per-split softmax states (m, l and the d-wide accumulator for every
 * query head and key split).  Returns 0 for an invalid or unsupported shape.
 */
size_t fa_decode_workspace_bytes(int B, int H, int H_kv, int N, int d);

/*
 * fa_decode -- one new query row per (batch, query head) against a
 * key/value cache: O = softmax(scale * q K^T) V and LSE, every cached key
 * visible.  Decoding has no query-block parallelism ("FlashAttention-2 --
 * Deeper Math", "What FA-2 does not fix"), so the keys are split across
 * the GPU: every SM streams an equal run of the cache, its warps keep the
 * online-softmax state of "Understanding FlashAttention Pt 1", section 2.4,
 * for their keys, and a second kernel merges the partial states with the
 * same rule.  The workspace size depends on B, H and H_kv only.
 *
 *   Q, O     bf16 [B, H, d] (the newest token of each sequence and head)
 *   K, V     bf16 [B, H_kv, N, d], N cached positions
 *   LSE      fp32 [B, H]
 *   H_kv     divides H; H / H_kv in {1, 2, 4, 8} (FA_ERR_UNSUPPORTED else);
 *            each K/V row is read once for all query heads of its group
 *   d        64, 128 or 256; B * H_kv <= 65535
 *   workspace  caller-owned device memory of at least
 *            fa_decode_workspace_bytes(B, H, H_kv, N, d) bytes, 256-byte
 *            aligned; its contents are scratch and it must not overlap the
 *            other buffers
 * Checks, errors and asynchrony as fa_fwd (FA_ERR_WORKSPACE for a missing,
 * small or misaligned workspace).  Two kernels run on `stream`.
 */
int fa_decode(const void *Q, const void *K, const void *V, void *O, float *LSE,
              void *workspace, size_t workspace_bytes, int B, int H, int H_kv,
              int N, int d, float scale, fa_stream_t stream);

/*
 * fa_decode_noalloc -- fa_decode for callers that cannot allocate device
 * memory when they decode (an allocation can block on or synchronise with
 * queued device work, can fail once a host framework's pool owns the free
 * memory, and some plugin hosts give a component only its input and output
 * buffers).  The pages have no counterpart: this is an interface variant.
 * Same arguments as fa_decode minus the workspace: the split states live in
 * a 16 MiB area of device memory that the library owns (every GPU that
 * loads the library keeps it reserved until the process exits).
 *   - Requests whose states need more than 16 MiB, i.e.
 *     fa_decode_workspace_bytes(B, H, H_kv, N, d) > 16 MiB, return
 *     FA_ERR_WORKSPACE (fa_last_error_detail says why) and enqueue nothing.
 *   - Allocates nothing, on the host or the device.
 *   - The area's device address belongs to the CUDA context: the first
 *     call in each context (per device, with that device current) looks it
 *     up without allocating and caches it with the context's unique id; a
 *     later call in another context, or after cudaDeviceReset(), looks it up
 *     again.  Make that first call in a context before any stream capture.
 *   - Every call shares the one area: calls that overlap on the GPU (other
 *     streams, other host threads) race and must be ordered by the caller.
 *     Nothing in it has to start at zero: each call writes every state it
 *     later reads.
 */
int fa_decode_noalloc(const void *Q, const void *K, const void *V, void *O, float *LSE,
                      int B, int H, int H_kv, int N, int d, float scale,
                      fa_stream_t stream);

/*
 * fa_device_error -- synchronises `stream`, then reads and clears the
 * library's device status word on the current device.  Returns FA_OK, or
 * FA_ERR_TIMEOUT if a kernel since the last call gave up on a bounded wait
 * (every wait inside the kernels has a time limit; on expiry the kernel
 * drains its own copies, frees its tensor memory and exits early, leaving
 * its outputs undefined), FA_ERR_CHECK if a device index check of the debug
 * build failed (a timeout caused by it is not reported separately), or
 * FA_ERR_LAUNCH if the synchronisation itself reported a CUDA error.
 */
int fa_device_error(fa_stream_t stream);

/*
 * fa_last_device_status -- the raw device status behind the calling
 * thread's last fa_device_error (or fa_selftest_bounded_wait) result: 0 if
 * that returned FA_OK, else (kernel << 8) | code for the first kernel, in
 * the order below, whose status word was set:
 *   kernel  1 forward (d 64, 128)   2 forward (d 256)   3 backward (d 64, 128)
 *           4 backward (d 256)      5 decoding
 *   code    1 .. 127: the bounded wait that ran out (each kernel numbers
 *           its own waits; 127 is the self-test's wait);
 *           0x80 | n: device check n failed (debug build, fa_debug.h).
 * Host-only; never fails.
 */
int fa_last_device_status(void);

/*
 * fa_selftest_bounded_wait -- runs a one-CTA kernel that waits on a barrier
 * nothing ever signals, with the same bounded-wait code the forward kernel
 * uses and a limit of `limit_us` microseconds (1 .. 1000000).  It checks
 * that an expired wait ends the kernel with a status instead of a hang.
 * Returns the device status the kernel left (FA_ERR_TIMEOUT when the
 * mechanism works), after synchronising `stream`.  The status word is
 * cleared before returning.
 */
int fa_selftest_bounded_wait(int limit_us, fa_stream_t stream);

/* Static description of a status code; never NULL. */
const char *fa_status_string(int status);

/* Text of the last CUDA failure seen by this thread inside the library
 * (the failing call and CUDA's error name), or "" if none.  The buffer is
 * thread-local and stays valid until this thread's next failing call. */
const char *fa_last_error_detail(void);

/* Library ABI version: major*10000 + minor*100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
