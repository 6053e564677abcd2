/*
 * mha_fwd.h - fused multi-head attention forward pass for NVIDIA GB300
 * (sm_103a), C ABI.
 *
 * The operation is the FlashAttention-2 forward pass: "two back-to-back
 * GEMMs with an online softmax in between" (ML-Triton paper, section 2.5,
 * Algorithm 1).  For every batch b, head h and query row i:
 *
 *     s_ij  = scale * <q_i, k_j>                 for j in J_i
 *     J_i   = {0 .. N-1}, or {0 .. i} when causal != 0
 *     O_i   = sum_j softmax(s_i)_j * v_j         (Triton-learning blog,
 *                                                 Puzzle 9 definition)
 *     LSE_i = ln sum_j exp(s_ij)                 (natural log)
 *
 * The row maximum and row sum are carried across key tiles with the online
 * merge of the blog's Puzzle 8 and the output rescale of its Puzzle 9.
 * S and P never reach global memory.
 *
 * Conventions shared by every entry point:
 *   - Tensors are contiguous, row-major, and live in device memory.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and returns once the work is queued.
 *   - The caller allocates and owns every buffer.  The library allocates no
 *     device memory; it keeps one status word per device in module memory.
 *   - No call throws, aborts or exits.  A non-zero return means nothing
 *     useful was written to the outputs.
 *   - Per-device set-up (the architecture check, kernel attributes and the
 *     status word's address) happens on the first call on each device and
 *     is cached.  cudaDeviceReset discards the module memory that cache
 *     points into: do not call the library on a device after resetting it.
 */
#ifndef MHA_FWD_H
#define MHA_FWD_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum {
    MHA_OK = 0,
    MHA_ERR_INVALID_ARG = 1,     /* negative size, NULL pointer, bad scale   */
    MHA_ERR_UNSUPPORTED_DIM = 2, /* head dimension d is not 64 or 128         */
    MHA_ERR_MISALIGNED = 3,      /* a pointer is not 16-byte aligned          */
    MHA_ERR_CUDA = 4,            /* a CUDA runtime or driver call failed      */
    MHA_ERR_TIMEOUT = 5,         /* a device-side wait ran past its limit     */
    MHA_ERR_NO_DEVICE = 6,       /* no usable sm_103 device is current        */
    MHA_ERR_SCRATCH_LIMIT = 7    /* mha_fwd_kv_noalloc: the problem needs more
                                    scratch than the built-in buffer holds   */
} mha_status;

/*
 * mha_fwd - attention forward pass.
 *
 *   q, k, v : bf16 [B, H, N, d], device, read only.
 *   o       : bf16 [B, H, N, d], device, written (rounded to nearest even).
 *   lse     : fp32 [B, H, N], device, written: LSE_i as defined above.
 *   B, H, N : batch, heads, sequence length (queries = keys = N), each >= 0.
 *             B*H*N == 0 is a no-op that returns MHA_OK.  B*H <= INT_MAX and
 *             B*H*ceil(N/256) <= 2^30 (tensors of that size would not fit
 *             in device memory), else MHA_ERR_INVALID_ARG.
 *   d       : head dimension, 64 or 128.
 *   scale   : score multiplier, finite and > 0 (usually 1/sqrt(d) in fp32).
 *   causal  : 0 = every key; non-zero = key j > query i excluded (square,
 *             top-left aligned mask).
 *   stream  : cudaStream_t to launch on.
 *
 * All five pointers must be non-NULL and 16-byte aligned, and `o` / `lse`
 * must not overlap the inputs.  Errors in the arguments are reported before
 * any CUDA call.  MHA_ERR_CUDA reports a failed launch; faults that happen
 * while the kernel runs surface at the caller's next synchronising CUDA call.
 */
int mha_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
            int B, int H, int N, int d, float scale, int causal, void *stream);

/*
 * mha_fwd_kv - attention forward for a few queries against a long key/value
 * sequence (decode), computed by splitting the keys across CTAs and merging
 * the partial results by their log-sum-exp ("flash decoding": the split of
 * keys and values across workers and the reduction of their partial results
 * that the ML-Triton paper describes in section 3.2).
 *
 *   q       : bf16 [B, H, Nq, d], device, read only; 0 <= Nq <= 16.
 *   k, v    : bf16 [B, H, Nk, d], device, read only; Nk >= 1.
 *   o       : bf16 [B, H, Nq, d], device, written.
 *   lse     : fp32 [B, H, Nq], device, written (natural log).
 *   d       : 64 or 128.  scale: finite and > 0.
 *   causal  : 0 = every query sees every key; non-zero = the queries are the
 *             last Nq positions of the sequence (bottom-right alignment):
 *             query i sees keys 0 .. Nk-Nq+i.  With Nq == Nk this is the
 *             mask of mha_fwd.  A query with no visible key gets O = 0 and
 *             LSE = -inf.
 *   num_splits : number of key splits, or 0 to let the library choose.
 *   workspace, workspace_bytes : device scratch owned by the caller, 16-byte
 *             aligned, at least mha_fwd_kv_workspace_size(...) bytes, not
 *             overlapping any other argument.  Its contents need no
 *             initialisation and are garbage afterwards.
 *   stream  : cudaStream_t; three kernels are queued on it: one that
 *             zeroes a work-tile counter in the workspace, the partial pass
 *             and the merge.  The last two are launched as programmatic
 *             dependents of the kernel before them: each may start while
 *             that one runs and waits for its results before reading them.
 *
 * B*H == 0 or Nq == 0 is a no-op.  Errors as for mha_fwd.
 */
int mha_fwd_kv(const void *q, const void *k, const void *v, void *o, float *lse,
               int B, int H, int Nq, int Nk, int d, float scale, int causal,
               int num_splits, void *workspace, size_t workspace_bytes, void *stream);

/*
 * mha_fwd_paged - mha_fwd_kv over a paged K/V cache: the cache is split into
 * fixed-size blocks of page_size keys, and each sequence reaches its keys
 * through a block table (the paged-attention layout the ML-Triton paper
 * evaluates in sections 3.2 and 4.3).
 *
 *   q           : bf16 [B, H, Nq, d], device; 0 <= Nq <= 16.
 *   k_cache,
 *   v_cache     : bf16 [num_blocks, H, page_size, d], device.
 *   block_table : int32 [B, max_blocks], device: logical page i of batch
 *                 entry b is physical block block_table[b*max_blocks + i].
 *                 An id outside [0, num_blocks) reads as zeros.
 *   seq_lens    : int32 [B], device: keys cached for each batch entry
 *                 (clamped to max_blocks*page_size); key t of entry b is row
 *                 t % page_size of block block_table[b][t / page_size].
 *   o, lse      : as for mha_fwd_kv.
 *   page_size   : 16, 32, 64, 128 or 256.
 *   num_blocks  : >= 1, with (num_blocks + 1) * H <= INT_MAX.
 *   causal      : bottom-right aligned per batch entry (query i of entry b
 *                 sees keys 0 .. seq_lens[b]-Nq+i); a query with no visible
 *                 key gets O = 0, LSE = -inf.
 *   workspace   : at least mha_fwd_kv_workspace_size(B, H, Nq,
 *                 max_blocks*page_size, d, num_splits) bytes.
 * block_table and seq_lens must be 4-byte aligned; every other pointer
 * 16-byte aligned.  Other conventions and errors as for mha_fwd_kv.
 */
int mha_fwd_paged(const void *q, const void *k_cache, const void *v_cache,
                  const int *block_table, const int *seq_lens, void *o, float *lse,
                  int B, int H, int Nq, int d, int page_size, int num_blocks,
                  int max_blocks, float scale, int causal, int num_splits,
                  void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes mha_fwd_kv needs for this shape and split request (0 for
 * an empty problem or invalid arguments).  A pure function of its arguments;
 * no CUDA call. */
size_t mha_fwd_kv_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits);

/*
 * mha_fwd_kv_noalloc - mha_fwd_kv for callers that cannot allocate device
 * memory.  (The pages this library follows have no counterpart: this entry
 * point exists for deployment reasons only.)
 *
 * Some callers hold raw device pointers to their inputs and outputs but
 * cannot obtain a workspace: a plug-in inside another runtime that owns all
 * allocations, a service that reserves its memory at start-up and may not
 * allocate while serving, a host program with no access to the allocator
 * behind its buffers.  This call takes the same arguments as mha_fwd_kv
 * minus the workspace and uses a scratch buffer of 16 MiB (16777216 bytes)
 * that the library keeps in its own module memory on every GPU that loads
 * it, for the life of the process.  It allocates nothing.
 *
 *   - Problems whose workspace (mha_fwd_kv_workspace_size with the same
 *     arguments) exceeds 16 MiB are rejected with MHA_ERR_SCRATCH_LIMIT
 *     before any CUDA call; other argument errors as for mha_fwd_kv.
 *   - The first call on each device looks up the buffer's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture begins.
 *   - All calls on a device share the one buffer, and it keeps whatever the
 *     last call left there.  Nothing in it needs to start at zero: every
 *     element a call reads back was written earlier in the same call.  Calls
 *     whose execution overlaps on the GPU (for example on two streams) race
 *     on the buffer and must be serialised by the caller.
 *   - If mha_device_status reports MHA_ERR_TIMEOUT after a call, that call's
 *     o and lse are undefined: a work tile that gave up may have left its
 *     part of the buffer holding an earlier call's data.
 *   - The buffer's device address is cached per device.  After
 *     cudaDeviceReset the library's module memory is gone; the library must
 *     not be called again on that device in the same process.
 */
int mha_fwd_kv_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                       int B, int H, int Nq, int Nk, int d, float scale, int causal,
                       int num_splits, void *stream);

/*
 * mha_bwd - gradients of the attention forward pass (mha_fwd) with respect
 * to q, k and v, for a loss whose gradient with respect to O is dout.
 *
 * The pages describe the forward pass only; these are the derivatives of
 * its definition (chain rule through the row softmax), in the
 * FlashAttention-2 arrangement that recomputes P from the saved LSE.  For
 * each batch b, head h, with P_ij = exp(scale <q_i, k_j> - LSE_i) on the key
 * set J_i of mha_fwd (and 0 elsewhere):
 *
 *     D_i   = sum_c dout_ic O_ic
 *     dS_ij = P_ij (<dout_i, v_j> - D_i)
 *     dq_i  = scale sum_j dS_ij k_j
 *     dk_j  = scale sum_i dS_ij q_i
 *     dv_j  = sum_i P_ij dout_i
 *
 *   q, k, v    : bf16 [B, H, N, d], device, the forward inputs.
 *   o, lse     : the forward outputs of mha_fwd for these inputs (bf16
 *                [B, H, N, d] and fp32 [B, H, N]); they are used as given.
 *   dout       : bf16 [B, H, N, d], device, gradient of the loss w.r.t. O.
 *   dq, dk, dv : bf16 [B, H, N, d], device, written.
 *   d, scale, causal : as passed to mha_fwd.
 *   workspace, workspace_bytes : device scratch owned by the caller, at
 *                least mha_bwd_workspace_size(B, H, N, d) bytes (fp32 D_i
 *                per row); contents need no initialisation.
 *   stream     : cudaStream_t; three kernels are queued on it.
 *
 * Every pointer must be non-NULL and 16-byte aligned; the three outputs and
 * the workspace must not overlap each other or any input.  B*H*N == 0 is a
 * no-op.  Errors as for mha_fwd.
 */
int mha_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
            const void *dout, void *dq, void *dk, void *dv, int B, int H, int N, int d,
            float scale, int causal, void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes mha_bwd needs (0 for invalid arguments).  No CUDA call. */
size_t mha_bwd_workspace_size(int B, int H, int N, int d);

/* A short, static, human-readable description of a status code. */
const char *mha_strerror(int status);

/*
 * mha_device_status - synchronise `stream`, then read (and, if `reset` is
 * non-zero, clear) the current device's status word, which records a
 * device-side wait that ran out (every wait in the kernel is bounded).
 * Returns MHA_OK, MHA_ERR_TIMEOUT, or MHA_ERR_CUDA if the read failed.
 * `detail`, if non-NULL, receives the raw status word (0 when clean).
 */
int mha_device_status(void *stream, int reset, unsigned *detail);

/*
 * mha_fwd_tile_order - which work order mha_fwd uses for a shape; host
 * only, no CUDA call.  *order = 0: the default order (work tiles of 256
 * query rows, heads fastest, causal m-blocks heaviest first, dealt to the
 * persistent CTAs in snake rounds); *order = 1: the head-major order (the
 * m-blocks of one head adjacent; under the causal mask a CTA takes m-blocks
 * M-1-i and i of a head together), which keeps the K/V of the few heads in
 * flight in L2.  mha_fwd picks 1 when d == 128, all heads' K/V
 * (2*B*H*N*d*2 bytes) exceed 96 MiB, and its rounds of equal work items
 * fill at least 95% of the grid's slots.  `sms` is the multiprocessor count
 * that mha_fwd takes from the current device (152 on a GB300).
 * Errors: MHA_ERR_INVALID_ARG for a negative size, sms <= 0, a null
 * `order` or the sizes mha_fwd rejects; MHA_ERR_UNSUPPORTED_DIM unless d
 * is 64 or 128.
 */
int mha_fwd_tile_order(int B, int H, int N, int d, int causal, int sms, int *order);

/*
 * mha_set_wait_limit - set the cycle budget of every device-side wait for
 * launches made after this call (default 2^31 SM cycles, about one second).
 * `cycles` must be > 0.  Affects only this process.
 */
int mha_set_wait_limit(long long cycles);

/*
 * mha_wait_selftest - launch one block that waits, with the same bounded
 * wait as the attention kernel, on a barrier that nothing completes, for
 * at most `cycles` SM cycles; then synchronise `stream` and report.
 * Returns MHA_ERR_TIMEOUT when the bounded wait gave up as designed (and
 * clears the status word it set), MHA_OK if it did not.
 */
int mha_wait_selftest(long long cycles, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MHA_FWD_H */
