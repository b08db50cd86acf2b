/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused attention forward.
 *
 * The operation (one call):
 *
 *     O   = softmax(Q K^T * sm_scale + mask) V
 *     lse = log(sum_j exp(sm_scale * q_i . k_j))   over the attended keys j
 *
 * over Q, K, V of shape [B, H, L, D].  The masks are the three the source
 * pages define:
 *   ATTN_MASK_DENSE       every key is attended (the "Triton-CUDA Attention"
 *                         page, standard Flash Attention example);
 *   ATTN_MASK_CAUSAL      key j is attended by query i iff j <= i (the
 *                         "Fused Attention" page, stage-2 mask, top-left
 *                         aligned, L_q = L_k);
 *   ATTN_MASK_BLOCK_DIAG  key j is attended by query i iff floor(j/bs) ==
 *                         floor(i/bs): only the diagonal bs x bs blocks of the
 *                         L x L attention matrix take part (the "TLX Block
 *                         Attention" page, block-diagonal definition).
 * The computation is tiled with the online-softmax recurrence (the
 * "Triton-CUDA Attention" page, online softmax section), so the L x L matrix
 * is never written to memory.  lse is the natural-log log-sum-exp of the
 * scaled scores (the "Fused Attention" page, epilogue m_i += log(l_i)).
 *
 * Layout: q, k, v and o are contiguous row-major [B, H, L, D] arrays of the
 * element type `dtype` (fp16 or bf16), D innermost; lse is a contiguous fp32
 * [B, H, L] array.  All five pointers are DEVICE pointers on the current CUDA
 * device, each 16-byte aligned.  The caller owns every buffer; the library
 * never allocates, frees or retains them.
 */
#ifndef ATTN_FWD_GB300_ATTN_H
#define ATTN_FWD_GB300_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_MASK_DENSE = 0,
    ATTN_MASK_CAUSAL = 1,
    ATTN_MASK_BLOCK_DIAG = 2
} attn_mask_kind;

typedef enum {
    ATTN_F16 = 0,
    ATTN_BF16 = 1
} attn_dtype;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_NULL = 1,          /* a required pointer is NULL                        */
    ATTN_ERR_SHAPE = 2,         /* B, H or L negative, or a size overflows           */
    ATTN_ERR_BLOCK_SIZE = 3,    /* block-diagonal: bs <= 0 or bs does not divide L   */
    ATTN_ERR_UNSUPPORTED = 4,   /* head_dim, dtype, mask kind or bs not supported    */
    ATTN_ERR_ALIGN = 5,         /* a pointer is not 16-byte aligned                  */
    ATTN_ERR_CUDA = 6,          /* a CUDA runtime/driver call failed                 */
    ATTN_ERR_TIMEOUT = 7,       /* a device-side pipeline wait ran out (see below)   */
    ATTN_ERR_ARG = 8            /* sm_scale not finite, or another bad argument      */
} attn_status;

/*
 * attn_fwd -- enqueue one fused attention forward on `stream`.
 *
 *   q, k, v     inputs, [B, H, L, D] of `dtype`, device memory, read only.
 *   o           output, [B, H, L, D] of `dtype`, device memory, fully written.
 *   lse         output, [B, H, L] fp32, device memory; may be NULL (not written).
 *   B, H, L     batch, heads, sequence length (queries = keys = L).  A zero
 *               size is an empty problem: ATTN_OK, nothing is launched.
 *   D           head dim: a multiple of 8 from 8 to 256.  Kernels exist for
 *               64, 128 and 256; any other D runs in the next one up, the
 *               columns past D loading as zeros (same results, the MMA work of
 *               the larger head dim).
 *   mask_kind   an attn_mask_kind.
 *   block_size  the block size bs of ATTN_MASK_BLOCK_DIAG (ignored otherwise);
 *               bs must divide L and be a divisor or a multiple of 128.
 *   sm_scale    the score scale (the pages use 1/sqrt(D)); any finite value.
 *   dtype       an attn_dtype.
 *   stream      a cudaStream_t (NULL = the legacy default stream).
 *
 * Returns ATTN_OK once the kernel is enqueued; the outputs are valid after
 * the stream is synchronised.  The kernel is launched as a programmatic
 * dependent of the previous kernel on `stream` (its CTAs may be scheduled
 * while that kernel finishes, but they wait for its completion before any
 * global memory access), so stream ordering is unchanged for the caller.
 * Argument errors are detected on the host before any CUDA call
 * (attn_fwd_check runs the same checks alone) and nothing is launched or
 * written.  A failed launch returns ATTN_ERR_CUDA.  Every wait inside the
 * kernel is bounded (about one second); if one runs out the kernel stops,
 * frees its tensor memory and records ATTN_ERR_TIMEOUT in a per-device status
 * word that attn_last_device_status() reads.  Reentrant; safe from several
 * host threads.
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             int B, int H, int L, int D, int mask_kind, int block_size,
             float sm_scale, int dtype, void *stream);

/*
 * attn_fwd_work -- the algorithmic work of one attn_fwd call, for throughput
 * and roofline figures.  flops = 4 * D * (attended (i, j) pairs summed over
 * B*H heads): two flops per multiply-add, for both Q K^T and P V; masked pairs
 * are not counted.  bytes = Q, K and V read once plus O written once
 * (4 * B*H*L*D * element size); lse bytes are not counted.  Either output
 * pointer may be NULL.  Returns an attn_status (same validation as attn_fwd).
 */
int attn_fwd_work(int B, int H, int L, int D, int mask_kind, int block_size,
                  int dtype, double *flops, double *bytes);

/*
 * attn_fwd_check -- the host-side argument checks of attn_fwd (and of
 * attn_fwd_noalloc, which runs the same ones), alone: the same arguments
 * without the stream, the same status attn_fwd would return before any CUDA
 * call (ATTN_OK for an empty problem or for arguments that pass).  It makes no
 * CUDA call and never reads or writes through the pointers, which are only
 * tested for NULL and for 16-byte alignment; so a caller (or a test) may
 * check arguments on a machine without a GPU, or with addresses that are not
 * allocated, without anything being launched.
 */
int attn_fwd_check(const void *q, const void *k, const void *v, const void *o, const float *lse,
                   int B, int H, int L, int D, int mask_kind, int block_size,
                   float sm_scale, int dtype);

/* Human-readable name of an attn_status (static storage; never NULL). */
const char *attn_status_string(int status);

/*
 * attn_last_device_status -- read and clear the device status word of CUDA
 * device `device` (the word in-kernel timeouts write).  Synchronises that
 * device first.  *status receives ATTN_OK, ATTN_ERR_TIMEOUT, or ATTN_ERR_CUDA
 * when a kernel found its tensor memory somewhere it cannot be (and did no
 * work); *detail (may be NULL) receives the raw word (the wait site of the
 * first timeout in bits 8-15).
 * Returns an attn_status for the query itself.
 */
int attn_last_device_status(int device, int *status, unsigned int *detail);

/*
 * attn_fwd_noalloc -- attn_fwd for callers that may not allocate device
 * memory: a serving runtime that reserves its whole memory budget at start-up
 * and forbids later allocations, or a host framework whose own pool must stay
 * the only owner of device memory.  (The source pages have no counterpart;
 * this entry point exists for such callers only.)
 *
 * Same arguments, layout and results as attn_fwd.  attn_fwd keeps its
 * device status word in memory the library cudaMallocs on the first call on
 * each device; this variant instead keeps it in a fixed 256-byte array
 * compiled into the library (ATTN_NOALLOC_SCRATCH_BYTES per device, held by
 * every GPU that loads the library until the process exits), and calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 *   status_out  optional HOST pointer (may be NULL).  If given, the device
 *               status word of this call (0, or an attn_status in its low
 *               byte, as attn_last_device_status reports) is copied there on
 *               `stream`; read it after the stream is synchronised (pinned
 *               memory keeps the copy asynchronous).
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and clears it; make that first call before any
 * stream capture.  Every call clears the status word on `stream` and then
 * launches.  All calls share the one array, so calls that overlap on the GPU
 * (different streams, no ordering) race on the status word.  The scratch a
 * call needs does not grow with the problem (one 32-bit word); a call that
 * would need more than the array holds is refused with ATTN_ERR_UNSUPPORTED.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES 256
int attn_fwd_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int H, int L, int D, int mask_kind, int block_size,
                     float sm_scale, int dtype, void *stream, unsigned int *status_out);

/*
 * attn_fwd_fp8v -- the FP8 P.V variant of the "Fused Attention" page: V is
 * given in float8 e5m2 and transposed, P is rounded to e5m2 before the P.V
 * product (which runs on the tensor cores in 8-bit), and the softmax
 * denominator sums the unrounded weights.  P is rounded against the exact
 * running max of the key tiles seen so far (128 keys a tile, in order), as in
 * the page's recurrence.
 *
 *   vt          V^T: [B, H, D, L] float8 e5m2 bytes (keys innermost), device
 *               memory, 16-byte aligned.
 *   the rest    as for attn_fwd (q, k fp16/bf16 [B, H, L, D]; o in their type).
 *
 * L must be a multiple of 16 (each V^T row is L bytes, and TMA needs row
 * strides in multiples of 16 bytes): other L give ATTN_ERR_UNSUPPORTED.
 * Same errors, timeouts and stream behaviour as attn_fwd otherwise.
 */
int attn_fwd_fp8v(const void *q, const void *k, const void *vt, void *o, float *lse,
                  int B, int H, int L, int D, int mask_kind, int block_size,
                  float sm_scale, int dtype, void *stream);

/* The host-side argument checks of attn_fwd_fp8v alone (as attn_fwd_check:
 * no CUDA call, the pointers never dereferenced). */
int attn_fwd_fp8v_check(const void *q, const void *k, const void *vt, const void *o,
                        const float *lse, int B, int H, int L, int D, int mask_kind,
                        int block_size, float sm_scale, int dtype);

/*
 * attn_fwd_host -- the whole forward for inputs and outputs in HOST memory:
 * copies q, k, v to the device, runs attn_fwd, copies o (and lse) back and
 * synchronises `stream` before returning, so the host outputs are valid on
 * return.
 *
 *   q_h, k_h, v_h   host inputs, [B, H, L, D] of `dtype` (page-locked memory
 *                   keeps the copies asynchronous and at full speed).
 *   o_h             host output, [B, H, L, D] of `dtype`.
 *   lse_h           host output, [B, H, L] fp32; may be NULL.
 *   q_d, k_d, v_d, o_d, lse_d
 *                   device buffers of the same shapes that the caller owns and
 *                   may reuse across calls (lse_d may be NULL when lse_h is).
 *   the rest        as for attn_fwd.
 *
 * The B*H heads are cut into chunks (attn_fwd_host_chunks) that flow through
 * three stages at once: the library's copy-in stream copies chunk c+1's q, k, v
 * while `stream` runs the forward of chunk c and the library's copy-out stream
 * copies chunk c-1's o and lse back.  Both copy streams start after the work
 * already queued on `stream`, and `stream` waits for both before the call
 * synchronises it.  Each chunk's forward is attn_fwd over that chunk's heads;
 * the results are those of one attn_fwd over all of them (no mask depends on
 * the head).  Calls from several host threads are serialised while they
 * enqueue.  Returns an attn_status: argument errors as attn_fwd (plus
 * ATTN_ERR_NULL for a missing host or device buffer) before any copy;
 * ATTN_ERR_CUDA if a copy, a launch or the synchronisation fails (the copies
 * already queued still finish before the call returns).  A device-side timeout
 * is read with attn_last_device_status, as for attn_fwd.
 */
int attn_fwd_host(const void *q_h, const void *k_h, const void *v_h, void *o_h, float *lse_h,
                  void *q_d, void *k_d, void *v_d, void *o_d, float *lse_d,
                  int B, int H, int L, int D, int mask_kind, int block_size,
                  float sm_scale, int dtype, void *stream);

/* The chunking attn_fwd_host uses on a device with `sms` SMs: heads per
 * chunk and number of chunks (both 0 for an empty problem).  Pure host
 * arithmetic, no CUDA call: the count minimises a three-stage pipeline model
 * (copy in, forward, copy out) with rates measured on GB300, at most 16
 * chunks.  Returns ATTN_ERR_ARG for sms <= 0, else as attn_fwd_check's shape
 * checks. */
int attn_fwd_host_chunks(int B, int H, int L, int D, int mask_kind, int block_size, int dtype, int sms,
                         int *heads_per_chunk, int *chunks);

/* Number of work units and CTAs attn_fwd would launch for these arguments on
 * the current device (for tests and reports); returns an attn_status. */
int attn_fwd_plan(int B, int H, int L, int D, int mask_kind, int block_size,
                  int dtype, int *units, int *ctas, int *threads, int *smem_bytes);

/*
 * attn_debug_inject -- TEST HOOK, not for production use.  mode 1 makes every
 * following attn_fwd or attn_bwd kernel start with its copy-issuing warp doing nothing, so
 * each consumer's bounded wait runs out after about one second: the kernel
 * records ATTN_ERR_TIMEOUT in the device status word, frees its tensor memory
 * and returns (outputs undefined), without hanging the GPU.  mode 0 restores
 * normal operation.  Process-wide, not thread-safe; attn_fwd_noalloc ignores it.
 */
int attn_debug_inject(int mode);

/*
 * attn_bwd -- enqueue the backward of attn_fwd on `stream`: the gradients of
 * sum(dout * O) with respect to q, k and v, for the same mask, block size and
 * sm_scale, from the forward's o and lse (the "Fused Attention" page saves
 * exactly these for a backward it does not define; the gradients follow from
 * the definition above by the chain rule through the softmax):
 *
 *     P  = exp(sm_scale Q K^T - lse)  (0 outside the mask),  Di = dout_i . o_i
 *     dv = P^T dout,   dS = P * (dout v^T - Di),
 *     dq = sm_scale dS k,   dk = sm_scale dS^T q
 *
 *   q, k, v, o, dout  [B, H, L, D] of `dtype`, device memory, read only
 *                     (o and lse as attn_fwd wrote them).
 *   lse               [B, H, L] fp32, device memory, read only.
 *   dq, dk, dv        outputs, [B, H, L, D] of `dtype`, device memory, fully
 *                     written (no accumulation into them; no atomics, so the
 *                     results are deterministic).
 *   workspace         device scratch of at least attn_bwd_workspace_size(B, H,
 *                     L) bytes, 16-byte aligned, owned by the caller, free for
 *                     reuse once the call's work on `stream` has completed.
 *   D                 a multiple of 8 from 8 to 256 (kernels for 64, 128 and
 *                     256; other D run zero-padded to the next of these);
 *                     other arguments as for attn_fwd.
 * Every pointer must be 16-byte aligned (ATTN_ERR_ALIGN otherwise).
 *
 * Three kernels: the row-statistics kernel and the dK/dV kernel on `stream`,
 * the dQ kernel (which needs only the former) on a second stream the library
 * owns, forked from `stream` after the row-statistics kernel and joined back
 * into it before the call returns, so work enqueued on `stream` afterwards
 * waits for all three.  The fork and join use events and are valid inside
 * stream capture; concurrent calls serialise only their enqueueing.
 * Returns ATTN_OK once enqueued;
 * ATTN_ERR_ARG if workspace_bytes is too small or sm_scale is not finite;
 * argument errors as attn_fwd, all before any CUDA call; device-side
 * timeouts are reported through attn_last_device_status.
 */
int attn_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
             const float *lse, void *dq, void *dk, void *dv, void *workspace,
             size_t workspace_bytes, int B, int H, int L, int D, int mask_kind,
             int block_size, float sm_scale, int dtype, void *stream);

/* The host-side argument checks of attn_bwd alone (as attn_fwd_check: no
 * CUDA call, the pointers never dereferenced). */
int attn_bwd_check(const void *q, const void *k, const void *v, const void *o, const void *dout,
                   const float *lse, const void *dq, const void *dk, const void *dv,
                   const void *workspace, size_t workspace_bytes, int B, int H, int L, int D,
                   int mask_kind, int block_size, float sm_scale, int dtype);

/* Bytes of workspace attn_bwd needs: two fp32 values per row, rows padded to
 * whole 128-row tiles per head (0 for negative sizes). */
size_t attn_bwd_workspace_size(int B, int H, int L);

/* Algorithmic work of one attn_bwd: flops = 2.5 x the forward's (five
 * products of its size: S, dP, dV, dK, dQ), bytes = q, k, v, o, dout read and
 * dq, dk, dv written once, plus lse; returns an attn_status. */
int attn_bwd_work(int B, int H, int L, int D, int mask_kind, int block_size, int dtype,
                  double *flops, double *bytes);

/* ABI version of this header: (major << 16) | minor. */
int attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FWD_GB300_ATTN_H */
