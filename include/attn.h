/*
 * attn.h — C ABI of the GB300 (sm_103a) fused exact attention forward and
 * its gradient (attn_bwd, near the end).
 *
 * The operation (what every entry point below computes) is the one spelled
 * out step by step in "Profiling in PyTorch (Part 3): Attention is all you
 * profile", section "Naive attention":
 *
 *     scores = q · kᵀ;  scores *= scale;  scores.masked_fill(mask, −inf);
 *     attn = softmax(scores, dim=-1);  out = attn · v
 *
 * with the causal mask of that page's "Math backend" section (ones → tril:
 * key j > query i is masked) and scale = 1/√head_dim as in its
 * NaiveCausalAttention module.  It is computed the way the same page's "Why
 * flash attention exists" passage and the FlashAttention-2 blog
 * ("FlashAttention (Original)": tiling, reduced HBM reads/writes;
 * "FlashAttention-2 Optimizations" §2-§3: causal skip, parallelism over the
 * sequence) describe: K and V are walked in tiles with a running softmax and
 * the [S, S] score matrix never reaches HBM.  In addition each row's natural
 * logsumexp  lse[i] = ln Σ_{j unmasked} exp(scale · q_i · k_j)  is written
 * (the pages do not define it; this is the FlashAttention convention).
 *
 * Layout (the native [batch, heads, seq, head_dim] layout the cuDNN backend of
 * the same page consumes without transposes): q, k, v and out are contiguous
 * row-major bf16 tensors of shape [B, H, S, D]; lse is contiguous fp32
 * [B, H, S].  Query and key lengths are equal (S).
 *
 * Ownership: the caller owns every buffer.  The library keeps, per device and
 * until process exit: one pair of device status words (cudaMalloc'd on the
 * first call on that device), three streams and a few events for
 * attn_fwd_staged (created on its first call on that device), and the static
 * ATTN_NOALLOC_SCRATCH_BYTES array of attn_fwd_noalloc (part of the loaded
 * module on every GPU that loads the library).  Beyond that it allocates
 * nothing, keeps no reference to any buffer after a call returns, and never
 * synchronises the stream inside attn_fwd.  Entry points are thread-safe and
 * reentrant.
 *
 * Error behaviour: argument errors are reported before anything is launched
 * and nothing is written.  A failed launch returns ATTN_ERR_CUDA.  Every wait
 * inside the kernel is bounded; a wait that runs out records ATTN_ERR_TIMEOUT
 * in the device status word (read with attn_device_status) and the kernel
 * returns without trapping.
 */
#ifndef EXACT_ATTENTION_68_ATTN_H_
#define EXACT_ATTENTION_68_ATTN_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* NULL pointer, size < 1, overflow, scale not finite and > 0, causal not 0/1, aliasing */
  ATTN_ERR_UNSUPPORTED = 2,  /* head_dim not a multiple of 8 or above 256 (128 for the backward), or no sm_103a device */
  ATTN_ERR_MISALIGNED = 3,   /* a pointer not 16-byte aligned */
  ATTN_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed (launch, copy, tensor-map encode) */
  ATTN_ERR_TIMEOUT = 5,      /* a bounded in-kernel wait ran out (reported by attn_device_status) */
  ATTN_ERR_DEVICE_CHECK = 6  /* a debug build's in-kernel index check failed; the access was
                                skipped (reported by attn_device_status; release builds have
                                no such checks) */
} attn_status_t;

/* The 16-bit type of q, k, v, out (and dout, dq, dk, dv) for the _ex entry points. */
typedef enum {
  ATTN_BF16 = 0,  /* bfloat16: what every other entry point uses */
  ATTN_F16 = 1    /* IEEE half */
} attn_dtype_t;

/* The wait bound attn_fwd and attn_bwd use (nanoseconds per in-kernel wait). */
#define ATTN_DEFAULT_WAIT_TIMEOUT_NS 2000000000ull

/*
 * attn_fwd — fused attention forward on device buffers.
 *
 *   q, k, v  device pointers, bf16 [B, H, S, D] contiguous, 16-byte aligned (read only)
 *   out      device pointer, bf16 [B, H, S, D] contiguous, 16-byte aligned (written)
 *   lse      device pointer, fp32 [B, H, S] contiguous, 4-byte aligned (written)
 *   B, H, S  batch, heads, sequence length; each >= 1, B·H < 2^31, S < 2^31
 *   D        head dimension: a multiple of 8, at most 256 (the backward: at most
 *            128).  64, 128 and 256 run on kernels of that width; any other D
 *            runs on the next width up with the columns past D read as zero
 *            (exact: they add nothing to q·kᵀ), so it costs what that width costs
 *   scale    multiplier of q·kᵀ (normally 1/sqrt(D)); must be finite and > 0
 *   causal   1: mask key j > query i; 0: no mask
 *   stream   CUDA stream the work is enqueued on (0 = legacy default stream)
 *
 * Asynchronous: returns once the kernel is enqueued.  out/lse must not
 * overlap q, k, v or each other.
 */
ATTN_API attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                       int64_t B, int64_t H, int64_t S, int64_t D, float scale, int causal,
                       cudaStream_t stream);

/*
 * attn_fwd_staged — the same forward, fed from and returned to HOST memory.
 *
 * q_h, k_h, v_h (bf16 [B,H,S,D]) are copied host→device into the caller's
 * device buffers q_d, k_d, v_d; the forward runs on them writing out_d, lse_d;
 * out_d and lse_d are copied back to out_h (bf16 [B,H,S,D]) and lse_h (fp32
 * [B,H,S]).  The (b, h) slices are split into chunks (about 48 MB of inputs
 * each, at most 8) whose uploads, kernels and downloads overlap on three
 * streams the library keeps per device; that work starts after everything
 * already enqueued on `stream`, and `stream` waits for all of it, so the call
 * behaves as one stream-ordered operation on `stream`.  Pass page-locked host
 * memory for the copies to be asynchronous.  Returns after enqueueing; the
 * host results are valid once the stream is synchronised, and the host and
 * device buffers must not be touched by other work until then.  Same argument
 * rules as attn_fwd for the device side; host pointers must be non-NULL.
 * Staged calls on one device are enqueued one at a time (a lock).
 */
ATTN_API attn_status_t attn_fwd_staged(const void* q_h, const void* k_h, const void* v_h,
                              void* out_h, float* lse_h,
                              void* q_d, void* k_d, void* v_d, void* out_d, float* lse_d,
                              int64_t B, int64_t H, int64_t S, int64_t D, float scale,
                              int causal, cudaStream_t stream);

/*
 * attn_fwd_bounded — attn_fwd with an explicit bound on every in-kernel wait.
 *
 * wait_timeout_ns bounds each wait of the kernel on a pipeline barrier
 * (attn_fwd uses 2 s).  When a wait runs out the kernel records
 * ATTN_ERR_TIMEOUT in the device status word, every role leaves its loop,
 * waits (bounded) for its own copies and tensor-core work in flight, frees its
 * tensor memory and returns.  A bound of 0 makes the first wait that is not
 * already satisfied run out: this is how the timeout path is tested.
 */
ATTN_API attn_status_t attn_fwd_bounded(const void* q, const void* k, const void* v, void* out,
                               float* lse, int64_t B, int64_t H, int64_t S, int64_t D,
                               float scale, int causal, uint64_t wait_timeout_ns,
                               cudaStream_t stream);

/*
 * attn_device_status — synchronise `stream`, then read and clear the status
 * word of the current device.  Returns ATTN_OK, ATTN_ERR_DEVICE_CHECK (a kernel
 * of a debug build recorded a failed index check since the last read),
 * ATTN_ERR_TIMEOUT (a kernel on this device recorded a timeout since the last
 * read) or ATTN_ERR_CUDA.
 */
ATTN_API attn_status_t attn_device_status(cudaStream_t stream);

/*
 * attn_fwd_noalloc — attn_fwd for callers that must not allocate device memory.
 *
 * The pages have no counterpart to this entry point.  It exists for programs
 * whose device memory belongs to their own allocator (memory reserved up front
 * and handed out in slices), code held to a fixed device-memory budget, and
 * latency-critical paths that may not pay for cudaMalloc, which can
 * synchronise the whole device.  attn_fwd allocates its device status words
 * with cudaMalloc on its first call on each device; this entry point keeps
 * them in a static device array of ATTN_NOALLOC_SCRATCH_BYTES instead, held
 * by every GPU that loads the library until the process exits, and calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * Arguments, layout, ownership and argument errors are those of attn_fwd.
 * check_status: 1 = also synchronise `stream` and return ATTN_ERR_TIMEOUT if
 * this call's kernel recorded a wait that ran out (ATTN_ERR_DEVICE_CHECK for a
 * failed index check of a debug build).  A stream that is being captured into
 * a graph cannot be synchronised, so check_status = 1 on such a stream is
 * rejected with ATTN_ERR_INVALID_ARG before anything is enqueued.
 * 0 = return once enqueued, giving up that report: no entry point reads the
 * static array's status words (attn_device_status reads attn_fwd's), the next
 * call clears them, and a kernel whose wait ran out may have left out and lse
 * partly written without the caller learning of it.
 * The scratch this kernel needs (two status words, 8 bytes) does not grow with
 * B, H, S or D.  The array's size is fixed when the library is built, and the
 * build checks that the kernel's need fits it.
 *
 * The first call on a device sets that device up (looks up the device address
 * of the array with the device current); make that first call before any
 * stream capture.  Every call on a device shares the one array and clears it
 * (cudaMemsetAsync on `stream`) before its kernel starts: calls whose work
 * overlaps on the GPU (different streams, or another host thread) race on it,
 * and a status read may then belong to another call.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES 256
ATTN_API attn_status_t attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out,
                                        float* lse, int64_t B, int64_t H, int64_t S, int64_t D,
                                        float scale, int causal, int check_status,
                                        cudaStream_t stream);

/*
 * attn_bwd — gradient of attn_fwd with respect to q, k and v.
 *
 * The pages define the forward only; the same profiling page's passage on
 * in-place operations notes that the backward reuses what the forward saved.
 * For an upstream gradient dout = ∂L/∂out this computes the exact gradient of
 * the five forward steps (chain rule in reverse): with P the attention weights
 * recomputed from the saved lse, dP = dout·vᵀ and
 * delta_i = Σ_d dout[i,d]·out[i,d],
 *
 *     dS = P ⊙ (dP − delta),  dq = scale·dS·k,  dk = scale·dSᵀ·q,  dv = Pᵀ·dout.
 *
 *   q, k, v     the forward's inputs, device bf16 [B, H, S, D], 16-byte aligned (read)
 *   out, lse    the forward's results for those inputs: out bf16 [B, H, S, D]
 *               (16-byte aligned), lse fp32 [B, H, S] (4-byte aligned) (read)
 *   dout        device bf16 [B, H, S, D], 16-byte aligned (read)
 *   dq, dk, dv  device bf16 [B, H, S, D], 16-byte aligned (written)
 *   delta       device fp32 [B, H, S], 4-byte aligned: workspace the call
 *               writes (rowsum(dout ⊙ out)) and reads back; its contents after
 *               the call are that rowsum
 *   B, H, S, D, scale, causal, stream   as for attn_fwd (the same values the
 *               forward used)
 *
 * Two kernels are enqueued on `stream` (dq and delta, then dk and dv); each
 * gradient row is written by exactly one CTA, with no atomics, so results are
 * bitwise reproducible.  Asynchronous; allocates nothing beyond the status
 * word attn_fwd also uses.  Outputs must not overlap each other or any input.
 * Errors as attn_fwd; a wait that runs out is reported by attn_device_status.
 */
ATTN_API attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* out,
                                const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                float* delta, int64_t B, int64_t H, int64_t S, int64_t D,
                                float scale, int causal, cudaStream_t stream);

/* attn_bwd with an explicit bound on every in-kernel wait (see attn_fwd_bounded). */
ATTN_API attn_status_t attn_bwd_bounded(const void* q, const void* k, const void* v,
                                        const void* out, const float* lse, const void* dout,
                                        void* dq, void* dk, void* dv, float* delta, int64_t B,
                                        int64_t H, int64_t S, int64_t D, float scale, int causal,
                                        uint64_t wait_timeout_ns, cudaStream_t stream);

/*
 * attn_fwd_ex / attn_bwd_ex — attn_fwd_bounded / attn_bwd_bounded for a chosen
 * 16-bit type.  With dtype = ATTN_F16 every 16-bit tensor (q, k, v, out; for
 * the backward also dout, dq, dk, dv) holds IEEE half values, and the
 * tensor-core operands the kernels form from P and dS are rounded to half as
 * well; lse and delta stay fp32.  Layouts, ownership and errors as for the
 * bf16 entry points; a dtype other than ATTN_BF16 or ATTN_F16 is
 * ATTN_ERR_INVALID_ARG.  Pass ATTN_DEFAULT_WAIT_TIMEOUT_NS for the usual bound.
 */
ATTN_API attn_status_t attn_fwd_ex(const void* q, const void* k, const void* v, void* out,
                                   float* lse, int64_t B, int64_t H, int64_t S, int64_t D,
                                   float scale, int causal, attn_dtype_t dtype,
                                   uint64_t wait_timeout_ns, cudaStream_t stream);
ATTN_API attn_status_t attn_bwd_ex(const void* q, const void* k, const void* v, const void* out,
                                   const float* lse, const void* dout, void* dq, void* dk,
                                   void* dv, float* delta, int64_t B, int64_t H, int64_t S,
                                   int64_t D, float scale, int causal, attn_dtype_t dtype,
                                   uint64_t wait_timeout_ns, cudaStream_t stream);

/*
 * attn_shard_range — the (batch, head) slices that rank `rank` of `world`
 * processes takes when one forward is split over several GPUs, one process
 * per GPU.
 *
 * The FlashAttention-2 blog ("FlashAttention-2 Optimizations" §3) parallelises
 * the forward over batch and heads (and the sequence); every (b, h) slice is
 * computed from its own q, k, v rows alone, so a split over processes needs no
 * exchange of data between them.  Slices are numbered b·H + h (the order of
 * the [B, H, S, D] layout); rank r takes the contiguous range
 * [*first, *first + *count), the first (units mod world) ranks one slice more
 * than the others, so the ranges of ranks 0 .. world-1 cover 0 .. units-1
 * once, in order.  A rank's slices of a contiguous [B, H, S, D] tensor are
 * themselves a contiguous [count, S, D] tensor starting at element
 * first·S·D: attn_fwd with B = 1, H = count on pointers offset that
 * far computes exactly those slices.  A rank may get no slice (count 0) when
 * world > units.
 *
 *   units        number of slices, B·H (>= 0)
 *   world, rank  number of processes (>= 1) and this process's index in [0, world)
 *   first, count outputs (host pointers)
 *
 * Host-only arithmetic: no CUDA call, no allocation.  Returns
 * ATTN_ERR_INVALID_ARG (outputs untouched) for units < 0, world < 1, rank
 * outside [0, world) or a NULL output pointer.
 */
ATTN_API attn_status_t attn_shard_range(int64_t units, int world, int rank, int64_t* first,
                                        int64_t* count);

/* Static, human-readable name of a status code. */
ATTN_API const char* attn_status_string(attn_status_t status);

/*
 * The cause of the most recent ATTN_ERR_CUDA returned on the calling thread:
 * the cudaError_t of the call that failed, or -1 when a TMA tensor map could
 * not be encoded; 0 if no such error has been returned on this thread.
 */
ATTN_API int attn_last_cuda_error(void);

/* ABI version of this library (incremented on any signature change). */
ATTN_API int attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTENTION_68_ATTN_H_ */
