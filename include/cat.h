/*
 * cat.h — C ABI of the GB300 CAT library (libcat.so): the forward pass, its
 * backward pass, and the 2-D (BCCB) circulant attention of a second page.
 *
 * CAT (circular-convolutional attention), as defined on the notes page
 * "CAT: Circular-Convolutional Attention for Sub-Quadratic Transformers",
 * section 方法详解 (method):
 *   - 整体框架 (overall framework): CAT replaces multi-head self-attention;
 *     its parameters are W_A (attention projection, one column per head) and
 *     W_V (value projection).  V = X·W_V is an INPUT here: the value
 *     projection is an ordinary dense GEMM and is not part of this library.
 *   - 关键设计, "circulant attention matrix construction": per head h,
 *     Z = X·W_A[:, h], Z* = softmax over the N tokens, and circ(Z*) is the
 *     N x N circulant whose rows are successive cyclic shifts.
 *   - 关键设计, "FFT acceleration": circ(Z*)·V = IFFT(FFT(Z*) ⊙ FFT(V)),
 *     exact, O(N log N); this orientation gives circ(Z*)[i,j] = Z*[(i-j) mod N].
 *
 * Data layout (all dense, row-major, caller-owned device memory unless a
 * function says otherwise):
 *   X   [B, N, D]   tokens
 *   W_A [D, H]      one score column per head
 *   V   [B, N, D]   projected values; head h owns columns [h·D/H, (h+1)·D/H)
 *   O   [B, N, D]   output, same layout as V
 *   z*  [B, H, N]   fp32 softmax weights (only from cat_forward_zstar)
 * X, W_A, V and O all have the plan's dtype.  All arithmetic is fp32:
 * bf16 inputs are widened exactly, bf16 outputs are rounded to nearest-even.
 *
 * Every function returns a cat_status (0 = CAT_OK, negative = error) and
 * never aborts, exits or traps.  GPU work is enqueued asynchronously on the
 * plan's stream; errors raised by kernels are reported by cat_plan_sync.
 */
#ifndef CAT_H_
#define CAT_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque plan: shape, dtype, stream, device workspace, twiddle tables. */
typedef struct cat_plan_s *cat_plan_t;

/* Storage type of X, W_A, V and O. */
typedef enum { CAT_F32 = 0, CAT_BF16 = 1 } cat_dtype_t;

/* Status codes. */
enum {
  CAT_OK = 0,
  CAT_ERR_INVALID_ARG = -1,   /* bad shape, null pointer, D % H != 0, ...   */
  CAT_ERR_UNSUPPORTED_N = -2, /* N has a prime factor > 7 or exceeds limits */
  CAT_ERR_MISALIGNED = -3,    /* a device pointer is not 16-byte aligned    */
  CAT_ERR_PLAN_MISMATCH = -4, /* call shape/dtype differs from the plan's   */
  CAT_ERR_ALLOC = -5,         /* device or host allocation failed           */
  CAT_ERR_CUDA = -6,          /* a CUDA runtime call or launch failed       */
  CAT_ERR_DEVICE_STATUS = -7, /* a kernel reported an internal check failure*/
  CAT_ERR_ALIAS = -8,         /* O overlaps X, W_A or V                     */
  CAT_ERR_TOO_LARGE = -9      /* beyond cat_forward_noalloc's fixed workspace */
};

/* Size limits of the library. */
#define CAT_MAX_N (1 << 22)   /* longest sequence                          */
#define CAT_MAX_D 8192        /* widest model dimension                    */

/*
 * cat_plan_create — validate a problem shape and build everything the
 * forward pass needs: the execution path (single-CTA shared-memory FFT for
 * N up to 16384, four-step multi-CTA FFT above), fp32 twiddle tables
 * computed in fp64 on the host, and the device workspace (scores, softmax
 * weights, their spectra, four-step scratch).  The plan owns that memory.
 *
 *   out    : receives the plan (set to NULL on failure)
 *   B      : batch size, >= 0 (B = 0 makes cat_forward a no-op)
 *   N      : sequence length, 1 <= N <= CAT_MAX_N, 7-smooth (only prime
 *            factors 2, 3, 5, 7)
 *   D, H   : model width and head count, 1 <= H <= D <= CAT_MAX_D, D % H == 0
 *   dtype  : CAT_F32 or CAT_BF16
 *   stream : cudaStream_t to enqueue on (NULL = legacy default stream); the
 *            caller keeps ownership and must keep it alive while the plan
 *            uses it.
 * Errors: CAT_ERR_INVALID_ARG, CAT_ERR_UNSUPPORTED_N, CAT_ERR_ALLOC,
 * CAT_ERR_CUDA.  Uses the CUDA device current at the call.
 */
int cat_plan_create(cat_plan_t *out, int B, int N, int D, int H, int dtype,
                    void *stream);

/*
 * cat_plan_query — the plan cat_plan_create would build for this shape,
 * without touching the device or allocating: *workspace_bytes (may be
 * NULL) receives the device workspace it would allocate, and desc (may be
 * NULL; capacity len bytes, NUL-terminated, truncated if needed) the same
 * one-line description cat_plan_describe gives (path, factorisation,
 * launch shapes).  The backward workspace, allocated at a plan's first
 * backward call, is not included.  Errors: those of cat_plan_create's
 * shape validation (CAT_ERR_INVALID_ARG, CAT_ERR_UNSUPPORTED_N).
 */
int cat_plan_query(int B, int N, int D, int H, int dtype,
                   size_t *workspace_bytes, char *desc, int len);

/* Release a plan and its device memory.  NULL is accepted (no-op).
 * Synchronises the plan's stream first.  Destroying twice is undefined. */
int cat_plan_destroy(cat_plan_t plan);

/* Change the stream later calls enqueue on. */
int cat_plan_set_stream(cat_plan_t plan, void *stream);

/*
 * cat_forward — O = CAT(X, W_A, V) for every batch and head (both designs
 * of the notes page cited above): scores, softmax over tokens, spectrum of
 * z* once per (b, h), then per value column IFFT(FFT(z*) ⊙ FFT(v)).
 *
 * X, W_A, V: device pointers, read only.  O: device pointer, written.
 * All four must be 16-byte aligned and O must not overlap the others.
 * B, N, D, H, dtype must equal the plan's (CAT_ERR_PLAN_MISMATCH).
 * Asynchronous on the plan's stream: work that the fast long-sequence path
 * (head width 64, N = 512·N2 with N2 in 32..256) spreads over the plan's two
 * internal streams forks from and joins back into the plan's stream, so the
 * call is ordered like a single kernel on it.  The plan's workspace is
 * reused, so two calls on one plan must not run concurrently on different
 * streams.
 */
int cat_forward(cat_plan_t plan, const void *X, const void *W_A, const void *V,
                void *O, int B, int N, int D, int H, int dtype);

/*
 * cat_forward_fused — the value projection and the scores from one pass
 * over X, then the forward: V = X·W_V (written to V) and z = X·W_A from the
 * same tensor-core GEMM [V | z] = X·[W_V | W_A] (the notes page cited
 * above, 整体框架 overall framework: a CAT layer projects X with W_V for
 * the values and W_A for the scores), then O = CAT(X, W_A, V) exactly as
 * cat_forward computes it from those V and z.
 *
 * X [B, N, D], W_V [D, D] (row-major, V[b, n, :] = X[b, n, :]·W_V) and
 * W_A [D, H]: device pointers, read only.  V and O [B, N, D]: device
 * pointers, written.  bf16 only (CAT_ERR_INVALID_ARG otherwise), D a
 * multiple of 64, H <= 16; products of bf16 values are exact, accumulation
 * fp32; V is rounded to bf16 (nearest even); the scores are kept as
 * double-float sums of 64-wide fp32 slices.  All pointers 16-byte aligned;
 * V and O must not overlap the inputs or each other (CAT_ERR_ALIAS).  The
 * first call allocates the plan's transposed-weight workspace (2·D·(D+16)
 * bytes; CAT_ERR_ALLOC).  Asynchronous on the plan's stream.
 */
int cat_forward_fused(cat_plan_t plan, const void *X, const void *W_V,
                      const void *W_A, void *V, void *O, int B, int N, int D,
                      int H, int dtype);

/*
 * cat_project — the fused projection alone: V = X·W_V (written to V) and
 * z* = softmax over the tokens of X·W_A (fp32 [B, H, N], written to the
 * device pointer zstar), from the same one-pass tensor-core GEMM as
 * cat_forward_fused.  Arguments, limits and errors as cat_forward_fused;
 * zstar must not overlap X or V (CAT_ERR_ALIAS).
 */
int cat_project(cat_plan_t plan, const void *X, const void *W_V, const void *W_A,
                void *V, float *zstar, int B, int N, int D, int H, int dtype);

/*
 * cat_forward_zstar — only the first two steps (score projection and
 * softmax over the N tokens, "circulant attention matrix construction"):
 * writes z* as fp32 [B, H, N] to the device pointer zstar (16-byte aligned).
 */
int cat_forward_zstar(cat_plan_t plan, const void *X, const void *W_A,
                      float *zstar, int B, int N, int D, int H, int dtype);

/*
 * cat_forward_host — the same forward on HOST buffers, copies included: X,
 * W_A, V are read from host memory and O is written to host memory before
 * the call returns (it synchronises).  With B >= 2 the call runs one batch
 * per step and overlaps the copies with the compute: batch b's inputs copy
 * in on one internal stream while batch b - 1 computes on the plan's stream
 * and batch b - 2's output copies out on another.  The first call sets up
 * plan-owned device staging (two batches' worth, or the whole problem when
 * B = 1), two internal one-batch plans and the copy streams, which the plan
 * keeps; CAT_ERR_ALLOC if that fails.  Pinned (page-locked) host memory is
 * needed for the copies to overlap; pageable memory works but serialises.
 * Kernel status of the internal plans is reported by cat_plan_sync.
 */
int cat_forward_host(cat_plan_t plan, const void *X, const void *W_A,
                     const void *V, void *O, int B, int N, int D, int H,
                     int dtype);

/*
 * cat_backward — gradients of a loss L through the forward pass, given the
 * upstream gradient dO = dL/dO.  The notes page cited above trains CAT
 * layers with the usual losses and optimisers (section 损失函数 / 训练策略,
 * loss and training strategy) but prints no gradients; these follow from
 * the forward definitions by the chain rule, per (b, h):
 *   dV   = circ(z*)^T dO          dV[j, c] = sum_i z*[(i - j) mod N] dO[i, c]
 *   dz*[k] = sum_{c in h} sum_i dO[i, c] V[(i - k) mod N, c]
 *          = Re IFFT( sum_c FFT(dO[:, c]) ⊙ conj(FFT(V[:, c])) )
 *   dz   = z* ⊙ (dz* - <z*, dz*>)  (softmax Jacobian)
 *   dW_A[d, h] = sum_{b, n} X[b, n, d] dz[b, h, n]
 *   dX[b, n, d] = sum_h dz[b, h, n] W_A[d, h]
 * z* is recomputed from X and W_A (nothing is kept from a forward call).
 *
 * X, W_A, V, dO: device pointers, read only ([B,N,D], [D,H], [B,N,D],
 * [B,N,D]).  dX [B,N,D], dW_A [D,H], dV [B,N,D]: device pointers, written;
 * dW_A is overwritten, not accumulated into.  All seven have the plan's
 * dtype (bf16 gradients are rounded to nearest-even from fp32), must be
 * 16-byte aligned (CAT_ERR_MISALIGNED), and no output may overlap an input
 * or another output (CAT_ERR_ALIAS).  Shape arguments must equal the plan's.
 * The first call configures and allocates the plan's backward workspace
 * (correlation scratch, dz*, dz, dW_A partial sums), which the plan keeps;
 * CAT_ERR_ALLOC if that fails.  Asynchronous on the plan's stream; the
 * plan's forward workspace is reused, so a backward and a forward on one
 * plan must not run concurrently on different streams.
 */
int cat_backward(cat_plan_t plan, const void *X, const void *W_A, const void *V,
                 const void *dO, void *dX, void *dW_A, void *dV, int B, int N,
                 int D, int H, int dtype);

/*
 * cat_backward_dz — only the score-side gradients of cat_backward: writes
 * dz* = dL/dz* and dz = dL/dz (the softmax backward of dz*), each fp32
 * [B, H, N], to the device pointers dzstar and dz (16-byte aligned, not
 * overlapping the inputs or each other: CAT_ERR_ALIAS).  Inputs and errors
 * as for cat_backward.
 */
int cat_backward_dz(cat_plan_t plan, const void *X, const void *W_A,
                    const void *V, const void *dO, float *dzstar, float *dz,
                    int B, int N, int D, int H, int dtype);

/*
 * 2-D circulant attention — the page "Vision Transformers are Circulant
 * Attention Learners": for tokens on an h x w grid (token n = y·w + x) the
 * attention map is modelled as a BCCB matrix (block circulant with
 * circulant blocks) with generator σ(a), so that O = σ(a) ⊛ V, a 2-D
 * circular convolution, computed with 2-D FFTs; a comes from Q and K by
 * FFTs and an element-wise product.  The page prints no formula for a; the
 * reading taken is the channel-averaged 2-D circular cross-correlation
 *     a[b, hd, k] = (1/dh) Σ_{c in head hd} Σ_i Q[b, i, c] · K[b, i ⊖ k, c]
 * (i ⊖ k: grid-wise difference mod (h, w)), σ the softmax over the N = h·w
 * lags, and O[b, i, c] = Σ_j σ(a)[b, hd(c), i ⊖ j] · V[b, j, c].
 *
 * cat_plan_create_2d — a plan for B batches on an h x w grid (1 <= h, w <=
 * 16384, each 7-smooth, h·w <= CAT_MAX_N), model width D, H heads, dtype,
 * stream; errors as cat_plan_create.  A 2-D plan serves only the cat2d_*
 * calls (the 1-D calls return CAT_ERR_PLAN_MISMATCH), and the cat2d_* calls
 * take only 2-D plans.  It allocates its whole workspace at creation.
 */
int cat_plan_create_2d(cat_plan_t *out, int B, int h, int w, int D, int H,
                       int dtype, void *stream);

/*
 * cat2d_forward — O = σ(a) ⊛ V for every batch and head.  Q, K, V: device
 * pointers [B, h·w, D], read only; O: device pointer [B, h·w, D], written;
 * all in the plan's dtype, 16-byte aligned, O not overlapping Q, K or V.
 * Asynchronous on the plan's stream.
 */
int cat2d_forward(cat_plan_t plan, const void *Q, const void *K, const void *V,
                  void *O, int B, int h, int w, int D, int H, int dtype);

/*
 * cat2d_scores — only the scores a (before the softmax), fp32 [B, H, h·w],
 * to the device pointer a (16-byte aligned, not overlapping Q or K:
 * CAT_ERR_ALIAS).
 */
int cat2d_scores(cat_plan_t plan, const void *Q, const void *K, float *a,
                 int B, int h, int w, int D, int H, int dtype);

/*
 * cat_plan_sync — wait for the plan's stream, then read the device status
 * word the kernels set when an internal check fails (a bad index that was
 * skipped instead of accessed).  Returns CAT_OK, CAT_ERR_DEVICE_STATUS
 * (the word is cleared after reporting) or CAT_ERR_CUDA.
 */
int cat_plan_sync(cat_plan_t plan);

/*
 * cat_plan_describe — copy a one-line, NUL-terminated description of the
 * plan (path, factorisation, launch shapes, workspace bytes) into buf
 * (capacity len bytes, truncated if needed).
 */
int cat_plan_describe(cat_plan_t plan, char *buf, int len);

/*
 * cat_plan_timing — stage timing for profiling.  max_calls > 0 arms the plan
 * to record CUDA events around its three stages (score; softmax and, on the
 * shared-memory and fast paths, the spectrum of z*; the circulant product,
 * which on the general long-sequence path includes the spectrum of z*) on
 * its stream for the next max_calls cat_forward calls, discarding earlier
 * records; max_calls = 0 turns recording off.  On the fast path an event is
 * also recorded after each of passes A, B and C of every chunk.  While
 * recording, a forward runs its kernels one after another on the plan's
 * stream (the fast path otherwise replays a graph that overlaps chunks on
 * two internal streams), so each stage's and each pass's time is its own.
 * Synchronises the plan's stream.  The plan owns the events.
 * Errors: CAT_ERR_INVALID_ARG, CAT_ERR_ALLOC, CAT_ERR_CUDA.
 */
int cat_plan_timing(cat_plan_t plan, int max_calls);

/*
 * cat_plan_stage_times — wait for the plan's stream and write into ms[0..2]
 * (host array, cap >= 3) the milliseconds each stage took, summed over the
 * calls recorded since cat_plan_timing; *ncalls (may be NULL) receives how
 * many calls that was.  Errors: CAT_ERR_INVALID_ARG, CAT_ERR_CUDA.
 */
int cat_plan_stage_times(cat_plan_t plan, float *ms, int cap, int *ncalls);

/*
 * cat_plan_pass_times — fast path only: wait for the plan's stream and write
 * into ms[0..2] (host array, cap >= 3) the milliseconds that passes A, B and
 * C took, each summed over all chunks of the calls recorded since
 * cat_plan_timing; *launches (may be NULL) receives how many launches of
 * each pass that was (chunks per call times calls), so ms[i] / *launches is
 * one launch's average duration.  Errors: CAT_ERR_INVALID_ARG (no plan, cap
 * < 3, or not the fast path), CAT_ERR_CUDA.
 */
int cat_plan_pass_times(cat_plan_t plan, float *ms, int cap, int *launches);

/* Limits of cat_forward_noalloc's fixed device workspace. */
#define CAT_NOALLOC_MAX_ROWS (1 << 18) /* B·H·N                                 */
#define CAT_NOALLOC_MAX_N 16384        /* sequence length                       */

/*
 * cat_forward_noalloc — the same forward as cat_forward (short-sequence
 * shared-memory path), for callers that cannot allocate device memory: a
 * process whose device memory has been handed to a caching or pooled
 * allocator (where cudaMalloc would fail or fragment the pool), or a
 * latency-critical caller that cannot absorb the device-wide
 * synchronisation cudaMalloc and cudaFree imply.  It needs no plan and
 * never calls cudaMalloc, cudaFree or any allocating routine.  The notes
 * page has no counterpart to this entry point; it only changes where the
 * workspace lives.
 *
 * The workspace (scores, z*, spectra, twiddles, status word; about 5 MiB)
 * is one fixed array in the library's device image, which every GPU that
 * loads the library holds until the process exits.  Its size bounds the
 * problem: B·H·N <= CAT_NOALLOC_MAX_ROWS and N <= CAT_NOALLOC_MAX_N, else
 * CAT_ERR_TOO_LARGE.  Other shape rules and host-side errors are those of
 * cat_plan_create and cat_forward.  The kernels' own status word (a failed
 * internal check, which cat_plan_sync reports for plan calls) has no reader
 * here: it is cleared at every call and not reported, so only the returned
 * status (argument and launch errors) tells the caller of a failure.
 *
 * X, W_A, V (read) and O (written): device pointers as for cat_forward.
 * stream: cudaStream_t to enqueue on (NULL = legacy default stream).
 * The call is asynchronous.  The first call on each device also does a
 * one-time set-up on the host (it looks up the array's device address and
 * raises the kernels' shared-memory limits), so make that first call before
 * any stream capture.  All calls share the one array and it keeps the last
 * call's contents: calls whose GPU work overlaps (on different streams, or
 * from different host threads) race on it and must be ordered by the
 * caller.
 */
int cat_forward_noalloc(const void *X, const void *W_A, const void *V, void *O, int B,
                        int N, int D, int H, int dtype, void *stream);

/*
 * cat_probe_dft32 — measurement only, not part of the forward or backward:
 * applies one length-32 DFT stage `rounds` times (each scaled by
 * 1/sqrt(32)) to `nsig` complex fp32 signals (device pointers x, y,
 * [nsig][32] interleaved re/im), keeping each signal on chip, so that the
 * time is the stage's own cost.  mode 0: the register DFT-32 on the FP32
 * pipe (one signal per thread); mode 1 / 2: the stage as a dense 64 x 64 real
 * contraction on the tensor cores (tcgen05, 128 signals per CTA) with the
 * operands split into 2 / 3 bf16 terms (about 16 / 24 significant bits).
 * For the choice of where the small-DFT stages of the circulant product
 * run (the notes page's "FFT acceleration" design fixes the transform, not
 * the unit).  Asynchronous on `stream`.  Errors: CAT_ERR_INVALID_ARG,
 * CAT_ERR_ALLOC, CAT_ERR_CUDA.
 */
int cat_probe_dft32(const void *x, void *y, int nsig, int mode, int rounds, void *stream);

/* Static string for a status code ("CAT_OK", "CAT_ERR_INVALID_ARG", ...). */
const char *cat_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* CAT_H_ */
