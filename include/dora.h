/*
 * dora.h -- C ABI of the DoRA per-module hot path on one GB300 (sm_103a).
 *
 * Two operations, both defined in "Scaling DoRA: High-Rank Adaptation via
 * Factored Norms and Fused Kernels" (Zelenin, Zhuravlyova):
 *
 *   dora_factored_norm  wnorm_j = || W_j + s (B A)_j ||_2,  g_j = m_j / max(wnorm_j, eps)
 *       The DoRA weight is W' = m * (W + sBA) / ||W + sBA||_row (English summary,
 *       "The Problem").  The row norm is evaluated through the factored identity
 *       ||W+sBA||^2_row = ||W||^2_row + 2s rowsum(B o U) + s^2 rowsum((BG) o B),
 *       U = W A^T, G = A A^T (English summary, "Factored Norm"; Chinese write-up
 *       sections 1.2 and 1.2.1), clamped at zero under the root and divided
 *       with eps as a floor (Chinese write-up section 1.2.2; Algorithm 1 of
 *       section 5.1).  The dense product BA is never formed.
 *
 *   dora_compose        out = (g - 1) * base + g * (s * lora)
 *       The numerically stable compose (Chinese write-up sections 2.1 and
 *       2.1.1; English summary, "Fused Kernels"), one pass, fp32 registers,
 *       stored once.
 *
 * Conventions shared by every entry point
 *   - All tensors are dense, row-major, contiguous, in device memory (any
 *     pointer the CUDA runtime can address from the device: cudaMalloc'd,
 *     managed, or torch-allocated).  The caller owns every buffer; the
 *     library allocates nothing and keeps no per-call state.
 *   - Element type `dtype` is DORA_BF16 (bfloat16 bit patterns) or DORA_F32.
 *     It applies to W, A, B, m, base, lora and out.  wnorm and g are always
 *     float32.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Argument checks run on the host before anything is
 *     enqueued; on an argument error nothing is launched.
 *   - Return value: a dora_status.  DORA_ERR_CUDA means a CUDA runtime call
 *     failed while enqueueing (the stream may hold part of the work).
 *     Failures detected on the device (a pipeline wait that ran out of its
 *     time limit) are recorded in the workspace and reported by
 *     dora_check_status.
 */
#ifndef DORA_H_
#define DORA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dora_status {
    DORA_OK = 0,
    DORA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, aliasing, bad dtype */
    DORA_ERR_UNSUPPORTED = 2,  /* legal but outside what the kernels handle: r > 512,
                                  a row stride that is not a multiple of 16 bytes,
                                  a pointer not 16-byte aligned (norm only) */
    DORA_ERR_WORKSPACE = 3,    /* workspace null, misaligned or too small */
    DORA_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
    DORA_ERR_TIMEOUT = 5,      /* device side: a bounded pipeline wait expired */
    DORA_ERR_NO_DEVICE = 6     /* no usable sm_100-family device for this library */
} dora_status;

typedef enum dora_dtype {
    DORA_BF16 = 0,
    DORA_F32 = 1
} dora_dtype;

/* Largest adapter rank the norm supports: U = W A^T for a 128-row tile lives
 * in tensor memory, 512 fp32 columns per SM. */
#define DORA_MAX_RANK 512

/*
 * Bytes of device workspace dora_factored_norm needs for this shape.
 * The workspace holds a small control block (the device status word, the
 * main pass's work counter and per-row-group completion counters, zeroed by
 * every call), the scaled Gram matrix G' = (s/2) A A^T -- as a bf16 split
 * G'_hi + G'_lo for bf16 inputs; in fp32, with the K-segment partials of
 * A A^T (up to 24 x r x r), for fp32 inputs -- and per-segment partial sums
 * of the norm terms.  It does not depend on d_in: about 1.6 MB at
 * d_out = 8192, r = 384 (bf16) and 27.3 MB at d_out = 8192, r = 512 (fp32).
 * Returns 0 for an invalid shape (negative sizes, bad dtype, r > DORA_MAX_RANK).
 */
size_t dora_norm_workspace_size(int64_t d_out, int64_t d_in, int64_t r, int dtype);

/*
 * Factored row norm and magnitude scale of one DoRA module.
 *
 *   W      [d_out x d_in]  frozen base weight, dtype
 *   A      [r x d_in]      LoRA down projection, dtype
 *   B      [d_out x r]     LoRA up projection, dtype
 *   s      LoRA scale (alpha / r or any real); s == 0 or r == 0 skips the
 *          cross and BA-norm terms (Algorithm 1 notes, section 5.1)
 *   m      [d_out]         DoRA magnitude, dtype
 *   eps    floor of the divisor in g = m / max(wnorm, eps) (eps > 0)
 *   wnorm  [d_out] float32 output, the row norm ||W + sBA||_row
 *   g      [d_out] float32 output, m / max(wnorm, eps)
 *   workspace / workspace_bytes  device scratch of at least
 *          dora_norm_workspace_size(d_out, d_in, r, dtype) bytes, 256-byte
 *          aligned; its contents need no initialisation and are overwritten.
 *          One workspace must not be used by two calls in flight at once.
 *   stream cudaStream_t
 *
 * Requirements (else DORA_ERR_UNSUPPORTED): d_in * elem_size and r * elem_size
 * multiples of 16 bytes; W, A, B 16-byte aligned; r <= DORA_MAX_RANK.
 * wnorm and g must not overlap each other or any input.
 * Precision: for bf16 inputs every product of stored values is exact in
 * fp32; for fp32 inputs the products of W A^T, A A^T and B G' are each
 * formed from three TF32 tensor-core products (hi*hi + lo*hi + hi*lo, the
 * "3xTF32" scheme: a few units of 2^-20 relative), and the sum of squares
 * of W is taken in fp32 on the CUDA cores.  Every sum is accumulated in
 * fp32; the three terms are assembled in double-float
 * arithmetic (a value held as an unevaluated sum of two floats, about 48
 * significant bits), the square root and the division each take one
 * correction step in that arithmetic, and each result is rounded once to fp32.
 */
int dora_factored_norm(const void* W, const void* A, const void* B, int dtype,
                       int64_t d_out, int64_t d_in, int64_t r, float s,
                       const void* m, float eps, float* wnorm, float* g,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * Same as dora_factored_norm, and records `ev_main_begin` / `ev_main_end`
 * (cudaEvent_t, either may be NULL) on `stream` immediately before and after
 * the launch of the U = W A^T main-pass kernel, so a caller can time that
 * kernel alone with cudaEventElapsedTime.
 */
int dora_factored_norm_timed(const void* W, const void* A, const void* B, int dtype,
                             int64_t d_out, int64_t d_in, int64_t r, float s,
                             const void* m, float eps, float* wnorm, float* g,
                             void* workspace, size_t workspace_bytes, void* stream,
                             void* ev_main_begin, void* ev_main_end);

/*
 * dora_factored_norm without a caller-supplied workspace: it allocates no
 * device memory at any point.  The paper has no counterpart; this entry point
 * exists for callers that cannot allocate device memory -- for example a
 * plug-in running inside a host program whose allocator owns all of the
 * device's free memory and offers it no hook, or code on a path where
 * cudaMalloc/cudaFree are off limits because they synchronize the device and
 * can fail under memory pressure.
 *
 * Arguments, results and requirements are those of dora_factored_norm.  The
 * workspace is instead a 32 MiB array in the library's own device memory
 * (a file-scope __device__ array): every GPU that loads the library holds it
 * until the process exits.  32 MiB covers d_out up to 253 888 rows at
 * r = 512 (257 468 at r = 384, 261 564 at r = 128) for bf16 inputs and
 * 57 328 rows at r = 512 (146 904 at r = 384, 249 280 at r = 128) for fp32
 * inputs; a shape whose
 * dora_norm_workspace_size exceeds 32 MiB is refused with DORA_ERR_WORKSPACE
 * before anything is enqueued.
 *   - Every call looks up the array's device address (cudaGetSymbolAddress,
 *     with the caller's device current), so the address stays right after a
 *     cudaDeviceReset.  The first call on each device may load the library's
 *     device code there; make that first call before any stream capture.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents (every value a call reads from it, the call itself writes
 *     first).  Calls that overlap on the GPU race: issue them on one stream,
 *     or otherwise order them.
 *   - A device-side pipeline timeout is recorded in the shared array and is
 *     not reported by this entry point; use dora_factored_norm with your own
 *     workspace and dora_check_status where that matters.
 */
int dora_factored_norm_noalloc(const void* W, const void* A, const void* B, int dtype,
                               int64_t d_out, int64_t d_in, int64_t r, float s,
                               const void* m, float eps, float* wnorm, float* g,
                               void* stream);

/*
 * The norm with d_in sharded across devices (row-parallel tensor
 * parallelism: each device holds the columns [k0, k1) of W and of A, and all
 * of B and m).  Every term of the factored norm is a sum over d_in: the base
 * term ||W_j||^2, the cross term rowsum(B o U) with U = W A^T, and the Gram
 * matrix G = A A^T that the BA-norm term rowsum((B G) o B) is built from
 * (Chinese write-up, section 1.2.1 and Algorithm 1 of section 5.1, steps 4a-f
 * and 6).  So each device computes the three for its slice, the devices add
 * them with one all-reduce (sum) of 2 d_out + r^2 floats, and each device
 * then finishes the norm from the sums.  The write-ups mention DoRA training
 * beside tensor-parallel inference (section 4.1) but give no sharded norm;
 * this split of the work is a reading of section 1.2.1's algebra.
 *
 * Partials layout (float32, contiguous, 2 * d_out + r * r values):
 *   [0, d_out)                 base_j  = sum_k W_jk^2                over the slice
 *   [d_out, 2 d_out)           cross_j = sum_l B_jl (W A^T)_jl      over the slice
 *   [2 d_out, 2 d_out + r^2)   G       = A A^T, [r x r] row-major    over the slice
 * The partials do not depend on s, eps or m.
 */

/* Floats of the partials buffer: 2 * d_out + r * r (0 for an invalid shape). */
size_t dora_norm_partials_floats(int64_t d_out, int64_t r);

/*
 * The partials of one d_in slice.
 *   W  [d_out x d_in]  this slice's columns of the frozen weight, dtype
 *   A  [r x d_in]      this slice's columns of the down projection, dtype
 *   B  [d_out x r]     the whole up projection, dtype
 *   partials  [2 d_out + r^2] float32 output (4-byte aligned; must not
 *          overlap an input)
 *   workspace / workspace_bytes  at least dora_norm_workspace_size(d_out,
 *          d_in, r, dtype) bytes, 256-byte aligned, no initialisation needed
 * Requirements and errors as dora_factored_norm (d_in here is the slice
 * width).  An empty slice (d_in = 0) writes zeros; r = 0 writes base and a
 * zero cross; d_out = 0 writes G only.  Precision: as dora_factored_norm --
 * fp32 sums of exact bf16 products, or 3xTF32 products for fp32 inputs --
 * with each sum rounded once to fp32 when it is stored.
 */
int dora_norm_partials(const void* W, const void* A, const void* B, int dtype,
                       int64_t d_out, int64_t d_in, int64_t r, float* partials,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace dora_norm_finalize_partials needs (0 for an invalid shape). */
size_t dora_norm_finalize_workspace_size(int64_t d_out, int64_t r, int dtype);

/*
 * wnorm and g from partials summed over every slice of d_in (after the
 * caller's all-reduce):
 *   wnorm_j = sqrt(max(base_j + 2 s cross_j + s^2 rowsum((B G) o B)_j, 0)),
 *   g_j = m_j / max(wnorm_j, eps)
 * with the BA-norm term taken on the tensor cores from the summed G (bf16
 * inputs: G' = (s/2) G split into two bf16 terms, as dora_factored_norm
 * does).  partials: [2 d_out + r^2] float32 in the layout above; B [d_out x r],
 * m [d_out] in dtype; wnorm, g [d_out] float32 outputs; workspace of
 * dora_norm_finalize_workspace_size bytes, 256-byte aligned.  s == 0 or
 * r == 0 skips the BA-norm term and B is not read.  Errors as
 * dora_factored_norm.
 */
int dora_norm_finalize_partials(const float* partials, const void* B, int dtype,
                                int64_t d_out, int64_t r, float s, const void* m, float eps,
                                float* wnorm, float* g, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * Stable fused compose.
 *
 *   base, lora  [T x d_out]  dtype (base = the frozen layer's output, lora =
 *               the adapter branch's output, one row per token)
 *   g           [d_out] float32, one scale per output feature, broadcast over T
 *   s           LoRA scale
 *   out         [T x d_out]  dtype; may equal base or lora (in place), must not
 *               partially overlap them
 *
 * Evaluation order: s * lora first, then g * (.), plus (g - 1) * base with the
 * exact rounding error of that product carried (an error-free product), all in
 * fp32 registers, rounded once to dtype.  T == 0 or d_out == 0 is a no-op.
 * Any alignment and any d_out are accepted (the 16-byte vector path covers
 * aligned rows, the same kernel handles the rest element by element).
 */
int dora_compose(const void* base, const void* lora, const float* g, float s,
                 int dtype, int64_t T, int64_t d_out, void* out, void* stream);

/*
 * Grouped calls: one launch sequence for a whole stack of adapted modules
 * (the Chinese write-up, sections 2.2 and 4.2, notes that launch latency
 * dominates small shapes such as the 512-row KV projections).  Results are
 * those of the per-module calls, up to the order of fp32 sums.
 */

/* One module of a grouped norm: the dora_factored_norm arguments that differ
 * per module (same meaning, layout and requirements). */
typedef struct dora_norm_module {
    const void* W;        /* [d_out x d_in] */
    const void* A;        /* [r x d_in] */
    const void* B;        /* [d_out x r] */
    const void* m;        /* [d_out] */
    float* wnorm;         /* [d_out] output */
    float* g;             /* [d_out] output */
    int64_t d_out;
    int64_t d_in;
} dora_norm_module;

/* Bytes of workspace for dora_factored_norm_grouped over these modules
 * (0 for an invalid argument). */
size_t dora_norm_grouped_workspace_size(const dora_norm_module* modules, int n_modules,
                                        int64_t r, int dtype);

/*
 * dora_factored_norm for every module of `modules`, all with the same rank r,
 * dtype, s and eps.  bf16 inputs run as one Gram launch and one persistent
 * main-pass launch over the work items of all modules; other cases call the
 * per-module path in turn.  The module table is read from host memory during
 * the call (copied to the workspace), so the array may be freed on return.
 * workspace: dora_norm_grouped_workspace_size bytes, 256-byte aligned, no
 * initialisation needed.  Errors as dora_factored_norm (the first invalid
 * module makes the call return before anything is enqueued).
 */
int dora_factored_norm_grouped(const dora_norm_module* modules, int n_modules, int dtype,
                               int64_t r, float s, float eps, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * A grouped norm prepared once and run many times.  dora_factored_norm_grouped
 * encodes a TMA descriptor set and copies a table entry for every module on
 * each call: host work that grows with the module count and, since the copy
 * reads pageable memory, blocks the host.  A plan does that once; a run only
 * zeroes a few control words and launches the Gram and main-pass kernels.
 * This fits a training loop, where the frozen weights W and the adapter
 * parameters A, B, m keep their buffers and are updated in place.
 *
 * dora_norm_grouped_plan_create: checks the modules as the grouped call does
 * (apart from s and eps, which come with each run; a module may have null A
 * and B and then only runs with s = 0), writes the module tables into
 * `workspace` (dora_norm_grouped_workspace_size bytes, 256-byte aligned) on
 * `stream` and synchronizes `stream` before returning, so a run may use any
 * stream.  On success *plan holds a new handle; on error *plan is NULL and
 * nothing is left allocated.
 *
 * The plan refers to, and does not own, the workspace and every buffer named
 * in `modules` (the array itself may be freed on return).  They must stay
 * allocated, with the same shapes, until dora_norm_grouped_plan_destroy, and
 * the workspace must not be used for anything else meanwhile.  The contents
 * of W, A, B and m may change between runs.  Runs on one plan must not
 * overlap in time (they share the workspace): issue them on one stream or
 * order them with events.
 *
 * dora_norm_grouped_plan_run: dora_factored_norm_grouped's result for these
 * s and eps, written to each module's wnorm and g.  Returns
 * DORA_ERR_INVALID_ARG for a NULL plan or when the current device is not the
 * one the plan was created on; otherwise errors as dora_factored_norm_grouped.
 *
 * dora_norm_grouped_plan_destroy: frees the handle (host memory only; NULL is
 * accepted).  It does not wait for runs in flight, which may still read the
 * workspace: keep the workspace until they complete.
 */
typedef struct dora_norm_grouped_plan_s* dora_norm_grouped_plan;

int dora_norm_grouped_plan_create(const dora_norm_module* modules, int n_modules, int dtype,
                                  int64_t r, void* workspace, size_t workspace_bytes,
                                  void* stream, dora_norm_grouped_plan* plan);
int dora_norm_grouped_plan_run(dora_norm_grouped_plan plan, float s, float eps, void* stream);
void dora_norm_grouped_plan_destroy(dora_norm_grouped_plan plan);

/* One module of a grouped compose: the dora_compose arguments that differ per
 * module. */
typedef struct dora_compose_module {
    const void* base;     /* [T x d_out] */
    const void* lora;     /* [T x d_out] */
    const float* g;       /* [d_out] */
    void* out;            /* [T x d_out] output */
    int64_t T;
    int64_t d_out;
} dora_compose_module;

/* Bytes of workspace for dora_compose_grouped over n_modules modules. */
size_t dora_compose_grouped_workspace_size(int n_modules);

/*
 * dora_compose for every module, one launch when every module has 16-byte
 * rows and 16-byte aligned pointers (else one dora_compose per module).
 * Same s and dtype for all.  workspace: dora_compose_grouped_workspace_size
 * bytes, 256-byte aligned.
 */
int dora_compose_grouped(const dora_compose_module* modules, int n_modules, float s, int dtype,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * Training path of the compose ("Scaling DoRA", Chinese write-up sections
 * 2.2, 4.2 and 5.2: the fused backward tier).  The norm is a detached
 * constant in the backward (section 1.2.2), so with g = m / max(wnorm, eps)
 *
 *   d out / d base = g - 1,   d out / d lora = g s,   d out / d g = base + s lora.
 */

/*
 * Forward of the training path: out as dora_compose, and
 *   inner = base + s * lora    [T x d_out], dtype (rounded once from fp32)
 * the activation the magnitude gradient needs, written in the same pass.
 * Skip this entry point (call dora_compose) when the magnitude is frozen.
 * out and inner must not overlap each other or the inputs.  T == 0 or
 * d_out == 0 is a no-op.  Any alignment and d_out are accepted.
 */
int dora_compose_train(const void* base, const void* lora, const float* g, float s, int dtype,
                       int64_t T, int64_t d_out, void* out, void* inner, void* stream);

/* Bytes of workspace dora_compose_backward needs when it computes dmag
 * (the per-row-block partial column sums): 1024 * d_out at T >= 256,
 * 4 * T * d_out below.  0 for an invalid shape. */
size_t dora_compose_backward_workspace_size(int64_t T, int64_t d_out);

/*
 * Backward of the compose, one pass over the upstream gradient:
 *   d_out_grad  [T x d_out] dtype   dL/d out
 *   d_base      [T x d_out] dtype   output, (g - 1) * d_out_grad
 *   d_lora      [T x d_out] dtype   output, g * s * d_out_grad
 *   g           [d_out] float32
 * and, when dmag is not NULL (a trainable magnitude),
 *   dmag_j = sum_t d_out_grad_tj * inner_tj / max(wnorm_j, eps)   [d_out] float32
 * with inner from dora_compose_train, wnorm [d_out] float32 from the norm,
 * and a workspace of dora_compose_backward_workspace_size bytes (16-byte
 * aligned; no initialisation needed).  The column sums are taken over fixed
 * row blocks and added in block order: the same result on every call, no
 * atomics.  With dmag NULL, inner, wnorm and workspace are not read and may
 * be NULL.  Outputs must not overlap each other or the inputs.
 */
int dora_compose_backward(const void* d_out_grad, const void* inner, const float* g,
                          const float* wnorm, float eps, float s, int dtype, int64_t T,
                          int64_t d_out, void* d_base, void* d_lora, float* dmag,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Waits for `stream`, then reads the device status word of `workspace` (as
 * last written by dora_factored_norm on it): DORA_OK, or DORA_ERR_TIMEOUT if
 * a kernel gave up on a pipeline wait (its outputs are then undefined, the
 * CUDA context stays usable).  Returns DORA_ERR_CUDA if the copy fails.
 */
int dora_check_status(const void* workspace, void* stream);

/*
 * Self-test of the device-side failure detection: zeroes the status word at
 * the start of `workspace` (256-byte aligned, at least 256 bytes), then runs
 * one block that waits -- with the bounded wait every pipeline role uses -- on
 * a barrier that nothing completes, gives up after `timeout_us` microseconds
 * (1 .. 1 000 000) and records DORA_ERR_TIMEOUT in that word, as a pipeline
 * role does when a wait runs out.  The kernel then returns and the CUDA
 * context stays usable; dora_check_status(workspace, stream) reads the word.
 * Returns DORA_ERR_WORKSPACE / DORA_ERR_INVALID_ARG for bad arguments before
 * anything is enqueued.
 */
int dora_selftest_timeout(void* workspace, size_t workspace_bytes, unsigned timeout_us,
                          void* stream);

/*
 * Self-test of the main pass's work decomposition (host only, no GPU): plans
 * a bf16 single-module norm of d_out x d_in at rank r (1 .. DORA_MAX_RANK)
 * exactly as dora_factored_norm does on a device with `clusters` co-resident
 * CTA pairs (1 .. 65535; 76 on a GB300), enumerates every piece of work the
 * launched pairs would run -- K segments handed out in item order, the static
 * ranges of each pair (issued from the last piece to the first), the piece
 * table (one piece per pair, with fewer pair tiles than pairs), or whole
 * tiles and a piece table (each pair w whole pair tiles, then at most one
 * piece of the tiles left over) -- and checks that the pieces of every
 * 256-row pair tile cover its K tiles once, in K order, numbered 0 .. n - 1
 * with n <= 16 (the partial planes of the workspace), and that a piece table
 * gives each launched pair at most one piece.  Writes the schedule chosen
 * (*schedule: 0 K segments, 1 static ranges, 2 piece table, 3 whole tiles
 * and a piece table), the largest number of pieces of one tile, and the
 * number of defects found (0 when the plan is sound).  Returns DORA_ERR_INVALID_ARG
 * for bad arguments, else DORA_OK.
 */
int dora_selftest_schedule(int64_t d_out, int64_t d_in, int64_t r, int clusters,
                           int* schedule, int* max_pieces, int64_t* defects);

/*
 * The same check for a grouped launch (host only, no GPU): plans the work
 * items of one grouped main pass over n_modules bf16 modules (d_out[i] x
 * d_in[i], all at rank r) as dora_factored_norm_grouped and the grouped plan
 * do on a device with `clusters` co-resident CTA pairs, then maps every item
 * to its module and piece through the kernel's own search and decode, and
 * checks the module order (longest K first) and that every pair tile of
 * every module is covered once, in K order, by at most 16 numbered pieces.
 * Writes the largest number of pieces of one tile and the number of defects
 * (0 when sound).  Returns DORA_ERR_INVALID_ARG for bad arguments (including
 * more than 2^22 pair tiles in all), else DORA_OK.
 */
int dora_selftest_grouped_schedule(const int64_t* d_out, const int64_t* d_in, int n_modules,
                                   int64_t r, int clusters, int* max_pieces, int64_t* defects);

/* Number of CUDA kernels this library has launched in this process so far
 * (all devices, all entry points); a diagnostic counter. */
uint64_t dora_launch_count(void);

/* Static, human-readable name of a dora_status value. */
const char* dora_status_string(int status);

/* Library ABI version: (major << 16) | minor.  1.1 added the two schedule
 * self-tests, 1.2 the d_in-sharded norm (partials and finalize); nothing was
 * removed or changed. */
int dora_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DORA_H_ */
