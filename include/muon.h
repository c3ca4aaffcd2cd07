/*
 * muon.h - C ABI of the B300 (sm_103a) Muon optimizer step.
 *
 * What is computed
 * ----------------
 * "How to train a GPT model in 3 minutes: an analysis of modded-nanogpt's
 * optimizations", section 2 (custom Muon optimizer): Muon replaces AdamW for
 * the hidden projection matrices. It follows spectral gradient descent, whose
 * step direction is the orthogonal polar factor U V^T of the update, and it
 * reaches that factor with a Newton-Schulz iteration instead of an SVD. The
 * record analysis "2026-05-27_MuddGatedAndDC", section 6.2 (per-parameter
 * optimizer table), routes projection matrices to Muon and gates to Adam.
 *
 * The pages print no formula. This library computes, per matrix, the plainest
 * reading of that description:
 *
 *   1. momentum   buf <- beta*buf + g;  u = g + beta*buf (Nesterov) or u = buf
 *   2. normalise  X0 = u / (||u||_F + eps)
 *   3. orient     X = X0^T when rows > cols (n = min(rows,cols) <= m = max)
 *   4. iterate    A = X X^T;  B = b*A + c*A*A;  X <- a*X + B X      (k times)
 *   5. restore    O = X^T if step 3 transposed, else X
 *   6. update     W <- W * (1 - lr * wd) - lr * s * O,  s = max(1, rows/cols)^0.5 (or 1)
 *
 * muon_step runs 1-6, muon_orthogonalize runs 2-5.
 *
 * Conventions
 * -----------
 * - Every matrix is row-major: element (i, j) sits at ptr + i*ld + j, in
 *   elements, with ld >= cols. All pointers are DEVICE pointers on the
 *   handle's device, and the caller owns them.
 * - Descriptor arrays (muon_matrix*) are HOST arrays. They are read during
 *   the call and not kept.
 * - `stream` is a cudaStream_t passed as void*. NULL means the legacy default
 *   stream. All GPU work is queued on it in order, and no call waits for the
 *   GPU except muon_get_error and muon_profile_read.
 * - Arithmetic: operands of the Newton-Schulz products are bf16 and
 *   accumulation is fp32 on the tensor cores. Momentum, norms and updates use
 *   fp32 math.
 * - A call with a matrix set it has not seen before builds a plan: it groups
 *   the matrices by oriented shape and allocates device workspace
 *   (cudaMalloc). That first call synchronises the device. Later calls with
 *   the same shapes reuse the plan and allocate nothing.
 * - Calls on one handle must not overlap on the GPU, i.e. they must be on
 *   one stream or otherwise ordered, because they share the plan's workspace.
 * - Errors: argument errors are found on the host before any launch. They
 *   return MUON_ERR_INVALID and have no side effect. CUDA errors return
 *   MUON_ERR_CUDA. A device-side wait that runs past its time limit (about
 *   two seconds) ends its kernel early and raises a device flag, which
 *   muon_get_error reports as MUON_ERR_TIMEOUT. muon_last_error gives a
 *   one-line message for the last failure on the handle.
 */
#ifndef MUON_H
#define MUON_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct muon_ctx* muon_handle;

typedef enum {
  MUON_OK = 0,
  MUON_ERR_INVALID = 1,      /* bad argument; nothing was launched */
  MUON_ERR_CUDA = 2,         /* a CUDA runtime or driver call failed */
  MUON_ERR_NOMEM = 3,        /* workspace allocation failed */
  MUON_ERR_UNSUPPORTED = 4,  /* device is not sm_103 / sm_100 class */
  MUON_ERR_TIMEOUT = 5       /* a device-side bounded wait expired */
} muon_status;

typedef enum { MUON_F32 = 0, MUON_BF16 = 1 } muon_dtype;

/* One matrix: row-major, device pointer, ld in elements (ld >= cols).
 * A matrix with rows == 0 or cols == 0 is accepted and skipped. */
typedef struct {
  void* ptr;
  int64_t rows;
  int64_t cols;
  int64_t ld;
  int32_t dtype; /* muon_dtype */
} muon_matrix;

/* Newton-Schulz and update settings kept by the handle.
 * steps: iterations k (>= 0). a, b, c: the odd polynomial a*x + b*x^3 + c*x^5
 * applied to the singular values. eps: added to ||u||_F, outside the square
 * root. scale_lr_by_shape: nonzero applies s = max(1, rows/cols)^0.5 in step 6,
 * zero applies s = 1. weight_decay (>= 0): decoupled decay, step 6 becomes
 * W <- W * (1 - lr * weight_decay) - lr * s * O. The energy-efficiency article
 * on Modded-NanoGPT (hyperparameter paragraph) reports wd = 1.0; the form is
 * this library's reading.
 * precise_carry (0, 1 or 2): 0 rounds X to bf16 after every iteration, the
 * stated bf16 arithmetic. 1 carries X between iterations as two bf16 parts,
 * hi = bf16(X) and lo = bf16(X - hi). The tensor cores still take hi. The
 * a*X term, X0 and the final O use hi + lo (about 16 significant bits), so
 * rounding noise does not build up over the iterations. On gradients with a
 * few dominant directions this cuts the distance to the exact iteration by
 * one to two orders of magnitude. It costs a second pair of X buffers in
 * the workspace, 4 more bytes per element in each combine pass, and combines
 * that stage their two 64-column units one after the other. 2 (the default,
 * MUON_CARRY_WHEN_C) carries X exactly for the calls whose c is nonzero
 * (muon_step: the handle's c; muon_orthogonalize: the call's c): a quintic's
 * slope a > 1 at zero amplifies the rounding noise that gradients with a few
 * dominant directions put into their small singular values, and with X
 * rounded every iteration the GPT-2 124M spiked gradients end 2.1e-2 from the
 * exact iteration under (15, -10, 3)/8, against 5e-4 with the carry; the
 * cubic's slope 1.5 leaves them at 8e-3 without it.
 * persistent (0, 1 or 2): 1 runs every Newton-Schulz iteration of a call in
 * one persistent launch (up to 16 iterations per launch), whose clusters take
 * the Gram and combine tiles of all matrices from host-built work lists and
 * wait on per-matrix stage counters in global memory. 0 runs one launch per
 * Gram and per combine phase over the whole batch. 2 (the default,
 * MUON_PERSISTENT_AUTO) chooses per call: the per-phase launches when one
 * iteration gives every resident 2-CTA cluster 800 or more 64-wide k-blocks
 * of 256 x 256 tiles (each phase then streams enough tiles that its ramp and
 * tail cost less than the persistent launch's item changes), the persistent
 * launch otherwise (muon_launch_choice reports the choice). All compute the
 * same thing with the same roundings. Calls with more than 1024 distinct
 * oriented shapes always take the per-phase launches. */
#define MUON_CARRY_WHEN_C 2
#define MUON_PERSISTENT_AUTO 2
typedef struct {
  int32_t steps;
  float a, b, c;
  float eps;
  int32_t scale_lr_by_shape;
  float weight_decay;
  int32_t precise_carry;
  int32_t persistent;
} muon_config;

/* Fills *cfg with the defaults: steps 5, (a,b,c) = (1.5, -0.5, 0), eps 1e-7,
 * scale_lr_by_shape 1, weight_decay 0, precise_carry MUON_CARRY_WHEN_C, persistent MUON_PERSISTENT_AUTO. The cubic coefficients
 * are the iteration's textbook form; the pages give none. */
void muon_default_config(muon_config* cfg);

/* Creates a handle on CUDA device `device`. cfg may be NULL (defaults).
 * Allocates a small device block (error flag). Returns MUON_ERR_UNSUPPORTED
 * if the device is not compute capability 10.x. *out is NULL on failure. */
muon_status muon_create(muon_handle* out, int device, const muon_config* cfg);

/* Frees the handle and its workspace after synchronising the device. NULL is
 * a no-op. */
muon_status muon_destroy(muon_handle h);

/* Steps 2-5 on `count` matrices: out[j] = NS_k(in[j]), the Newton-Schulz
 * orthogonalisation of in[j] with `steps` iterations of the polynomial (a, b, c)
 * and the handle's eps. in[j] and out[j] have the same rows and cols; dtype F32
 * or BF16 each (all in[] share one dtype, all out[] share one dtype). out[j]
 * may be in[j] (in place). Distinct out[] must not overlap. count == 0 is a
 * no-op. */
muon_status muon_orthogonalize(muon_handle h, const muon_matrix* in, const muon_matrix* out,
                               int count, int steps, float a, float b, float c, void* stream);

/* Steps 1-6 on `count` matrices with the handle's Newton-Schulz settings:
 *   momentum[j] <- beta*momentum[j] + grads[j]
 *   u = grads[j] + beta*momentum[j]   (nesterov != 0)   or   u = momentum[j]
 *   params[j]  <- params[j] * (1 - lr * weight_decay) - lr * s_j * NS_k(u)
 * params: F32 or BF16 (all alike). grads: F32 or BF16 (all alike).
 * momentum: F32. All three of matrix j have the same rows and cols and must
 * not overlap one another. count == 0 is a no-op. */
/* Both entry points are stream-ordered. The first call for a set of shapes
 * allocates and uploads its plan synchronously; later calls with the same
 * shapes, iteration count and c launch kernels only, so such a call may be
 * captured in a CUDA graph (the graph keeps the tensors' addresses). */
muon_status muon_step(muon_handle h, const muon_matrix* params, const muon_matrix* grads,
                      const muon_matrix* momentum, int count, float lr, float beta, int nesterov,
                      void* stream);

/* Synchronises `stream`, then returns and clears the device error flag
 * (MUON_OK or MUON_ERR_TIMEOUT), or MUON_ERR_CUDA if the sync failed. */
muon_status muon_get_error(muon_handle h, void* stream);

/* Static name of a status code. Never NULL. */
const char* muon_status_string(muon_status s);

/* One-line message for the last failure on h (empty string if none; a fixed
 * message for h == NULL). Valid until the next call on h. */
const char* muon_last_error(muon_handle h);

/* Host-only argument checks that muon_orthogonalize / muon_step run before
 * launching anything. They touch no GPU and can be called without a device.
 * On failure, msg (if not NULL, capacity msg_len) receives the reason. */
muon_status muon_check_orthogonalize(const muon_matrix* in, const muon_matrix* out, int count,
                                     int steps, char* msg, int msg_len);
muon_status muon_check_step(const muon_matrix* params, const muon_matrix* grads,
                            const muon_matrix* momentum, int count, char* msg, int msg_len);

/* Host-only plan arithmetic, no GPU: for `count` matrices of shape
 * rows[j] x cols[j], writes the number of distinct oriented shapes (groups),
 * the 128x256 tiles of the Gram products X X^T that reach the upper triangle,
 * the 128x256 tiles of the B X products, and the algorithmic flops of one Newton-Schulz
 * iteration (n(n+1)m for the upper-triangle Gram plus 2 n^2 m for B X, per
 * matrix, plus n^2(n+1) for A*A when c != 0 is selected by with_c). Any output
 * pointer may be NULL. */
muon_status muon_plan_stats(const int64_t* rows, const int64_t* cols, int count, int with_c,
                            int* groups, int64_t* gram_tiles, int64_t* combine_tiles,
                            double* flops_per_iter);

/* ---------------------------------------------------------------- sharding across ranks
 * Host-only, no GPU. The speedrun reduce-scatters gradients instead of
 * all-reducing them (energy-efficiency article on Modded-NanoGPT,
 * technical-evolution section; "How to train a GPT model in 3 minutes",
 * system optimisations, distributed communication) and merges the attention
 * and MLP parameters into one reduce_scatter call ("Muon Custom Sizing", in
 * the related-article list of the record analysis of
 * 2026-05-27_MuddGatedAndDC). With whole matrices as the unit, each of
 * `world` ranks owns a subset, gets its summed gradients from one in-place
 * reduce-scatter, runs muon_step on them, and one in-place all-gather
 * replicates the updated parameters.
 *
 * For `count` matrices rows[j] x cols[j]: owner[j] is the owning rank,
 * chosen longest-processing-time first by the algorithmic flops of one
 * Newton-Schulz iteration (n(n+1)m + 2n^2m, + n^2(n+1) when with_c), so the
 * ranks' loads (load[r], may be NULL, `world` entries) are balanced.
 * offset[j] is the element offset of matrix j (stored densely, ld = cols) in
 * a flat buffer of world * segment elements laid out rank-major: rank r's
 * matrices sit in index order inside [r*segment, (r+1)*segment), each
 * starting on a multiple of `align` elements. *segment is the common segment
 * length (a multiple of align, at least align). Deterministic: every rank
 * computes the same layout. Bad arguments give MUON_ERR_INVALID. */
muon_status muon_shard_layout(const int64_t* rows, const int64_t* cols, int count, int world, int with_c,
                              int64_t align, int* owner, int64_t* offset, int64_t* segment, double* load);

/* Device-memory cap for the handle's plans (workspaces and tile schedules),
 * in bytes; 0 removes the cap (the default). A call that needs a new plan
 * which would take the plans past the cap fails with MUON_ERR_NOMEM, exactly
 * as it does when cudaMalloc runs out of device memory: before anything is
 * launched, with the caller's tensors untouched and the plans already built
 * kept. A later call (with a higher cap, or after memory is freed) builds the
 * plan normally. bytes < 0 or h == NULL gives MUON_ERR_INVALID.
 * muon_workspace_bytes writes the device memory the plans hold now. */
muon_status muon_set_workspace_limit(muon_handle h, int64_t bytes);
muon_status muon_workspace_bytes(muon_handle h, int64_t* bytes);

/* Host-only, no GPU: which launches a handle whose muon_config.persistent is
 * `persistent` (0, 1 or 2) runs for `count` matrices rows[j] x cols[j] on a
 * device with `clusters` resident 2-CTA clusters (74 on a B300), c != 0 when
 * with_c: *use_persistent = 1 for the persistent launch, 0 for the per-phase
 * launches, and *kblocks_per_cluster the 64-wide k-blocks of one iteration's
 * 256 x 256 tiles per cluster that MUON_PERSISTENT_AUTO compares with 800.
 * Either output pointer may be NULL. */
muon_status muon_launch_choice(const int64_t* rows, const int64_t* cols, int count, int with_c, int clusters,
                               int persistent, int* use_persistent, double* kblocks_per_cluster);

/* Host-only, no GPU: the work lists of the persistent Newton-Schulz launch
 * (muon_config.persistent) for `count` matrices rows[j] x cols[j], `steps`
 * iterations (1 .. 16, one launch) and `clusters` 2-CTA clusters, as the
 * library builds them. An item is 4 int32: kind | group << 2 | flags << 12
 * (kind 0 Gram X X^T, 1 Gram A A, 2 combine; flags 1 first iteration,
 * 2 last iteration, 4 X in the second buffer), the matrix within its shape
 * group (groups are the distinct oriented shapes, in order of first
 * appearance), tile row | tile column << 16, and the number of finished
 * epilogue halves (four per tile) of the matrix the item waits for. Cluster c
 * takes items[begin[c] .. begin[c+1]) in order. More than 1024 distinct
 * oriented shapes give MUON_ERR_UNSUPPORTED (such calls run the per-phase
 * launches whatever muon_config.persistent says). Writes the item count to
 * *num_items; with items and begin NULL nothing else is written, otherwise
 * items needs room for 4 * *num_items values and begin for clusters + 1. */
muon_status muon_persistent_schedule(const int64_t* rows, const int64_t* cols, int count, int steps, int with_c,
                                     int clusters, int32_t* items, int64_t items_cap, int32_t* begin,
                                     int64_t* num_items);

/* Failure-detection self-test. Launches one kernel on `stream` that waits,
 * through the same bounded wait the GEMM kernels use, on a barrier that
 * nothing ever arrives at. After limit_ns (1e6 .. 2e9 ns, else
 * MUON_ERR_INVALID) the wait gives up, the kernel raises the handle's error
 * flag and returns, so the next muon_get_error reports MUON_ERR_TIMEOUT and
 * the context stays usable. Nothing traps or faults. */
muon_status muon_selftest_wait(muon_handle h, int64_t limit_ns, void* stream);

/* Failure-detection self-test of the persistent Newton-Schulz launch
 * (muon_config.persistent): one launch over a 256 x 256 matrix of the
 * handle's workspace whose first work item waits for a stage count its matrix
 * never reaches. Every wait of that launch gives up after limit_ns (1e6 ..
 * 2e9 ns, else MUON_ERR_INVALID); the CTAs that gave up stop, let their
 * copies and MMAs in flight land and free their tensor memory, the last one
 * resets the stage counters, and the device error flag is raised, so the next
 * muon_get_error reports MUON_ERR_TIMEOUT and later calls run normally.
 * Nothing traps or faults. The call waits for the launch (a few limit_ns at
 * most); the caller's tensors are not touched. */
muon_status muon_selftest_persistent(muon_handle h, int64_t limit_ns, void* stream);

/* Kernel timing, for benchmarks. While enabled, each kernel the handle
 * launches is bracketed by CUDA events on the launching stream.
 * muon_profile_read synchronises those events, writes per kernel kind the
 * summed milliseconds and launch counts since the last read (arrays of
 * MUON_KERNEL_KINDS entries, either may be NULL) and resets the sums. */
#define MUON_KERNEL_KINDS 9
/* kernel kinds: 0 momentum+norm, 1 norm, 2 scale+orient, 3 Gram X X^T,
 * 4 Gram A A (c != 0), 5 combine a X + B X, 6 update, 7 copy out,
 * 8 every Newton-Schulz iteration in one persistent launch */
muon_status muon_profile_enable(muon_handle h, int enable);
muon_status muon_profile_read(muon_handle h, double* ms, int64_t* launches);
const char* muon_kernel_name(int kind);
/* The SM clock the tensor-core GEMM kernels ran at while profiling was on:
 * their CTAs' summed clock64() cycles over their summed %globaltimer
 * nanoseconds, in MHz (0 if none ran). muon_profile_enable(h, 1) resets the
 * sums when it turns profiling on. Synchronous: call it after
 * muon_profile_read, which waits for the profiled kernels. */
muon_status muon_profile_clock(muon_handle h, double* sm_mhz);

/* ---------------------------------------------------------------- allocation-free normalisation
 * The pages have no counterpart to this entry point. It exists for callers
 * that cannot call cudaMalloc: code whose device memory is owned by another
 * pool or allocator, plugins whose host framework forbids allocation inside
 * its callbacks, and loops that must never hit the allocator's implicit
 * synchronisation. muon_create and the first call of a new shape set
 * allocate; this function never does.
 *
 * For each j: out[j] = in[j] / (||in[j]||_F + eps), the normalisation step
 * on its own (no Newton-Schulz iteration), with the same kernels as the
 * other entry points. Shapes, dtypes, layouts and in-place use follow
 * muon_orthogonalize. It needs no handle and runs on the CURRENT CUDA device,
 * on which every pointer must live.
 *
 * Scratch (partial sums, arrival tickets, inverse norms) lives in a static
 * device array inside the library, about 33 KB, that every GPU which loads
 * the library holds until the process exits. Limits: at most
 * MUON_NOALLOC_MAX_MATRICES matrices per call and at most
 * MUON_NOALLOC_MAX_ELEMENTS elements in total, counting each matrix in whole
 * blocks of 8192 elements. A call beyond either limit returns
 * MUON_ERR_INVALID with the reason in msg, and launches nothing.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress), and so does the first call after the device's
 * context has been created again (cudaDeviceReset). Make that first call
 * before any stream capture. A device index of 64 or more returns
 * MUON_ERR_UNSUPPORTED.
 * All calls share the one array: calls that overlap on the GPU (different
 * streams without ordering, or several host threads) race and give wrong
 * results. The tickets are cleared by every call; the other contents are left
 * over from the last call and are rewritten before use.
 * msg (capacity msg_len, may be NULL) receives the reason for any failure. */
#define MUON_NOALLOC_MAX_MATRICES 128
#define MUON_NOALLOC_MAX_ELEMENTS (1ll << 26)
muon_status muon_normalize_noalloc(const muon_matrix* in, const muon_matrix* out, int count, float eps,
                                   void* stream, char* msg, int msg_len);

#ifdef __cplusplus
}
#endif

#endif /* MUON_H */
