/*
 * mttkrp.h -- C ABI of the GB300 dense, matrix-free MTTKRP library.
 *
 * The operation ("A Performance Portable Matrix Free Dense MTTKRP in GenTen",
 * abstract and TL;DR): for a d-way dense tensor Y of shape I_0 x ... x I_{d-1},
 * factor matrices A_n (I_n x R) and a mode k, the matricized tensor times
 * Khatri-Rao product
 *
 *     M_k(i, r) = sum_{(i_n), n != k} Y(i_0, ..., i_{d-1}) * prod_{n != k} A_n(i_n, r),
 *
 * i.e. M_k = Y_(k) * (Khatri-Rao product of the A_n, n != k), computed without
 * ever forming the Khatri-Rao matrix (the matrix-free scheme of that paper,
 * whose memory grows with R * sum_n I_n instead of R * prod_{n != k} I_n).
 *
 * Layouts (all fp32, all device memory, all owned by the caller):
 *   Y        C-order contiguous (last index fastest), prod_n I_n elements.
 *   A_n      I_n x R row-major (r fastest).  The factor of the mode being
 *            computed is not read and may be NULL.
 *   M_k      I_k x R row-major; overwritten (not accumulated into).
 *   workspace  caller-allocated device scratch of mttkrp_workspace_bytes()
 *            bytes, 256-byte aligned; holds split partial sums, small
 *            factor-product tables and, for tensor-core modes on the
 *            fp16-image kernel, fp16 hi/lo images of Y (4 bytes an element
 *            per layout).  The library itself never allocates device memory.
 *
 * Execution: every compute call only enqueues kernels on the given CUDA
 * stream (a cudaStream_t passed as void*; NULL = the legacy default stream)
 * and returns without synchronising.  Results are bitwise reproducible from
 * run to run for a given plan (no atomics; split partial sums are added in a
 * fixed order, in fp64 or compensated fp32).  A plan and its workspace may be used by one stream
 * at a time; calls on one plan are not thread-safe.
 *
 * Around the MTTKRP the library also provides one CP-ALS sweep on the device
 * (mttkrp_cp_als_sweep, on a plan), and two dense kernels of the Jacobi-type
 * Tucker diagonalization setting that take plain pointers and no plan: the
 * mode-n product (mttkrp_ttm) and Givens rotations along a mode
 * (mttkrp_apply_rotations).
 *
 * Errors: every int-returning call returns MTTKRP_OK (0) or one of the codes
 * below; nothing is thrown across the ABI.  mttkrp_strerror() names a code and
 * mttkrp_last_error() gives the calling thread's last detailed message.
 * Argument errors are detected on the host before anything is enqueued.
 */
#ifndef MTTKRP_H_
#define MTTKRP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MTTKRP_MAX_ORDER 8

enum mttkrp_status {
    MTTKRP_OK = 0,
    MTTKRP_ERR_INVALID = 1,     /* bad argument: d, dims, R, mode, NULL, misalignment */
    MTTKRP_ERR_UNSUPPORTED = 2, /* valid, but not handled by the requested path */
    MTTKRP_ERR_WORKSPACE = 3,   /* no workspace set, or smaller than required */
    MTTKRP_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
    MTTKRP_ERR_HOST_ALLOC = 5,  /* host memory for the plan could not be allocated */
    MTTKRP_ERR_DEVICE = 6       /* a kernel reported a device-side error (bounded wait expired) */
};

/* Kernel family used for a mode.  AUTO lets the planner choose per mode. */
enum mttkrp_path {
    MTTKRP_PATH_AUTO = 0,
    MTTKRP_PATH_SIMT = 1,   /* fp32 FMA on the CUDA cores */
    MTTKRP_PATH_TC = 2,     /* tcgen05 tensor cores, fp32-accurate split (fp16 two-term or 3xTF32) */
    MTTKRP_PATH_TC_TF32 = 3, /* tcgen05 tensor cores, 3xTF32 split only (no fp16): for tensors whose
                                entries span more than the fp16 split's range (see mttkrp_plan) */
    MTTKRP_PATH_TC_EXPLICIT_KRP = 4 /* the matrix-based variant, for comparison: the Khatri-Rao
                                product of all modes but k is formed explicitly in the workspace
                                (4 * R * prod_{n != k} I_n bytes, plus padding) and Y_(k) is
                                multiplied by it on the tensor cores */
};

typedef struct mttkrp_plan_s* mttkrp_plan_t;

/*
 * Create a plan for a d-way tensor (2 <= d <= MTTKRP_MAX_ORDER) with the given
 * dims (each >= 1, product < 2^40) and rank R (1 <= R <= 65536).  Host-only:
 * validates, classifies every mode and chooses tiles and split counts; does
 * not touch the GPU.  *out receives an opaque handle owned by the library.
 * Returns MTTKRP_ERR_INVALID on bad arguments, MTTKRP_ERR_HOST_ALLOC if the
 * plan cannot be allocated.
 */
int mttkrp_plan(int d, const int64_t* dims, int64_t R, mttkrp_plan_t* out);

/* Force a kernel family for every mode (tests and benchmarks); AUTO restores
 * the planner's choice.  Returns MTTKRP_ERR_UNSUPPORTED if some mode cannot
 * run on that path.  Changes the workspace requirement. */
int mttkrp_plan_set_path(mttkrp_plan_t plan, int path);

/* Device workspace bytes needed by `mode` (0 <= mode < d), or the maximum over
 * all modes when mode == -1.  Returns 0 for an invalid plan or mode. */
size_t mttkrp_workspace_bytes(mttkrp_plan_t plan, int mode);

/* Attach caller-owned device scratch (256-byte aligned) of `bytes` bytes.
 * The plan keeps only the pointer; the caller keeps it alive while calls that
 * use it may still run on the GPU. */
int mttkrp_set_workspace(mttkrp_plan_t plan, void* dptr, size_t bytes);

/*
 * M_k for one mode.  Y: device pointer (16-byte alignment enables vector
 * loads; any 4-byte alignment works).  factors: HOST array of d device
 * pointers (factors[mode] is ignored).  out: device pointer to I_mode x R
 * floats.  stream: cudaStream_t as void*.  Enqueues the work and returns.
 */
int mttkrp(mttkrp_plan_t plan, const float* Y, const float* const* factors, int mode,
           float* out, void* stream);

/* M_k for every mode k = 0..d-1, back to back on one stream; outs is a HOST
 * array of d device pointers (outs[k] receives I_k x R floats). */
int mttkrp_all_modes(mttkrp_plan_t plan, const float* Y, const float* const* factors,
                     float* const* outs, void* stream);

/* Path the plan uses for `mode` (MTTKRP_PATH_SIMT or MTTKRP_PATH_TC), or -1. */
int mttkrp_plan_mode_path(mttkrp_plan_t plan, int mode);

/* Human-readable planner decisions for `mode` (tiles, split count, inner
 * group; tc_convert=1: when the mode is the first of a call to need the fp16
 * images of Y, its main kernel converts Y itself and writes the images, with
 * no separate pass) written into buf (NUL-terminated, truncated to len).
 * Returns the length the full text needs, or -1 for an invalid plan or mode. */
int mttkrp_plan_describe(mttkrp_plan_t plan, int mode, char* buf, size_t len);

/* Kernel timing for benchmarks.  When enabled (enable != 0), every call
 * records a pair of CUDA events on its stream around the main contraction
 * kernel of each mode; mttkrp_plan_kernel_times() waits for the recorded
 * events and copies up to `max` durations (milliseconds, in call order) of
 * `mode` into ms, returning how many were recorded since the last reset
 * (enable again to reset).  Events are created by the library (no device
 * memory is allocated).  Returns a negative value on error. */
int mttkrp_plan_set_timing(mttkrp_plan_t plan, int enable);
int mttkrp_plan_kernel_times(mttkrp_plan_t plan, int mode, float* ms, int max);

/* Number of kernels this plan has launched since it was created. */
int64_t mttkrp_plan_launch_count(mttkrp_plan_t plan);

/* Test hook for failure detection: the next `count` tensor-core kernel launches
 * withhold their first accumulator-ready signal, so the waiting warps' bounded
 * wait expires (after about one second), the kernel records a status bit,
 * drains its own copies and MMAs, frees its tensor memory and returns with an
 * incomplete result.  mttkrp_device_status() then reports the bit.  No fault,
 * trap or endless wait is involved.  count = 0 disarms it.  Returns the
 * previous count. */
int mttkrp_test_withhold_signal(int count);

/* Read and clear the device-side error word that kernels set when a bounded
 * wait expires (0 = none).  Synchronises the device.  Returns MTTKRP_OK or
 * MTTKRP_ERR_CUDA; the word is written to *word. */
int mttkrp_device_status(uint32_t* word);

void mttkrp_plan_destroy(mttkrp_plan_t plan);

const char* mttkrp_strerror(int code);

/* Last detailed error message of the calling thread ("" if none). */
const char* mttkrp_last_error(void);

/*
 * Allocation-free MTTKRP of one mode.  (No counterpart in the paper: this is a
 * deployment convenience of this library.)
 *
 * For callers that must not allocate device memory: a library embedded in a
 * program whose own allocator owns all of the GPU's memory and forbids other
 * allocations, or code on a latency-critical path where cudaMalloc/cudaFree,
 * which can block until the device is idle, are not acceptable.  Same result
 * as mttkrp() on the SIMT (CUDA-core) path, for the same d, dims, R, Y,
 * factors (HOST array of device pointers), mode, out and stream; no plan or
 * workspace is needed and nothing is allocated, on the host or the GPU.
 *
 * The scratch it needs lives in one static device array of
 * MTTKRP_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU that
 * loads the library holds until the process exits.  Problems whose scratch
 * would be larger (those with large split partial sums, e.g. a 128^4 tensor at
 * rank 256) are rejected with MTTKRP_ERR_WORKSPACE and a message, before any
 * work is enqueued.  The first call on a device looks up the array's device
 * address; make that first call before any stream capture.  Every call shares
 * the one array and leaves its contents behind; each call writes all the
 * scratch it reads, so nothing needs clearing, but calls that overlap on the
 * GPU (other streams or host threads at the same time) race on it.
 */
#define MTTKRP_NOALLOC_SCRATCH_BYTES (32u << 20)
int mttkrp_noalloc(int d, const int64_t* dims, int64_t R, const float* Y,
                   const float* const* factors, int mode, float* out, void* stream);

/*
 * CP-ALS sweep around the MTTKRP ("A Performance Portable Matrix Free Dense
 * MTTKRP in GenTen", Fig. 5: CP-ALS = per mode an MTTKRP plus the other
 * operations, an inner product and a Cholesky solve among them).  One call
 * updates every factor in turn, n = 0 .. d-1, each update using the newest
 * factors:
 *     V   = Hadamard product over m != n of A_m^T A_m        (R x R, fp64)
 *     M   = MTTKRP(Y, A, n)                                   (this plan)
 *     A_n = M V^{-1}  (Cholesky factor of V, fp64), then lambda_r = ||A_n(:, r)||_2
 *           and A_n(:, r) /= lambda_r (a zero column stays zero)
 * and then writes
 *     fit = 1 - ||Y - X||_F / ||Y||_F,  X = sum_r lambda_r a_r^(0) o ... o a_r^(d-1),
 * from ||X||^2 = lambda^T (Hadamard product of all Grams) lambda and
 * <Y, X> = sum_r lambda_r sum_i M(i, r) A_{d-1}(i, r) (M of the last mode).
 *
 * plan      a plan for Y's dims and the rank R; its workspace must be attached.
 * Y         device tensor (as for mttkrp).
 * factors   HOST array of d DEVICE pointers, each I_n x R fp32 row-major; all
 *           are read and overwritten with the normalised updated factors.
 * lambda    device, R fp32: the column norms of the last update (output).
 * norm_y2   device, one double: ||Y||_F^2.  If have_norm is 0 the call
 *           computes it first and stores it there.  have_norm = 1 states that
 *           Y is unchanged since the previous sweep on this plan and that no
 *           other call used the plan in between: the sweep then also reuses
 *           the max |Y| and fp16 images of Y that the previous sweep left in
 *           the plan's workspace, and, when it gets the same factor pointers
 *           and scratch as that sweep, the Gram matrices of the factors that
 *           sweep left in the scratch (so neither may change in between).
 * fit       device, one double (output); NaN if V was not positive definite.
 * scratch   device scratch of mttkrp_cp_als_scratch_bytes(plan) bytes, 256-byte
 *           aligned, caller-owned.
 * Enqueues on `stream` and returns without synchronising.  Errors: as mttkrp,
 * plus MTTKRP_ERR_WORKSPACE for a short scratch.
 */
size_t mttkrp_cp_als_scratch_bytes(mttkrp_plan_t plan);
int mttkrp_cp_als_sweep(mttkrp_plan_t plan, const float* Y, float* const* factors, float* lambda,
                        double* norm_y2, int have_norm, double* fit, void* scratch, size_t scratch_bytes,
                        void* stream);

/*
 * Givens rotations along one mode ("An HPC Approach to Accelerate Tensor
 * Decompositions", §2 and §4.3, "Application of Rotations"): Y is
 * multiplied in place in mode `mode` by R^T, where R is the identity except
 * for the 2 x 2 blocks [[c_g, -s_g], [s_g, c_g]] at rows and columns
 * (p_g, q_g) of a group of disjoint pivot pairs; for every fibre along the
 * mode,
 *     new[p_g] = c_g * old[p_g] + s_g * old[q_g],
 *     new[q_g] = c_g * old[q_g] - s_g * old[p_g],
 * and entries whose mode index is in no pair are not touched.
 *
 * d, dims   the tensor's order and shape (as for mttkrp_plan); Y is C-order
 *           fp32 device memory, 4-byte aligned (16-byte for vector access).
 * pairs     device, 2 * group_size int32: p_0, q_0, p_1, q_1, ...; the pairs
 *           must be disjoint (overlapping pairs race; indices out of range or
 *           p == q are skipped).
 * c, s      device, group_size fp32 each: cosine and sine of each rotation.
 * fp32 arithmetic (one fused multiply-add per output).  Enqueues on `stream`.
 * Errors: MTTKRP_ERR_INVALID for bad shapes, a mode out of range, a group
 * larger than half the mode size or NULL pointers; MTTKRP_ERR_CUDA.
 */
int mttkrp_apply_rotations(int d, const int64_t* dims, float* Y, int mode, const int32_t* pairs, const float* c,
                           const float* s, int group_size, void* stream);

/*
 * Dense mode-n product, TTM ("An HPC Approach to Accelerate Tensor
 * Decompositions", §2, eq. (1)): T = X x_mode M for a matrix M of size J x I_mode,
 *     T[i_0 .. i_{mode-1}, j, i_{mode+1} .. i_{d-1}]
 *         = sum over i of X[i_0 .. i_{mode-1}, i, i_{mode+1} .. i_{d-1}] * M[j, i].
 *
 * d, dims   X's order (1 <= d <= 8) and shape; X is C-order fp32 device memory.
 * M         device, J x dims[mode] fp32, row-major.
 * J         rows of M, 1 <= J <= 2^24; T has the shape of X with dims[mode]
 *           replaced by J (at most 2^40 elements, and at most 2^31 - 1 result
 *           tiles of 128 columns (p, q) x 32, 64 or 128 rows j).
 * T         device, caller-owned result buffer, C-order; must not overlap X or
 *           M.  Every element is written.
 * All pointers 4-byte aligned (16-byte alignment enables vector access).
 * fp32 products with fp32 accumulation over i in index order (fused
 * multiply-adds); the result does not depend on the launch configuration.
 * Enqueues on `stream` and returns without synchronising.
 * Errors: MTTKRP_ERR_INVALID for bad shapes, a mode out of range, J out of
 * range, NULL or misaligned pointers, or a result overlapping X or M;
 * MTTKRP_ERR_CUDA.
 */
int mttkrp_ttm(int d, const int64_t* dims, const float* X, int mode, const float* M, int64_t J, float* T,
               void* stream);

/*
 * The same mode-n product on the tensor cores, with a caller-owned workspace.
 * X viewed as [P, N, Q] (N = dims[mode]) and T as [P, J, Q]: T is computed as
 * the mode-0 MTTKRP of the two-way array Z[(p, q), i] = X[p, i, q] with the
 * single factor M^T (rank J) -- the fp16 two-term split of X (one power-of-two
 * scale for the whole tensor) and of M^T (a scale per column j), three
 * kind::f16 tensor-core products per fp32-accurate product, fp32 accumulation.
 *
 * mttkrp_ttm_workspace_bytes: device workspace bytes that path needs (about 4
 * bytes an element of X for its fp16 images, plus M^T and small tables), or 0
 * when it does not take the shape: J < 32, N < 16 or padded by more than half to
 * a multiple of 64, Q a multiple of 64 unless the mode is the innermost one (then
 * N a multiple of 8), more than 12 Gi elements, or more than 65535 x 128 rows
 * (p, q).  Returns 0 for invalid arguments too.
 * mttkrp_ttm_ws: arguments as mttkrp_ttm, plus workspace (device, 256-byte
 * aligned, caller-owned) of workspace_bytes bytes.  Runs on the tensor cores when
 * mttkrp_ttm_workspace_bytes() > 0, the workspace is that large and X is 16-byte
 * aligned; otherwise (no workspace, a shape the path does not take, a misaligned
 * X) it runs mttkrp_ttm's CUDA-core kernel.  Errors: as mttkrp_ttm, plus
 * MTTKRP_ERR_WORKSPACE for a workspace that is given but too small.
 */
size_t mttkrp_ttm_workspace_bytes(int d, const int64_t* dims, int mode, int64_t J);
int mttkrp_ttm_ws(int d, const int64_t* dims, const float* X, int mode, const float* M, int64_t J, float* T,
                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Several mode-n products of one tensor: T_t = X x_{modes[t]} Ms[t] for t <
 * nmodes (a Tucker form applies one product per mode, "An HPC Approach to
 * Accelerate Tensor Decompositions", §2, eq. (2)).  Each product is the one
 * mttkrp_ttm defines; the tensor-core products share one pass that writes the
 * fp16 images of X (and its scale), which is where the saving lies.
 *   mttkrp_ttm_multi_workspace_bytes: workspace bytes (device) for the products
 *     the tensor-core path takes: the images of X once plus the largest
 *     per-product region.  0 when none of them is taken, or for invalid
 *     arguments.
 *   mttkrp_ttm_multi: d, dims, X as mttkrp_ttm; modes (host, nmodes entries, each
 *     in [0, d), repeats allowed), Ms (host array of nmodes device pointers, Ms[t]
 *     Js[t] x dims[modes[t]] row-major), Js (host, nmodes entries >= 1), Ts (host
 *     array of nmodes device pointers, Ts[t] the result of product t, laid out as
 *     mttkrp_ttm's T; no T may overlap X, any M or another T).  workspace and
 *     workspace_bytes as mttkrp_ttm_ws: a product the tensor-core path takes runs
 *     there when the workspace is given and large enough and X is 16-byte aligned;
 *     every other product runs mttkrp_ttm's CUDA-core kernel.  The products are
 *     enqueued in order on `stream`; the call returns without waiting.
 * Errors: MTTKRP_ERR_INVALID (nmodes < 1 or above 64, NULL arrays, any product's
 * arguments as mttkrp_ttm checks them, overlapping results; nothing is enqueued),
 * MTTKRP_ERR_WORKSPACE (a workspace given but smaller than the bytes needed;
 * nothing is enqueued), MTTKRP_ERR_CUDA.
 */
size_t mttkrp_ttm_multi_workspace_bytes(int d, const int64_t* dims, int nmodes, const int* modes,
                                        const int64_t* Js);
int mttkrp_ttm_multi(int d, const int64_t* dims, const float* X, int nmodes, const int* modes,
                     const float* const* Ms, const int64_t* Js, float* const* Ts, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * Peak probes for the roofline of a benchmark (measurement only; the pages have
 * no counterpart).  Both enqueue one kernel on `stream` and return; the caller
 * times it with events.
 *   mttkrp_probe_fma: `blocks` x 256 threads, each running `iters` iterations of
 *     eight independent fp32 fused multiply-add chains; out (device, blocks x 256
 *     floats) receives each thread's sum.  flops = 16 x iters x blocks x 256.
 *   mttkrp_probe_mma: `blocks` CTAs (one per SM: launch as many as there are SMs),
 *     each with one thread issuing `iters` tcgen05 MMAs of M = 128, N = 256 back to
 *     back into tensor memory, kind::tf32 (kind 0, K = 8) or kind::f16 (kind 1,
 *     K = 16), on zero operands.  flops = 2 x 128 x 256 x K x iters x blocks.
 *     Its wait for the MMAs to finish is bounded (mttkrp_device_status reports
 *     an expiry).
 * Errors: MTTKRP_ERR_INVALID for bad counts or a NULL out; MTTKRP_ERR_CUDA.
 */
int mttkrp_probe_fma(int blocks, int iters, float* out, void* stream);
int mttkrp_probe_mma(int kind, int blocks, int iters, void* stream);

/* Library version as MAJOR * 10000 + MINOR * 100 + PATCH. */
int mttkrp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MTTKRP_H_ */
