// Internal declarations shared by the host planner and the kernel files of the
// MTTKRP library.  Nothing here is part of the C ABI (include/mttkrp.h).
//
// How a mode k is computed (the matrix-free scheme: the Khatri-Rao product is
// never formed).  Y is viewed as Y[p, i, q] with i = i_k, p the modes before k
// and q the modes after k.  The modes other than k are split into
//   * the inner group: the last few modes after k (when Q = prod_{n>k} I_n is
//     large enough), or all modes after k plus the last few modes before k;
//     its combined index j runs over J values;
//   * the pre modes: every other mode; their combined index is pi (npre values).
// Then  M_k(i, r) = sum_pi G(pi, r) sum_j Y(pi, i, j) Binner(j, r)  with
//   G(pi, r)     = prod over pre modes of A_n(i_n(pi), r)          (npre x R table)
//   Binner(j, r) = prod over inner-group modes of A_n(j_n(j), r)   (J x R table)
// so every Khatri-Rao row is G(pi, :) * Binner(j, :), built on the fly inside
// the kernels.  The two tables hold O(R (npre + J)) numbers, not the
// O(R prod_{n != k} I_n) of the explicit Khatri-Rao matrix.
//
// Offsets into Y: element (pi, i, j) sits at base(pi) + i * s_k + off(j) with
// off(j) = (j / Jq) * IQ + (j % Jq); Jq is the part of the inner group made of
// modes after k (contiguous in memory) and IQ the stride of mode k-1.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "mttkrp.h"

namespace mk {

constexpr int kMaxD = MTTKRP_MAX_ORDER;

struct ModeGeom {
    int k;
    int64_t I;     // rows of the output, I_k
    int64_t R;
    int64_t s_k;   // Y stride of mode k
    int64_t J;     // inner-group size
    int64_t Jq;    // part of J made of modes after k
    int64_t IQ;    // Y stride of mode k-1 (used only when J > Jq)
    int64_t npre;  // number of pre indices pi
    int ngroup;
    int group[kMaxD];  // inner-group modes, C order
    int npm;
    int pm[kMaxD];     // pre modes, C order
};

struct ModePlan {
    ModeGeom g;
    int path;           // MTTKRP_PATH_SIMT or MTTKRP_PATH_TC
    int bm, bn;         // output tile (rows x columns)
    int64_t splits;     // number of contiguous pi ranges (1 = split-free)
    int64_t pre_per_split;
    // tensor-core path only
    int tc_inner;       // 1: mode with stride 1 (Y tile arrives i-major and is transposed)
    int tc_ks;          // K-steps of 16 contraction indices per pi
    int tc_jq_steps;    // K-steps per value of the p-side part of the inner group
    int tc_small;       // 1: small I_k, tc_ps pre indices share one 128-row tile
    int tc_ps;
    int tc_tmem;        // 1: A operand staged in tensor memory (128 x 224 tiles, large R)
    int tc_h2;          // 1: two-term fp16 split (kind::f16, K-steps of 32); implies tc_tmem
    int tc_kw;          // contraction indices per K-step (16; 32 with tc_h2; 64 with tc_img)
    int tc_img;         // 1: two-term fp16 split from pre-split fp16 images of Y, both
                        //    operands in shared memory (K-steps of 64)
    int tc_img_t;       // tc_img for the innermost mode: from the transposed images
                        //    (Y viewed as P x I_{d-1}, stored I_{d-1} x P)
    int tc_img_mn;      // tc_img for the innermost mode: from the natural images, A read
                        //    MN-major (i contiguous) by the tensor cores
    // explicit Khatri-Rao product (the matrix-based comparison variant): the
    // inner group is every mode but k (one pre index), the B images hold the
    // whole product, and the contraction is split over B chunks, jc_per_split
    // chunks a CTA
    int explicit_krp;
    int jc_per_split;
    // workspace layout, byte offsets from the workspace base
    size_t off_partials, off_binner, off_gtab, off_base, total;
    size_t off_t1;      // explicit_krp: product of the inner group's factors but the last one
    size_t off_end;     // end of the mode's own regions (before plan-level regions)
    size_t off_img;     // tc_img: fp16 hi image of Y, then the lo image (shared by all modes)
    size_t off_timg;    // tc_img: the transposed hi and lo images
};

struct Plan {
    int d;
    int64_t dims[kMaxD];
    int64_t strides[kMaxD];
    int64_t R;
    int forced_path;
    ModePlan mode[kMaxD];
    // SIMT plan of every mode, used when a tensor-core mode is called with a
    // Y pointer that the tensor-memory accelerator cannot address (not 16-byte
    // aligned); its workspace need is included in mode[k].total
    ModePlan simt_alt[kMaxD];
    void* ws;
    size_t ws_bytes;
    int64_t launches;  // kernels launched so far
    // max |Y| (fp16-split path) already computed for the current call's Y
    mutable int ymax_ready;
    // fp16 images of Y (tc_img modes) already written for the current call's Y
    mutable int img_ready;
    // the next tensor-core launch converts Y in place and writes the images
    // (set by tc_prepare, cleared once the launch and its exact redo are enqueued)
    mutable int fuse_pending;
    // the mode whose main kernel converts Y when it is the first fp16 mode of a
    // call (-1: none); an all-modes call computes it first
    int fuse_mode;
    int img_nat, img_t;   // which images the plan's tc_img modes read (natural, transposed)
    // fp16 split: largest |Y| of every slab of mode 0 (fp32 bits) at off_slab in
    // the workspace.  nslab = I_0 when every fp16-split mode of the plan takes
    // per-slab scales (mode 0 is its output row or a pre mode), else 1 (one
    // scale for the whole tensor).
    int slab_on;
    int64_t nslab;
    size_t off_slab;
    // the last call on this plan was a CP-ALS sweep: max |Y| and the fp16 images
    // in the workspace are those of that sweep's Y
    int sweep_left_images;
    // and its scratch and factor pointers: a continuing sweep with the same ones
    // reuses the Gram matrices that sweep left in the scratch
    const void* sweep_scratch;
    const float* sweep_factors[kMaxD];
    // benchmark timing: event pairs around the main kernel of each mode
    int timing;
    int ev_cap[kMaxD];
    int ev_n[kMaxD];
    cudaEvent_t* ev_start[kMaxD];
    cudaEvent_t* ev_stop[kMaxD];
};

// Product table: row t of `tab` (R wide) = prod over the nm listed modes of
// fac[m](idx_m(t), r), idx decoded from t in C order over dim[]; base[t] (if
// non-null) = sum_m idx_m(t) * ystride[m].  nm = 0 gives rows of ones.
struct ProdTableArgs {
    int nm;
    int64_t dim[kMaxD];
    int64_t ystride[kMaxD];
    const float* fac[kMaxD];
    int64_t rows;
    int64_t R;
    float* tab;
    int64_t* base;
    // optional (fp16-split G tables with per-slab scales of Y): row t is also
    // multiplied by s_global / s_slab(t / slab_div), a power of two <= 1
    const uint32_t* slab_bits;
    const uint32_t* gmax_bits;
    int64_t slab_div;
    // non-null: the kernel runs only if *enable is set
    const uint32_t* enable;
};

struct SimtArgs {
    const float* Y;
    const float* binner;  // J x R
    const float* gtab;    // npre x R
    const int64_t* base;  // npre
    float* dst;           // out (splits == 1) or partials [splits][I][R]
    int64_t dst_split_stride;
    int64_t I, R, J, Jq, IQ, s_k, npre, pre_per_split;
};

// Y loader variants of the SIMT kernel
enum { kLoadScalar = 0, kLoadVecJ = 1, kLoadVecI = 2 };

cudaError_t launch_prod_table(const ProdTableArgs& a, cudaStream_t s);

// Givens rotations along one mode (rotations.cu); Y viewed as [P, N, Q]
cudaError_t launch_rotations(float* Y, int64_t P, int N, int64_t Q, const int* pairs, const float* c, const float* s,
                             int G, cudaStream_t stream);

// dense mode-n product T = X x_n M (ttm.cu); X [P, N, Q], M [J, N], T [P, J, Q]
int ttm_row_tile(int64_t J);
int64_t ttm_tiles(int64_t P, int64_t Q, int64_t J);
cudaError_t launch_ttm(const float* X, const float* M, float* T, int64_t P, int64_t N, int64_t Q, int64_t J,
                       cudaStream_t s);

// CP-ALS pieces (cpals.cu)
int cpals_gram_slabs(int64_t I, int R);   // partial Grams cpals_gram keeps (R x R fp64 each)
cudaError_t cpals_gram(const float* A, int64_t I, int R, double* G, double* part, cudaStream_t s);
// V = Hadamard product of the Grams but skip's; vhi, vlo (nullable): V as two fp32 words
cudaError_t cpals_hadamard(const double* G, int d, int skip, int R, double* V, float* vhi, float* vlo,
                           cudaStream_t s);
// lower Cholesky factor of V in place; dinv (R) receives the reciprocals of its diagonal
cudaError_t cpals_cholesky(double* V, int R, int* info, double* dinv, cudaStream_t s);
int cpals_cholesky_launches(int R);
// X = M (L L^T)^{-1}; mirrors L into the strict upper triangle of its storage first
cudaError_t cpals_solve(double* L, const double* dinv, int R, const float* M, int64_t I, double* X,
                        cudaStream_t s);
// A(:, r) = X(:, r) / ||X(:, r)||, lam[r] = ||X(:, r)|| (part: cpals_normalize_scratch_bytes(R))
size_t cpals_normalize_scratch_bytes(int R);
int cpals_normalize_launches();
cudaError_t cpals_normalize(const double* X, int64_t I, int R, float* A, float* lam, double* part, cudaStream_t s);
// fit = 1 - ||Y - X|| / ||Y|| (part: cpals_sumsq_scratch_bytes() of fp64 scratch)
cudaError_t cpals_fit(const double* H, const float* lam, const float* M, const float* A, int64_t I, int R,
                      const double* norm_y2, const int* info, double* fit, double* part, cudaStream_t s);
// X = M V^{-1} (fp64 out) for R <= cpals_mixed_max_rank(): V and its two fp32
// words (vhi, vlo: R x R each, as cpals_hadamard wrote them), factored in fp32
// (L: R x R, dinv: R; dblk:
// cpals_mixed_block_bytes(R), the inverted diagonal blocks, 16-byte aligned),
// rows solved in fp32 into x0 (I x R), residual M - x0 V (res: I x R) solved and
// added
int cpals_mixed_max_rank();
int cpals_mixed_launches(int R);
size_t cpals_mixed_block_bytes(int R);
cudaError_t cpals_solve_mixed(const double* V, int R, const float* M, int64_t I, double* X, float* vhi, float* vlo,
                              float* L, float* dinv, float* dblk, float* x0, float* res, int* info, cudaStream_t s);
size_t cpals_sumsq_scratch_bytes();
cudaError_t cpals_sum_squares(const float* Y, int64_t n, double* part, double* out, cudaStream_t s);
cudaError_t launch_reduce_splits(const float* part, int64_t splits, int64_t n, float* out,
                                 cudaStream_t s);
cudaError_t launch_simt(int bm, int bn, int amode, bool bvec, const SimtArgs& a,
                        int64_t splits, cudaStream_t s);
bool simt_tile_supported(int bm, int bn);
// peak probe of the fp32 FMA pipe (blocks x 256 threads; out: blocks x 256 floats)
cudaError_t launch_fma_probe(int blocks, int iters, float* out, cudaStream_t s);

}  // namespace mk
