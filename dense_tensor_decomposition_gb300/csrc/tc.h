// Tensor-core (tcgen05 / TMEM) path of the MTTKRP library: planner hooks and
// launcher.  See tc.cu for the kernel.
#pragma once

#include "internal.h"

namespace mk {

// Bytes of workspace the tensor-core path needs for its pre-split inner table.
size_t tc_binner_bytes(const ModePlan& mp);
// Whether the planner should choose the tensor-core path for this mode.
bool tc_prefer(const ModePlan& mp);
// Fill tiles and split counts for the tensor-core path; false if unsupported.
// allow_fp16 = false keeps the mode on the 3xTF32 kernels.
bool tc_plan(const Plan& p, ModePlan& mp, bool allow_fp16);
// Enqueue the passes over Y that an fp16-split mode needs before its tables are
// built: the largest magnitude of every slab of mode 0 and of the whole tensor
// (once per call), and the fp16 images of Y (tc_img modes, once per call).
// ws is the workspace base; *nlaunch receives the number of kernels enqueued.
int tc_prepare(const Plan& p, const ModePlan& mp, const float* Y, void* ws, cudaStream_t stream, int* nlaunch,
               char* errbuf, size_t errlen);
// Enqueue the tensor-core work of one mode (tables are already built).
// *nlaunch receives the number of kernels enqueued.  If start_ev is non-null,
// *start_ev is re-recorded just before the main kernel (after the tensor-core
// path's own preparation kernels) so that timing covers the main kernel only.
// With p.fuse_pending the main kernel converts Y in place and writes the images.
int tc_run(const Plan& p, const ModePlan& mp, const float* Y, const float* const* factors,
           const float* gtab, const int64_t* basetab, void* binner_ws, float* dst,
           cudaStream_t stream, int* nlaunch, cudaEvent_t* start_ev, char* errbuf, size_t errlen);
// After a converting launch (p.fuse_pending), each a launch that returns at
// once unless the conversion flagged a scaled value outside the fp16 range:
// tc_redo_images takes the exact maxima and writes the images; (the caller
// then rebuilds the mode's G table if it carries slab scales, gated on
// tc_redo_flag) tc_redo_main runs the mode's main kernel again on the images
// and clears p.fuse_pending.  The inputs are those of the tc_run they follow.
int tc_redo_images(const Plan& p, const ModePlan& mp, const float* Y, void* ws, cudaStream_t stream, int* nlaunch,
                   char* errbuf, size_t errlen);
const uint32_t* tc_redo_flag(const Plan& p, void* ws);
int tc_redo_main(const Plan& p, const ModePlan& mp, const float* Y, const float* const* factors,
                 const float* gtab, const int64_t* basetab, void* binner_ws, float* dst,
                 cudaStream_t stream, int* nlaunch, char* errbuf, size_t errlen);
// Whether a mode's main kernel can convert Y in place (natural K-major image
// tiles in one column tile, an inner group of whole modes after
// it, no transposed images in the plan).
bool tc_fuse_eligible(const Plan& p, const ModePlan& mp);
// The mode the plan converts in (p.fuse_mode): among the eligible modes, one
// whose tiles cover contiguous memory (stride of the mode = inner-group size),
// else the first; -1 if none.
int tc_pick_fuse_mode(const Plan& p);
// Peak probe of the tensor pipe: `blocks` CTAs (one per SM), each issuing `iters`
// M128 x N256 MMAs of kind::tf32 (kind 0, K = 8) or kind::f16 (kind 1, K = 16).
cudaError_t tc_launch_mma_probe(int kind, int blocks, int iters, cudaStream_t s);
// Mode-n product T = X x_n M on the tensor cores (X viewed [P, N, Q], M J x N, T
// [P, J, Q]): workspace bytes it needs (0: the shape is not taken), and the run.
size_t tc_ttm_workspace_bytes(int64_t P, int64_t N, int64_t Q, int64_t J);
int tc_ttm_run(const float* X, const float* M, float* T, int64_t P, int64_t N, int64_t Q, int64_t J, void* ws,
               cudaStream_t stream, char* errbuf, size_t errlen);
// The same in two parts, so that several products of one X share the first:
// tc_ttm_images writes the fp16 images of X (numel elements) and their scale at
// the start of ws; tc_ttm_product runs one product on them.  Every product of
// one X places the images at the same offset, so the workspace of several is
// the largest tc_ttm_workspace_bytes among them.
int tc_ttm_images(const float* X, int64_t numel, void* ws, cudaStream_t stream, char* errbuf, size_t errlen);
int tc_ttm_product(const float* M, float* T, int64_t P, int64_t N, int64_t Q, int64_t J, void* ws,
                   cudaStream_t stream, char* errbuf, size_t errlen);
// Device address of the error word on the current device (null on failure).
uint32_t* tc_status_ptr();
// Arm the failure-detection test hook for the next `count` launches.
int tc_set_withhold_signal(int count);
// Read and clear the device-side error word (synchronises the device).
cudaError_t tc_read_and_clear_status(uint32_t* word);

}  // namespace mk
