// msda_launch.h -- internal interface between the C-ABI layer (msda_api.cu)
// and the kernel launchers.  Not installed, not part of the C ABI.
#pragma once

#include <cuda_runtime.h>

#include "msda_device.cuh"

namespace msda {

// Everything the kernels need to know about the sizes and the levels; filled
// and checked on the host by msda_api.cu.
struct LaunchGeometry {
    Dims d;                 // d.M: sets of locations (heads, or head groups)
    LevelTable lv;
    unsigned char level_of[kMaxSamples];
    int D;                  // channels sampled with one set: head_dim, or heads per group * head_dim
};

cudaError_t launch_forward(const LaunchGeometry &g, int dtype, int D, const void *value, const float *loc,
                           const float *attn, void *out, cudaStream_t stream);

cudaError_t launch_forward_fused(const LaunchGeometry &g, int dtype, int D, const void *value, const float *ref,
                                 const float *off, const float *logits, void *out, cudaStream_t stream);

// Bytes of workspace for the deterministic backward: a header of one 32-bit
// scale bound per batch element (padded to 256 bytes), then the fixed-point
// accumulators.
size_t backward_workspace_bytes(const LaunchGeometry &g, int D, bool deterministic);

cudaError_t launch_backward(const LaunchGeometry &g, int dtype, int D, const void *value, const float *loc,
                            const float *attn, const void *grad_out, float *grad_value, float *grad_loc,
                            float *grad_attn, bool deterministic, bool accumulate, void *workspace,
                            cudaStream_t stream);

// Fused backward: gradients with respect to the raw reference points,
// sampling offsets (pixels of their level) and attention logits.
cudaError_t launch_backward_fused(const LaunchGeometry &g, int dtype, int D, const void *value, const float *ref,
                                  const float *off, const float *logits, const void *grad_out, float *grad_value,
                                  float *grad_ref, float *grad_off, float *grad_logits, bool det, bool accumulate,
                                  void *workspace, cudaStream_t stream);

// grad_value preparation (zeroing, or deterministic accumulators and one scale
// bound per batch element) and completion (fixed point to fp32), shared by the
// 2-D and 3-D backward.  attn == nullptr: the weights are softmax outputs whose
// rows sum to row_sum.
cudaError_t backward_prepare(const LaunchGeometry &g, int dtype, int D, const float *attn, float row_sum,
                             const void *grad_out, float *grad_value, bool det, bool accumulate, void *workspace,
                             unsigned long long **fixed, const unsigned **bound, cudaStream_t stream);
cudaError_t backward_finish(const LaunchGeometry &g, int D, float *grad_value, bool det, bool accumulate,
                            const unsigned long long *fixed, const unsigned *bound, cudaStream_t stream);

// 3-D (trilinear) variant: volumes (Dz, H, W) per level.
struct LevelTable3 {
    int Dz[kMaxLevels], H[kMaxLevels], W[kMaxLevels], start[kMaxLevels];
    float Dzf[kMaxLevels], Hf[kMaxLevels], Wf[kMaxLevels];
    float Sx[kMaxLevels], Sy[kMaxLevels], Sz[kMaxLevels];   // pixel scales (size, or size - 1)
    float shift;                                            // 0.5, or 0 with align_corners
};

struct LaunchGeometry3 {
    LaunchGeometry g;      // sizes, sample -> level map (its level table is unused)
    LevelTable3 lv;
};

cudaError_t launch_forward3d(const LaunchGeometry3 &g, int dtype, int D, const void *value, const float *loc,
                             const float *attn, void *out, cudaStream_t stream);
cudaError_t launch_backward3d(const LaunchGeometry3 &g, int dtype, int D, const void *value, const float *loc,
                              const float *attn, const void *grad_out, float *grad_value, float *grad_loc,
                              float *grad_attn, bool det, bool accumulate, void *workspace, cudaStream_t stream);

#ifdef MSDA_DEBUG
// debug build: each kernel translation unit's count of skipped bad accesses
// (reset: zero it after reading)
unsigned long long debug_count_forward(bool reset);
unsigned long long debug_count_backward(bool reset);
unsigned long long debug_count_3d(bool reset);
#endif

}  // namespace msda
