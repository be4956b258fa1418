/*
 * msda.h -- C ABI of libmsda, the multi-scale deformable attention
 * (MSDeformAttn) core for NVIDIA B300 (sm_103a).
 *
 * What the library computes.  For every batch element n, query q and head m,
 * the core samples a head_dim-channel vector from each of n_levels flattened
 * feature levels at n_points locations each, bilinearly, weights every sample
 * by its attention weight and sums them:
 *
 *   out[n][q][m*D + d] = sum_{l,k} A[n,q,m,l,k] * bilinear_l(value[n,:,m,d], loc[n,q,m,l,k])
 *
 * This is the inner sum of the MSDeformAttn formula, "可变形注意力：多尺度稀疏
 * 采样与视觉检测实战解析" §2.2 (and "可变形 DETR：加速收敛的稀疏注意力检测器"
 * §3.3); the value, offset, weight and output projections around it are not
 * part of this library.  Bilinear sampling follows that tutorial's §2.3 and the
 * grid_sample module of its §3.2: the pixel coordinate of a normalised
 * location is px = loc_x * W_l - 0.5, py = loc_y * H_l - 0.5 (align_corners
 * = False), the four integer neighbours are weighted (1-|dx|)(1-|dy|), and a
 * neighbour outside [0,W_l) x [0,H_l) contributes zero while the others keep
 * their weights (padding_mode = 'zeros').
 *
 * Conventions shared by every call:
 *   - All tensors are dense, row-major, and live in device memory owned by
 *     the caller, except spatial_shapes and level_start_index, which are
 *     HOST arrays (read during the call, not retained).  The library never
 *     allocates memory; temporary memory comes from the caller (workspace).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and enqueues work on the current CUDA device.
 *     A call returns after launching, not after the kernels finish.
 *   - Arguments are checked on the host before any launch.  A failed check
 *     returns MSDA_ERR_INVALID_ARG or MSDA_ERR_UNSUPPORTED and launches
 *     nothing; msda_last_error() then describes the failure (thread-local).
 *   - A launch failure returns MSDA_ERR_CUDA (cudaGetLastError after launch).
 *   - Calls with N == 0 or Len_q == 0 launch no sampling work; they still
 *     zero grad_value where the call says it does.
 *   - Inputs are assumed finite.  A non-finite value may reach samples whose
 *     corners fall outside the map (their loads are kept, with weight 0).
 *
 * Layouts (D = head_dim, M = n_heads, L = n_levels, K = n_points):
 *   value               [N][Len_in][M][D]            dtype (f32 or bf16)
 *   spatial_shapes      [L][2] = (H_l, W_l)           int64, host
 *   level_start_index   [L]                           int64, host;
 *                       level_start_index[0] = 0, [l+1] = [l] + H_l*W_l,
 *                       Len_in = sum_l H_l*W_l
 *   sampling_locations  [N][Len_q][M][L][K][2]        f32, (x, y), normalised
 *   attention_weights   [N][Len_q][M][L][K]           f32
 *   output              [N][Len_q][M*D]               dtype
 *   reference_points    [N][Len_q][L][2]              f32, (x, y), normalised
 *   sampling_offsets    [N][Len_q][M][L][K][2]        f32, in pixels of level l
 *   attention_logits    [N][Len_q][M][L*K]            f32
 *   grad_output         [N][Len_q][M*D]               dtype
 *   grad_value          [N][Len_in][M][D]             f32 (for both dtypes)
 *   grad_sampling_locations [N][Len_q][M][L][K][2]    f32
 *   grad_attention_weights  [N][Len_q][M][L][K]       f32
 *
 * Head groups (msda_problem.n_groups = G, 0 for G = M): the M heads form G
 * groups of M / G consecutive heads that share one set of locations and
 * weights (the DAT pages' sampler: one offset field per group of channels,
 * "un.csdn.net/yx18yrw9d9z8" §2.1-2.2).  Every per-sample tensor then has G in
 * place of M: sampling_locations [N][Len_q][G][L][K][2], attention_weights
 * [N][Len_q][G][L][K], sampling_offsets [N][Len_q][G][L][K][2],
 * attention_logits [N][Len_q][G][L*K] and their gradients; head m samples with
 * the set of group m / (M / G).  value, output and grad_value keep their
 * layouts.
 *
 * Supported: (M / G) * head_dim (the channels one set samples; head_dim when
 * G = M) a power of two from 8 to 256 (to 64 for the 3-D calls);
 * 1 <= n_levels <= 16; 1 <= n_levels * n_points <= 256; N*Len_q*G < 2^31;
 * (Len_in + 2*max W_l + 4) * M * D < 2^31.  value/output/grad_output/grad_value must be 16-byte
 * aligned, sampling_locations/reference_points/sampling_offsets 8-byte
 * aligned, the other f32 tensors 4-byte aligned.
 */
#ifndef MSDA_H_
#define MSDA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MSDA_API __attribute__((visibility("default")))
#else
#define MSDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum msda_status {
    MSDA_OK = 0,
    MSDA_ERR_INVALID_ARG = 1,   /* a null pointer, a bad size, inconsistent levels */
    MSDA_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels handle */
    MSDA_ERR_CUDA = 3,          /* the CUDA runtime reported an error */
    MSDA_ERR_WORKSPACE = 4      /* workspace missing, too small or misaligned */
} msda_status;

/* Storage type of value, output and grad_output.  Arithmetic is fp32. */
typedef enum msda_dtype {
    MSDA_F32 = 0,
    MSDA_BF16 = 1               /* bf16 storage, fp32 accumulation, RNE rounding of output */
} msda_dtype;

/* Sizes of one call (names follow the tutorial module's interface, §3.1). */
typedef struct msda_problem {
    int32_t N;          /* batch size */
    int32_t Len_in;     /* flattened value length, sum of H_l*W_l */
    int32_t n_heads;    /* M */
    int32_t head_dim;   /* D, channels per head */
    int32_t Len_q;      /* number of queries */
    int32_t n_levels;   /* L */
    int32_t n_points;   /* K, samples per level per head */
    int32_t dtype;      /* msda_dtype */
    uint32_t options;   /* MSDA_OPT_* bits, 0 for the default method */
    int32_t n_groups;   /* G: groups of heads sharing one set of locations and
                           weights; 0 (or n_heads) for one set per head */
} msda_problem;

/* msda_problem.options: readings of the method the pages leave open.
 *
 * MSDA_OPT_PER_LEVEL_SOFTMAX  the fused calls normalise the n_points logits
 *     of each level separately ("可变形注意力…" §2.2 prose: the normalisation
 *     runs over k for each level) instead of all n_levels*n_points of the
 *     (query, head) (its §3.2 module code; the default).  The unfused calls
 *     take the weights as given and ignore this bit.
 * MSDA_OPT_ALIGN_CORNERS  pixel coordinate px = loc_x * (W_l - 1),
 *     py = loc_y * (H_l - 1): pixel centres at i / (W_l - 1), as a sampler
 *     with grid_sample(align_corners=True) places them (the DAT pages'
 *     sampler).  The fused location is still loc = ref + off / (W_l, H_l);
 *     gradients follow (d px / d loc_x = W_l - 1).  Default: px = loc_x * W_l
 *     - 0.5 (align_corners=False). */
#define MSDA_OPT_PER_LEVEL_SOFTMAX  1u
#define MSDA_OPT_ALIGN_CORNERS      2u

/* msda_backward flags */
#define MSDA_DETERMINISTIC          1u  /* bitwise reproducible grad_value (fixed-point sums) */
#define MSDA_ACCUMULATE_GRAD_VALUE  2u  /* add into grad_value instead of overwriting it */

/*
 * msda_forward -- steps a3-a5: bilinear multi-level sampling, weighted sum.
 * "可变形注意力：多尺度稀疏采样与视觉检测实战解析" §2.2 (formula), §2.3
 * (bilinear, zero padding), §3.2 steps 4-5 (per-level sampling, weighted sum).
 *
 *   value               in   [N][Len_in][M][D], dtype
 *   spatial_shapes      in   host [L][2] (H, W)
 *   level_start_index   in   host [L]
 *   sampling_locations  in   [N][Len_q][M][L][K][2] f32
 *   attention_weights   in   [N][Len_q][M][L][K] f32 (used as given; no softmax)
 *   output              out  [N][Len_q][M*D], dtype; fully overwritten
 */
MSDA_API msda_status msda_forward(const msda_problem *problem, const void *value,
                         const int64_t *spatial_shapes, const int64_t *level_start_index,
                         const float *sampling_locations, const float *attention_weights,
                         void *output, void *stream);

/*
 * msda_forward_fused -- steps a1-a5 in one launch: the sampling location
 * loc = ref + off / (W_l, H_l) ("可变形 DETR：加速收敛的稀疏注意力检测器" §6,
 * reference_points + sampling_offsets / scale_factors), the softmax of the
 * raw logits over all L*K samples of one (query, head) (the tutorial module
 * of "可变形注意力…" §3.2: softmax over n_levels*n_points), then the sampling
 * of msda_forward.  Locations and weights stay in registers.
 *
 *   reference_points    in   [N][Len_q][L][2] f32, normalised (x, y)
 *   sampling_offsets    in   [N][Len_q][M][L][K][2] f32, pixels of level l
 *   attention_logits    in   [N][Len_q][M][L*K] f32
 *   output              out  [N][Len_q][M*D], dtype; fully overwritten
 */
MSDA_API msda_status msda_forward_fused(const msda_problem *problem, const void *value,
                               const int64_t *spatial_shapes, const int64_t *level_start_index,
                               const float *reference_points, const float *sampling_offsets,
                               const float *attention_logits, void *output, void *stream);

/*
 * Bytes of device workspace msda_backward and msda_backward_fused need for `flags` (0 unless
 * MSDA_DETERMINISTIC is set).  Host-only, launches nothing.
 */
MSDA_API size_t msda_backward_workspace_size(const msda_problem *problem, unsigned flags);

/*
 * msda_backward -- steps a6-a8, the gradient of msda_forward, derived from
 * the bilinear form of "可变形注意力…" §2.3 (continuous, so the gradient
 * reaches the offset branch).  With g = grad_output[n][q][m*D..]:
 *   grad_attention_weights[s]  = <g, sample_s>
 *   grad_sampling_locations[s] = A_s * <g, d sample_s / d(px, py)> * (W_l, H_l)
 *   grad_value[n][corner][m]  += A_s * w_corner * g      (corners inside the map)
 * At an integer pixel coordinate the location gradient is the one-sided
 * derivative of the cell that floor() selects.
 *
 *   grad_output            in   [N][Len_q][M*D], dtype
 *   grad_value             out  [N][Len_in][M][D] f32; zeroed first unless
 *                               MSDA_ACCUMULATE_GRAD_VALUE
 *   grad_sampling_locations out [N][Len_q][M][L][K][2] f32, overwritten
 *   grad_attention_weights out  [N][Len_q][M][L][K] f32, overwritten
 *   flags                  in   MSDA_DETERMINISTIC | MSDA_ACCUMULATE_GRAD_VALUE
 *   workspace              in   device memory of at least
 *                               msda_backward_workspace_size() bytes, 256-byte
 *                               aligned (may be NULL when that size is 0);
 *                               its contents on entry do not matter.
 * Default mode sums grad_value with fp32 atomics, so its low bits vary from
 * run to run.  MSDA_DETERMINISTIC sums in 64-bit fixed point, scaled from a
 * bound on the total so that no sum can overflow, then converts to fp32: the
 * result is bitwise identical from run to run.  The scale is chosen per batch
 * element from that element's rows alone, so a batch element's grad_value does
 * not depend on the other batch elements of the call: splitting a batch over
 * several calls (or GPUs) gives bitwise the same result.
 * grad_sampling_locations and grad_attention_weights are bitwise reproducible
 * in both modes, and depend only on their own (query, head) row.
 */
MSDA_API msda_status msda_backward(const msda_problem *problem, const void *value,
                          const int64_t *spatial_shapes, const int64_t *level_start_index,
                          const float *sampling_locations, const float *attention_weights,
                          const void *grad_output, float *grad_value,
                          float *grad_sampling_locations, float *grad_attention_weights,
                          unsigned flags, void *workspace, size_t workspace_bytes, void *stream);

/*
 * msda_backward_fused -- the gradient of msda_forward_fused: through the
 * sampling of msda_backward, then the location step loc = ref + off / (W_l, H_l)
 * ("可变形 DETR：加速收敛的稀疏注意力检测器" §6) and the softmax over the L*K
 * logits of one (query, head) ("可变形注意力…" §3.2 module):
 *   grad_sampling_offsets[s] = A_s * d/d(px, py)          (pixels of level l)
 *   grad_reference_points[n][q][l] = sum over heads m and points k of the
 *                              location gradient A_s * (W_l, H_l) * d/d(px, py)
 *   grad_attention_logits[s] = A_s * (g_s - sum_t A_t g_t),  g_s = <grad_output, sample_s>
 *   grad_value              as msda_backward, with A = softmax(logits)
 * The location and the softmax are recomputed from the raw inputs with the
 * arithmetic of msda_forward_fused, so the samples are the ones that call took.
 *
 *   reference_points       in   [N][Len_q][L][2] f32
 *   sampling_offsets       in   [N][Len_q][M][L][K][2] f32, pixels of level l
 *   attention_logits       in   [N][Len_q][M][L*K] f32
 *   grad_output            in   [N][Len_q][M*D], dtype
 *   grad_value             out  [N][Len_in][M][D] f32; zeroed first unless
 *                               MSDA_ACCUMULATE_GRAD_VALUE
 *   grad_reference_points  out  [N][Len_q][L][2] f32, overwritten
 *   grad_sampling_offsets  out  [N][Len_q][M][L][K][2] f32, overwritten
 *   grad_attention_logits  out  [N][Len_q][M][L*K] f32, overwritten
 *   flags, workspace       as msda_backward (same workspace size)
 * Every output except grad_value is bitwise reproducible in both modes;
 * grad_value is under MSDA_DETERMINISTIC.
 */
MSDA_API msda_status msda_backward_fused(const msda_problem *problem, const void *value,
                                         const int64_t *spatial_shapes, const int64_t *level_start_index,
                                         const float *reference_points, const float *sampling_offsets,
                                         const float *attention_logits, const void *grad_output, float *grad_value,
                                         float *grad_reference_points, float *grad_sampling_offsets,
                                         float *grad_attention_logits, unsigned flags, void *workspace,
                                         size_t workspace_bytes, void *stream);

/*
 * msda_backward_noalloc -- msda_backward in MSDA_DETERMINISTIC mode without a
 * caller workspace.  The pages have no counterpart of this entry point; it
 * exists for callers that cannot allocate device memory: a plugin that a host
 * application hands only its input and output buffers (and that may not call
 * cudaMalloc or the host's allocator), or a loop that must not allocate after
 * start-up because cudaMalloc/cudaFree can synchronize the device.
 *
 * The scratch lives in the library: one 64 MiB device array (fixed-point
 * accumulators, 8 bytes per grad_value element, after a header of 4 bytes per
 * batch element rounded up to 256), which every GPU that loads the library
 * holds until the process exits.  A problem that needs more (for N <= 64: one
 * with N * Len_in * n_heads * head_dim above 8,388,576 elements) is rejected
 * with MSDA_ERR_UNSUPPORTED before anything is launched; use msda_backward
 * with a workspace for it.
 *
 * Same arguments, results and checks as msda_backward with
 * flags = MSDA_DETERMINISTIC, except that there is no workspace and `flags`
 * accepts only MSDA_ACCUMULATE_GRAD_VALUE.  The call allocates nothing: no
 * cudaMalloc, no cudaFree.
 *
 * The first call on a device looks up the device address of the scratch
 * array (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  That address is cached per device for the life
 * of the process and is not looked up again: cudaDeviceReset destroys the
 * context that holds the array, so after a reset of a device this entry point
 * must not be called on it again in the same process (msda_backward with a
 * workspace has no such limit).  Every call clears the part of the scratch it
 * uses before summing into it.  All calls on one device share the one
 * array, so calls whose kernels overlap on the GPU (on different streams, or
 * from different threads) race on it and give wrong results: order them on
 * one stream or synchronize between them.
 */
MSDA_API msda_status msda_backward_noalloc(const msda_problem *problem, const void *value,
                                           const int64_t *spatial_shapes, const int64_t *level_start_index,
                                           const float *sampling_locations, const float *attention_weights,
                                           const void *grad_output, float *grad_value,
                                           float *grad_sampling_locations, float *grad_attention_weights,
                                           unsigned flags, void *stream);

/*
 * msda3d_forward / msda3d_backward -- the 3-D (volumetric or temporal)
 * variant: "可变形注意力…" §5.3, sampling points on voxel or video features,
 * offsets with a z (time) component, trilinear in place of bilinear
 * interpolation, the rest as msda_forward / msda_backward.
 *
 *   spatial_shapes      in   host [L][3] = (D_l, H_l, W_l); Len_in = sum D*H*W,
 *                            a level flattened z-major: row start + (z*H + y)*W + x
 *   sampling_locations  in   [N][Len_q][M][L][K][3] f32, (x, y, z) normalised
 *   attention_weights   in   [N][Len_q][M][L][K] f32 (as given)
 *   output              out  [N][Len_q][M*D], dtype
 *   grad_sampling_locations out [N][Len_q][M][L][K][3] f32
 *   the rest            as msda_forward / msda_backward (same workspace size)
 * pz = z * D_l - 0.5 (z * (D_l - 1) with MSDA_OPT_ALIGN_CORNERS), and likewise
 * x, y; each of the eight neighbours outside the volume contributes zero.
 * Locations and weights need 4-byte alignment; value, output, grad_output and
 * grad_value 16 bytes.  Len_in must stay below 2^28 and Len_in * M * D below 2^31.
 */
MSDA_API msda_status msda3d_forward(const msda_problem *problem, const void *value,
                                    const int64_t *spatial_shapes, const int64_t *level_start_index,
                                    const float *sampling_locations, const float *attention_weights,
                                    void *output, void *stream);

MSDA_API msda_status msda3d_backward(const msda_problem *problem, const void *value,
                                     const int64_t *spatial_shapes, const int64_t *level_start_index,
                                     const float *sampling_locations, const float *attention_weights,
                                     const void *grad_output, float *grad_value, float *grad_sampling_locations,
                                     float *grad_attention_weights, unsigned flags, void *workspace,
                                     size_t workspace_bytes, void *stream);

/* Name of a status code (static string). */
MSDA_API const char *msda_status_string(msda_status status);

/* Description of the last failure on the calling thread ("" if none). */
MSDA_API const char *msda_last_error(void);

/* Library version, major*10000 + minor*100 + patch. */
MSDA_API int msda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MSDA_H_ */
