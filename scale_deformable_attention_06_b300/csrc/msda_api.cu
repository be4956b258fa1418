// msda_api.cu -- the C ABI of libmsda (declared in include/msda.h): host-side
// argument checks, the per-level table, and dispatch to the kernel launchers.
// Nothing here allocates device memory.
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "../../include/msda.h"
#ifdef MSDA_DEBUG
#include "../../include/msda_debug.h"
#endif
#include "msda_launch.h"

namespace {

thread_local char g_last_error[512] = "";

msda_status fail(msda_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return s;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Head groups: n_groups groups of n_heads / n_groups consecutive heads share
// one set of locations and weights (0: one set per head).  A group's heads are
// contiguous in value and in the output, so the kernels see G "heads" of
// D = (n_heads / G) * head_dim channels; D must be a power of two from 8 to
// max_width.
msda_status group_width(const msda_problem *p, int max_width, int &G, int &D) {
    if (p->head_dim < 1) return fail(MSDA_ERR_INVALID_ARG, "head_dim %d below 1", p->head_dim);
    G = p->n_groups ? p->n_groups : p->n_heads;
    if (G < 1 || G > p->n_heads || p->n_heads % G)
        return fail(MSDA_ERR_INVALID_ARG, "n_groups %d does not divide n_heads %d", p->n_groups, p->n_heads);
    const int64_t width = (int64_t)(p->n_heads / G) * p->head_dim;
    if (width < 8 || width > max_width || (width & (width - 1)))
        return fail(MSDA_ERR_UNSUPPORTED, "channels a group samples with one set, (n_heads / n_groups) * head_dim "
                    "= %lld, not a power of two from 8 to %d", (long long)width, max_width);
    D = (int)width;
    return MSDA_OK;
}

// Checks the sizes and the levels and fills the launch geometry.
msda_status make_geometry(const msda_problem *p, const int64_t *shapes, const int64_t *starts,
                          msda::LaunchGeometry &g) {
    if (!p) return fail(MSDA_ERR_INVALID_ARG, "problem is NULL");
    if (p->N < 0 || p->Len_q < 0 || p->Len_in < 0)
        return fail(MSDA_ERR_INVALID_ARG, "negative size (N=%d Len_q=%d Len_in=%d)", p->N, p->Len_q, p->Len_in);
    if (p->n_heads < 1 || p->n_points < 1 || p->n_levels < 1)
        return fail(MSDA_ERR_INVALID_ARG, "n_heads, n_levels and n_points must be >= 1");
    if (p->options & ~(MSDA_OPT_PER_LEVEL_SOFTMAX | MSDA_OPT_ALIGN_CORNERS))
        return fail(MSDA_ERR_INVALID_ARG, "unknown option bits 0x%x", p->options);
    if (p->dtype != MSDA_F32 && p->dtype != MSDA_BF16)
        return fail(MSDA_ERR_UNSUPPORTED, "dtype %d is not MSDA_F32 or MSDA_BF16", p->dtype);
    int G = 0, D = 0;
    msda_status st = group_width(p, 256, G, D);
    if (st != MSDA_OK) return st;
    if (p->n_levels > msda::kMaxLevels)
        return fail(MSDA_ERR_UNSUPPORTED, "n_levels %d above %d", p->n_levels, msda::kMaxLevels);
    if ((int64_t)p->n_levels * p->n_points > msda::kMaxSamples)
        return fail(MSDA_ERR_UNSUPPORTED, "n_levels * n_points = %lld above %d",
                    (long long)p->n_levels * p->n_points, msda::kMaxSamples);
    if (!shapes || !starts) return fail(MSDA_ERR_INVALID_ARG, "spatial_shapes / level_start_index is NULL");
    int64_t expect = 0, maxW = 0;
    for (int l = 0; l < p->n_levels; ++l) {
        const int64_t H = shapes[2 * l], W = shapes[2 * l + 1];
        if (H < 1 || W < 1) return fail(MSDA_ERR_INVALID_ARG, "level %d has shape (%lld, %lld)", l, (long long)H, (long long)W);
        if (H > (1 << 24) || W > (1 << 24))
            return fail(MSDA_ERR_UNSUPPORTED, "level %d side above 2^24 (float pixel coordinates)", l);
        if (starts[l] != expect)
            return fail(MSDA_ERR_INVALID_ARG, "level_start_index[%d] = %lld, expected %lld", l, (long long)starts[l],
                        (long long)expect);
        expect += H * W;
        if (W > maxW) maxW = W;
    }
    if (expect != p->Len_in)
        return fail(MSDA_ERR_INVALID_ARG, "sum of H*W over levels is %lld but Len_in is %d", (long long)expect, p->Len_in);
    if (p->Len_in >= (int64_t(1) << 28))
        return fail(MSDA_ERR_UNSUPPORTED, "Len_in %d is not below 2^28 (pixel index of a corner record)", p->Len_in);
    const int64_t pix = (int64_t)p->n_heads * p->head_dim;
    if ((p->Len_in + 2 * maxW + 4) * pix >= (int64_t(1) << 31))
        return fail(MSDA_ERR_UNSUPPORTED, "(Len_in + 2 W + 4) * n_heads * head_dim exceeds 2^31");
    const int64_t rows = (int64_t)p->N * p->Len_q * G;
    if (rows >= (int64_t(1) << 31)) return fail(MSDA_ERR_UNSUPPORTED, "N * Len_q * n_groups exceeds 2^31");

    std::memset(&g, 0, sizeof(g));
    g.D = D;
    g.d.N = p->N;
    g.d.Len_in = p->Len_in;
    g.d.M = G;
    g.d.Len_q = p->Len_q;
    g.d.L = p->n_levels;
    g.d.K = p->n_points;
    g.d.P = p->n_levels * p->n_points;
    g.d.rows = (int)rows;
    g.d.qm = p->Len_q * G;
    g.d.pix = (int)pix;
    const bool align = (p->options & MSDA_OPT_ALIGN_CORNERS) != 0;
    g.d.per_level_softmax = (p->options & MSDA_OPT_PER_LEVEL_SOFTMAX) != 0;
    g.lv.shift = align ? 0.f : 0.5f;
    for (int l = 0; l < p->n_levels; ++l) {
        g.lv.H[l] = (int)shapes[2 * l];
        g.lv.W[l] = (int)shapes[2 * l + 1];
        g.lv.start[l] = (int)starts[l];
        g.lv.Hf[l] = (float)shapes[2 * l];
        g.lv.Wf[l] = (float)shapes[2 * l + 1];
        // pixel scale, and the fp32 factor from offset pixels to the pixel
        // coordinate: S / size, 1 without align_corners
        g.lv.Sx[l] = align ? (float)(shapes[2 * l + 1] - 1) : g.lv.Wf[l];
        g.lv.Sy[l] = align ? (float)(shapes[2 * l] - 1) : g.lv.Hf[l];
        g.lv.Rx[l] = align ? g.lv.Sx[l] / g.lv.Wf[l] : 1.f;
        g.lv.Ry[l] = align ? g.lv.Sy[l] / g.lv.Hf[l] : 1.f;
    }
    for (int s = 0; s < g.d.P; ++s) g.level_of[s] = (unsigned char)(s / p->n_points);
    return MSDA_OK;
}

// The 3-D variant: spatial_shapes is [L][3] = (D, H, W).  Same checks, with
// volumes in place of maps; the per-level softmax bit has no 3-D call to act on.
msda_status make_geometry3(const msda_problem *p, const int64_t *shapes, const int64_t *starts,
                           msda::LaunchGeometry3 &g3) {
    if (!p) return fail(MSDA_ERR_INVALID_ARG, "problem is NULL");
    if (p->N < 0 || p->Len_q < 0 || p->Len_in < 0)
        return fail(MSDA_ERR_INVALID_ARG, "negative size (N=%d Len_q=%d Len_in=%d)", p->N, p->Len_q, p->Len_in);
    if (p->n_heads < 1 || p->n_points < 1 || p->n_levels < 1)
        return fail(MSDA_ERR_INVALID_ARG, "n_heads, n_levels and n_points must be >= 1");
    if (p->options & ~(MSDA_OPT_PER_LEVEL_SOFTMAX | MSDA_OPT_ALIGN_CORNERS))
        return fail(MSDA_ERR_INVALID_ARG, "unknown option bits 0x%x", p->options);
    if (p->dtype != MSDA_F32 && p->dtype != MSDA_BF16)
        return fail(MSDA_ERR_UNSUPPORTED, "dtype %d is not MSDA_F32 or MSDA_BF16", p->dtype);
    int G = 0, D = 0;
    msda_status st = group_width(p, 64, G, D);
    if (st != MSDA_OK) return st;
    if (p->n_levels > msda::kMaxLevels)
        return fail(MSDA_ERR_UNSUPPORTED, "n_levels %d above %d", p->n_levels, msda::kMaxLevels);
    if ((int64_t)p->n_levels * p->n_points > msda::kMaxSamples)
        return fail(MSDA_ERR_UNSUPPORTED, "n_levels * n_points = %lld above %d",
                    (long long)p->n_levels * p->n_points, msda::kMaxSamples);
    if (!shapes || !starts) return fail(MSDA_ERR_INVALID_ARG, "spatial_shapes / level_start_index is NULL");
    int64_t expect = 0;
    for (int l = 0; l < p->n_levels; ++l) {
        const int64_t Dz = shapes[3 * l], H = shapes[3 * l + 1], W = shapes[3 * l + 2];
        if (Dz < 1 || H < 1 || W < 1)
            return fail(MSDA_ERR_INVALID_ARG, "level %d has shape (%lld, %lld, %lld)", l, (long long)Dz,
                        (long long)H, (long long)W);
        if (Dz > (1 << 24) || H > (1 << 24) || W > (1 << 24))
            return fail(MSDA_ERR_UNSUPPORTED, "level %d side above 2^24 (float pixel coordinates)", l);
        if (starts[l] != expect)
            return fail(MSDA_ERR_INVALID_ARG, "level_start_index[%d] = %lld, expected %lld", l, (long long)starts[l],
                        (long long)expect);
        expect += Dz * H * W;
        if (expect >= (int64_t(1) << 28)) break;
    }
    if (expect != p->Len_in)
        return fail(MSDA_ERR_INVALID_ARG, "sum of D*H*W over levels is %lld but Len_in is %d", (long long)expect,
                    p->Len_in);
    if (p->Len_in >= (int64_t(1) << 28))
        return fail(MSDA_ERR_UNSUPPORTED, "Len_in %d is not below 2^28 (voxel index of a corner record)", p->Len_in);
    const int64_t pix = (int64_t)p->n_heads * p->head_dim;
    if ((int64_t)p->Len_in * pix >= (int64_t(1) << 31))
        return fail(MSDA_ERR_UNSUPPORTED, "Len_in * n_heads * head_dim exceeds 2^31");
    const int64_t rows = (int64_t)p->N * p->Len_q * G;
    if (rows >= (int64_t(1) << 31)) return fail(MSDA_ERR_UNSUPPORTED, "N * Len_q * n_groups exceeds 2^31");

    std::memset(&g3, 0, sizeof(g3));
    g3.g.D = D;
    msda::Dims &d = g3.g.d;
    d.N = p->N;
    d.Len_in = p->Len_in;
    d.M = G;
    d.Len_q = p->Len_q;
    d.L = p->n_levels;
    d.K = p->n_points;
    d.P = p->n_levels * p->n_points;
    d.rows = (int)rows;
    d.qm = p->Len_q * G;
    d.pix = (int)pix;
    const bool align = (p->options & MSDA_OPT_ALIGN_CORNERS) != 0;
    g3.lv.shift = align ? 0.f : 0.5f;
    for (int l = 0; l < p->n_levels; ++l) {
        g3.lv.Dz[l] = (int)shapes[3 * l];
        g3.lv.H[l] = (int)shapes[3 * l + 1];
        g3.lv.W[l] = (int)shapes[3 * l + 2];
        g3.lv.start[l] = (int)starts[l];
        g3.lv.Dzf[l] = (float)g3.lv.Dz[l];
        g3.lv.Hf[l] = (float)g3.lv.H[l];
        g3.lv.Wf[l] = (float)g3.lv.W[l];
        g3.lv.Sx[l] = align ? (float)(g3.lv.W[l] - 1) : g3.lv.Wf[l];
        g3.lv.Sy[l] = align ? (float)(g3.lv.H[l] - 1) : g3.lv.Hf[l];
        g3.lv.Sz[l] = align ? (float)(g3.lv.Dz[l] - 1) : g3.lv.Dzf[l];
    }
    for (int s = 0; s < d.P; ++s) g3.g.level_of[s] = (unsigned char)(s / p->n_points);
    return MSDA_OK;
}

msda_status cuda_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return MSDA_OK;
    return fail(MSDA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace

// Helpers of msda_backward_noalloc (msda_noalloc.cu): the same host checks as
// msda_backward, reached from the other translation unit.
namespace msda {

msda_status noalloc_fail(msda_status s, const char *msg) { return fail(s, "%s", msg); }

msda_status noalloc_check_and_geometry(const msda_problem *problem, const int64_t *spatial_shapes,
                                       const int64_t *level_start_index, LaunchGeometry &g) {
    g_last_error[0] = 0;
    return make_geometry(problem, spatial_shapes, level_start_index, g);
}

msda_status noalloc_check_pointers(const msda_problem *problem, const LaunchGeometry &g, const void *value,
                                   const float *loc, const float *attn, const void *grad_out, const float *grad_value,
                                   const float *grad_loc, const float *grad_attn) {
    const size_t nval = (size_t)g.d.N * g.d.Len_in * g.d.M * g.D;
    if (nval > 0 && !grad_value) return fail(MSDA_ERR_INVALID_ARG, "grad_value is NULL");
    if (grad_value && !aligned(grad_value, 16)) return fail(MSDA_ERR_INVALID_ARG, "grad_value not 16-byte aligned");
    if (g.d.rows > 0) {
        if (!value || !loc || !attn || !grad_out || !grad_loc || !grad_attn)
            return fail(MSDA_ERR_INVALID_ARG, "a tensor pointer is NULL");
        if (!aligned(value, 16) || !aligned(grad_out, 16) || !aligned(loc, 8) || !aligned(grad_loc, 8) ||
            !aligned(attn, 4) || !aligned(grad_attn, 4))
            return fail(MSDA_ERR_INVALID_ARG, "misaligned tensor");
    }
    return MSDA_OK;
}

}  // namespace msda

extern "C" {

msda_status msda_forward(const msda_problem *problem, const void *value, const int64_t *spatial_shapes,
                         const int64_t *level_start_index, const float *sampling_locations,
                         const float *attention_weights, void *output, void *stream) {
    g_last_error[0] = 0;
    msda::LaunchGeometry g;
    msda_status st = make_geometry(problem, spatial_shapes, level_start_index, g);
    if (st != MSDA_OK) return st;
    if (g.d.rows == 0) return MSDA_OK;
    if (!value || !sampling_locations || !attention_weights || !output)
        return fail(MSDA_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if (!aligned(value, 16) || !aligned(output, 16) || !aligned(sampling_locations, 8) || !aligned(attention_weights, 4))
        return fail(MSDA_ERR_INVALID_ARG, "misaligned tensor (value/output 16 B, locations 8 B, weights 4 B)");
    return cuda_status(msda::launch_forward(g, problem->dtype, g.D, value, sampling_locations,
                                            attention_weights, output, static_cast<cudaStream_t>(stream)),
                       "msda_forward launch");
}

msda_status msda_forward_fused(const msda_problem *problem, const void *value, const int64_t *spatial_shapes,
                               const int64_t *level_start_index, const float *reference_points,
                               const float *sampling_offsets, const float *attention_logits, void *output,
                               void *stream) {
    g_last_error[0] = 0;
    msda::LaunchGeometry g;
    msda_status st = make_geometry(problem, spatial_shapes, level_start_index, g);
    if (st != MSDA_OK) return st;
    if (g.d.rows == 0) return MSDA_OK;
    if (!value || !reference_points || !sampling_offsets || !attention_logits || !output)
        return fail(MSDA_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if (!aligned(value, 16) || !aligned(output, 16) || !aligned(reference_points, 8) || !aligned(sampling_offsets, 8) ||
        !aligned(attention_logits, 4))
        return fail(MSDA_ERR_INVALID_ARG, "misaligned tensor (value/output 16 B, points/offsets 8 B, logits 4 B)");
    return cuda_status(msda::launch_forward_fused(g, problem->dtype, g.D, value, reference_points,
                                                  sampling_offsets, attention_logits, output,
                                                  static_cast<cudaStream_t>(stream)),
                       "msda_forward_fused launch");
}

size_t msda_backward_workspace_size(const msda_problem *problem, unsigned flags) {
    if (!problem || problem->N < 0 || problem->Len_in < 0 || problem->n_heads < 1 || problem->head_dim < 1) return 0;
    msda::LaunchGeometry g;
    std::memset(&g, 0, sizeof(g));
    g.d.N = problem->N;
    g.d.Len_in = problem->Len_in;
    g.d.M = problem->n_heads;         // n_heads * head_dim channels a pixel, grouped or not
    return msda::backward_workspace_bytes(g, problem->head_dim, (flags & MSDA_DETERMINISTIC) != 0);
}

msda_status msda_backward(const msda_problem *problem, const void *value, const int64_t *spatial_shapes,
                          const int64_t *level_start_index, const float *sampling_locations,
                          const float *attention_weights, const void *grad_output, float *grad_value,
                          float *grad_sampling_locations, float *grad_attention_weights, unsigned flags,
                          void *workspace, size_t workspace_bytes, void *stream) {
    g_last_error[0] = 0;
    msda::LaunchGeometry g;
    msda_status st = make_geometry(problem, spatial_shapes, level_start_index, g);
    if (st != MSDA_OK) return st;
    if (flags & ~(MSDA_DETERMINISTIC | MSDA_ACCUMULATE_GRAD_VALUE))
        return fail(MSDA_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
    const bool det = (flags & MSDA_DETERMINISTIC) != 0, acc = (flags & MSDA_ACCUMULATE_GRAD_VALUE) != 0;
    const size_t nval = (size_t)g.d.N * g.d.Len_in * g.d.M * g.D;
    if (nval > 0 && !grad_value) return fail(MSDA_ERR_INVALID_ARG, "grad_value is NULL");
    if (grad_value && !aligned(grad_value, 16)) return fail(MSDA_ERR_INVALID_ARG, "grad_value not 16-byte aligned");
    if (g.d.rows > 0) {
        if (!value || !sampling_locations || !attention_weights || !grad_output || !grad_sampling_locations ||
            !grad_attention_weights)
            return fail(MSDA_ERR_INVALID_ARG, "a tensor pointer is NULL");
        if (!aligned(value, 16) || !aligned(grad_output, 16) || !aligned(sampling_locations, 8) ||
            !aligned(grad_sampling_locations, 8) || !aligned(attention_weights, 4) || !aligned(grad_attention_weights, 4))
            return fail(MSDA_ERR_INVALID_ARG, "misaligned tensor");
    }
    const size_t need = msda::backward_workspace_bytes(g, g.D, det);
    if (need > 0) {
        if (!workspace || workspace_bytes < need)
            return fail(MSDA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace ? workspace_bytes : 0);
        if (!aligned(workspace, 256)) return fail(MSDA_ERR_WORKSPACE, "workspace not 256-byte aligned");
    }
    if (nval == 0 && g.d.rows == 0) return MSDA_OK;
    if (g.d.rows == 0 && acc) return MSDA_OK;
    return cuda_status(msda::launch_backward(g, problem->dtype, g.D, value, sampling_locations,
                                             attention_weights, grad_output, grad_value, grad_sampling_locations,
                                             grad_attention_weights, det, acc, workspace,
                                             static_cast<cudaStream_t>(stream)),
                       "msda_backward launch");
}

msda_status msda_backward_fused(const msda_problem *problem, const void *value, const int64_t *spatial_shapes,
                                const int64_t *level_start_index, const float *reference_points,
                                const float *sampling_offsets, const float *attention_logits, const void *grad_output,
                                float *grad_value, float *grad_reference_points, float *grad_sampling_offsets,
                                float *grad_attention_logits, unsigned flags, void *workspace, size_t workspace_bytes,
                                void *stream) {
    g_last_error[0] = 0;
    msda::LaunchGeometry g;
    msda_status st = make_geometry(problem, spatial_shapes, level_start_index, g);
    if (st != MSDA_OK) return st;
    if (flags & ~(MSDA_DETERMINISTIC | MSDA_ACCUMULATE_GRAD_VALUE))
        return fail(MSDA_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
    const bool det = (flags & MSDA_DETERMINISTIC) != 0, acc = (flags & MSDA_ACCUMULATE_GRAD_VALUE) != 0;
    const size_t nval = (size_t)g.d.N * g.d.Len_in * g.d.M * g.D;
    if (nval > 0 && !grad_value) return fail(MSDA_ERR_INVALID_ARG, "grad_value is NULL");
    if (grad_value && !aligned(grad_value, 16)) return fail(MSDA_ERR_INVALID_ARG, "grad_value not 16-byte aligned");
    if (g.d.rows > 0) {
        if (!value || !reference_points || !sampling_offsets || !attention_logits || !grad_output ||
            !grad_reference_points || !grad_sampling_offsets || !grad_attention_logits)
            return fail(MSDA_ERR_INVALID_ARG, "a tensor pointer is NULL");
        if (!aligned(value, 16) || !aligned(grad_output, 16) || !aligned(reference_points, 8) ||
            !aligned(sampling_offsets, 8) || !aligned(grad_reference_points, 8) || !aligned(grad_sampling_offsets, 8) ||
            !aligned(attention_logits, 4) || !aligned(grad_attention_logits, 4))
            return fail(MSDA_ERR_INVALID_ARG, "misaligned tensor");
    }
    const size_t need = msda::backward_workspace_bytes(g, g.D, det);
    if (need > 0) {
        if (!workspace || workspace_bytes < need)
            return fail(MSDA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace ? workspace_bytes : 0);
        if (!aligned(workspace, 256)) return fail(MSDA_ERR_WORKSPACE, "workspace not 256-byte aligned");
    }
    if (nval == 0 && g.d.rows == 0) return MSDA_OK;
    if (g.d.rows == 0 && acc) return MSDA_OK;
    return cuda_status(msda::launch_backward_fused(g, problem->dtype, g.D, value, reference_points,
                                                   sampling_offsets, attention_logits, grad_output, grad_value,
                                                   grad_reference_points, grad_sampling_offsets, grad_attention_logits,
                                                   det, acc, workspace, static_cast<cudaStream_t>(stream)),
                       "msda_backward_fused launch");
}

msda_status msda3d_forward(const msda_problem *problem, const void *value, const int64_t *spatial_shapes,
                           const int64_t *level_start_index, const float *sampling_locations,
                           const float *attention_weights, void *output, void *stream) {
    g_last_error[0] = 0;
    msda::LaunchGeometry3 g;
    msda_status st = make_geometry3(problem, spatial_shapes, level_start_index, g);
    if (st != MSDA_OK) return st;
    if (g.g.d.rows == 0) return MSDA_OK;
    if (!value || !sampling_locations || !attention_weights || !output)
        return fail(MSDA_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if (!aligned(value, 16) || !aligned(output, 16) || !aligned(sampling_locations, 4) || !aligned(attention_weights, 4))
        return fail(MSDA_ERR_INVALID_ARG, "misaligned tensor (value/output 16 B, locations and weights 4 B)");
    return cuda_status(msda::launch_forward3d(g, problem->dtype, g.g.D, value, sampling_locations,
                                              attention_weights, output, static_cast<cudaStream_t>(stream)),
                       "msda3d_forward launch");
}

msda_status msda3d_backward(const msda_problem *problem, const void *value, const int64_t *spatial_shapes,
                            const int64_t *level_start_index, const float *sampling_locations,
                            const float *attention_weights, const void *grad_output, float *grad_value,
                            float *grad_sampling_locations, float *grad_attention_weights, unsigned flags,
                            void *workspace, size_t workspace_bytes, void *stream) {
    g_last_error[0] = 0;
    msda::LaunchGeometry3 g;
    msda_status st = make_geometry3(problem, spatial_shapes, level_start_index, g);
    if (st != MSDA_OK) return st;
    if (flags & ~(MSDA_DETERMINISTIC | MSDA_ACCUMULATE_GRAD_VALUE))
        return fail(MSDA_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
    const bool det = (flags & MSDA_DETERMINISTIC) != 0, acc = (flags & MSDA_ACCUMULATE_GRAD_VALUE) != 0;
    const size_t nval = (size_t)g.g.d.N * g.g.d.Len_in * g.g.d.M * g.g.D;
    if (nval > 0 && !grad_value) return fail(MSDA_ERR_INVALID_ARG, "grad_value is NULL");
    if (grad_value && !aligned(grad_value, 16)) return fail(MSDA_ERR_INVALID_ARG, "grad_value not 16-byte aligned");
    if (g.g.d.rows > 0) {
        if (!value || !sampling_locations || !attention_weights || !grad_output || !grad_sampling_locations ||
            !grad_attention_weights)
            return fail(MSDA_ERR_INVALID_ARG, "a tensor pointer is NULL");
        if (!aligned(value, 16) || !aligned(grad_output, 16) || !aligned(sampling_locations, 4) ||
            !aligned(grad_sampling_locations, 4) || !aligned(attention_weights, 4) || !aligned(grad_attention_weights, 4))
            return fail(MSDA_ERR_INVALID_ARG, "misaligned tensor");
    }
    const size_t need = msda::backward_workspace_bytes(g.g, g.g.D, det);
    if (need > 0) {
        if (!workspace || workspace_bytes < need)
            return fail(MSDA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace ? workspace_bytes : 0);
        if (!aligned(workspace, 256)) return fail(MSDA_ERR_WORKSPACE, "workspace not 256-byte aligned");
    }
    if (nval == 0 && g.g.d.rows == 0) return MSDA_OK;
    if (g.g.d.rows == 0 && acc) return MSDA_OK;
    return cuda_status(msda::launch_backward3d(g, problem->dtype, g.g.D, value, sampling_locations,
                                               attention_weights, grad_output, grad_value, grad_sampling_locations,
                                               grad_attention_weights, det, acc, workspace,
                                               static_cast<cudaStream_t>(stream)),
                       "msda3d_backward launch");
}

const char *msda_status_string(msda_status s) {
    switch (s) {
        case MSDA_OK: return "MSDA_OK";
        case MSDA_ERR_INVALID_ARG: return "MSDA_ERR_INVALID_ARG";
        case MSDA_ERR_UNSUPPORTED: return "MSDA_ERR_UNSUPPORTED";
        case MSDA_ERR_CUDA: return "MSDA_ERR_CUDA";
        case MSDA_ERR_WORKSPACE: return "MSDA_ERR_WORKSPACE";
    }
    return "MSDA_ERR_UNKNOWN";
}

const char *msda_last_error(void) { return g_last_error; }

int msda_version(void) { return 100; }

}  // extern "C"

#ifdef MSDA_DEBUG
extern "C" unsigned long long msda_debug_violations(int reset) {
    cudaDeviceSynchronize();
    return msda::debug_count_forward(reset != 0) + msda::debug_count_backward(reset != 0) +
           msda::debug_count_3d(reset != 0);
}
#endif
