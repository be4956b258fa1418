/*
 * msda_oracle.c -- plain, slow, single-threaded fp64 CPU oracle for the
 * multi-scale deformable attention (MSDeformAttn) core.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this file: only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or constant
 * with the CUDA library; it is written straight from the pages' definition.
 *
 * Citation key (the pages this follows):
 *   [MSDA-tut]  "可变形注意力：多尺度稀疏采样与视觉检测实战解析" (bjdmk.com.cn)
 *               -- §2.2 multi-scale formula, §2.3 bilinear interpolation,
 *                  §3.1 interface, §3.2 the grid_sample module.
 *   [DDETR-tut] "可变形 DETR：加速收敛的稀疏注意力检测器" (freeguideonline.com)
 *               -- §3.2 single-scale formula, §3.3 multi-scale formula,
 *                  §6 forward pseudocode (location = reference + offset / scale).
 *   [DDETR-dep] "Deformable DETR的本质定位与设计动机" deployment notes
 *               (un.csdn.net/8fh7s5u7wxgo) -- §2.2 worked example.
 *
 * Layouts (all row-major, contiguous):
 *   value              [N][Len_in][n_heads][head_dim]         ([MSDA-tut] §3.2, value.view)
 *   spatial_shapes     [n_levels][2] = (H_l, W_l)              ([MSDA-tut] §3.1)
 *   level_start_index  [n_levels]                              ([MSDA-tut] §3.1)
 *   sampling_locations [N][Len_q][n_heads][n_levels][n_points][2], (x, y) in [0,1]
 *   attention_weights  [N][Len_q][n_heads][n_levels][n_points]
 *   output             [N][Len_q][n_heads*head_dim]  (head m owns channels m*D..m*D+D-1)
 *   reference_points   [N][Len_q][n_levels][2]
 *   sampling_offsets   [N][Len_q][n_heads][n_levels][n_points][2], in pixels of level l
 *   attention_logits   [N][Len_q][n_heads][n_levels*n_points]
 * Grouped entry points (*_grouped): the n_heads heads form n_groups groups of
 * n_heads / n_groups consecutive heads that share one set of locations and
 * weights, and every per-sample tensor has n_groups in place of n_heads
 * (sampling_locations [N][Len_q][n_groups][n_levels][n_points][2], ...); head m
 * samples with the set of group m / (n_heads / n_groups).  n_groups = n_heads is
 * the plain call.  (The DAT pages' sampler: one offset field per group of
 * channels, "可变形注意力…" is silent on it.)
 *
 * Readings taken where the pages are silent or disagree:
 *   - normalised -> pixel: px = loc_x * W_l - 0.5, py = loc_y * H_l - 0.5
 *     (grid_sample with align_corners=False, [MSDA-tut] §2.3 and §3.2).
 *   - zero padding per corner: a corner outside [0,W)x[0,H) contributes 0, the
 *     other corners keep their weights ([MSDA-tut] §2.3, padding_mode='zeros').
 *   - the softmax runs over all n_levels*n_points logits of one (query, head)
 *     ([MSDA-tut] §3.2 code: view(..., n_levels*n_points), softmax(dim=-1)).
 *   - fused offsets are in pixels of their level: loc = ref + off / (W_l, H_l)
 *     ([DDETR-tut] §6: reference_points + sampling_offsets / scale_factors).
 *   - the lower-left corner is x0 = floor(px), y0 = floor(py), taken on the
 *     fp64 pixel coordinate like every other step; at an exact integer px the
 *     corner x0 + 1 gets weight 0 and the location gradient is the one-sided
 *     derivative of the cell floor() selects.  Bilinear interpolation is
 *     continuous across cell edges, so a sample within rounding of an edge
 *     has the same output whichever cell is taken; only its location gradient
 *     jumps, and a comparison against this oracle has to allow either side
 *     there.
 *
 * Options (the last argument of the forward and backward entry points; bits):
 *   1  per-level softmax: the fused calls normalise the n_points logits of each
 *      level separately.  [MSDA-tut] §2.2 prose says the normalisation runs over
 *      k, per level; its §3.2 code normalises over all n_levels*n_points.  Both
 *      readings are offered; 0 is the code's.
 *   2  align_corners: px = loc_x * (W_l - 1), py = loc_y * (H_l - 1), the pixel
 *      centres sit at i / (W_l - 1) (grid_sample with align_corners=True, the
 *      convention of the DAT pages' sampler); the fused location is still
 *      loc = ref + off / (W_l, H_l).
 *
 * Return value of every entry point: 0 on success, -1 on a bad argument.
 */
#define OPT_PER_LEVEL_SOFTMAX 1
#define OPT_ALIGN_CORNERS 2
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Step a1: sampling location = reference point + offset / (W_l, H_l).        */
/* [DDETR-tut] §6; [MSDA-tut] §3.2 (the scale and unscale pair).              */
/* ------------------------------------------------------------------------- */
int msda_oracle_locations(int64_t N, int64_t Len_q, int64_t n_heads, int64_t n_levels,
                          int64_t n_points, const int64_t *spatial_shapes,
                          const double *reference_points, const double *sampling_offsets,
                          double *sampling_locations)
{
    if (N < 0 || Len_q < 0 || n_heads < 0 || n_levels < 0 || n_points < 0) return -1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t q = 0; q < Len_q; ++q)
            for (int64_t m = 0; m < n_heads; ++m)
                for (int64_t l = 0; l < n_levels; ++l) {
                    double H = (double)spatial_shapes[2 * l + 0];
                    double W = (double)spatial_shapes[2 * l + 1];
                    const double *ref = reference_points + ((n * Len_q + q) * n_levels + l) * 2;
                    for (int64_t k = 0; k < n_points; ++k) {
                        int64_t i = ((((n * Len_q + q) * n_heads + m) * n_levels + l) * n_points + k) * 2;
                        sampling_locations[i + 0] = ref[0] + sampling_offsets[i + 0] / W;
                        sampling_locations[i + 1] = ref[1] + sampling_offsets[i + 1] / H;
                    }
                }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Step a2: A = softmax over the n_levels*n_points logits of one (q, head),   */
/* max-subtracted.  [MSDA-tut] §3.2: softmax(dim=-1) over levels*points.      */
/* ------------------------------------------------------------------------- */
int msda_oracle_softmax(int64_t rows, int64_t cols, const double *logits, double *weights)
{
    if (rows < 0 || cols <= 0) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const double *x = logits + r * cols;
        double *y = weights + r * cols;
        double mx = x[0];
        for (int64_t j = 1; j < cols; ++j)
            if (x[j] > mx) mx = x[j];
        double sum = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            y[j] = exp(x[j] - mx);
            sum += y[j];
        }
        for (int64_t j = 0; j < cols; ++j) y[j] /= sum;
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Shared by forward and backward of both paths: one bilinear sample.         */
/* [MSDA-tut] §2.3: the four integer neighbours of (x, y), weights            */
/* (1-|dx|)(1-|dy|), a neighbour outside the map reads as zero.               */
/* ------------------------------------------------------------------------- */
typedef struct {
    int64_t x0, y0;     /* lower corner (column, row) in pixels of the level */
    double fx, fy;      /* px - x0, py - y0 */
    int64_t row[4];     /* value row (index into Len_in) of corner c, -1 if outside */
    double w[4];        /* bilinear weight of corner c (0 is kept for outside corners) */
} corners_t;
/* corner order c = 0:(x0,y0) 1:(x0+1,y0) 2:(x0,y0+1) 3:(x0+1,y0+1) */

static void make_corners(int64_t x0, int64_t y0, double fx, double fy, int64_t H, int64_t W,
                         int64_t start, corners_t *c)
{
    c->x0 = x0; c->y0 = y0; c->fx = fx; c->fy = fy;
    for (int j = 0; j < 2; ++j)
        for (int i = 0; i < 2; ++i) {
            int ci = 2 * j + i;
            int64_t xc = x0 + i, yc = y0 + j;
            c->w[ci] = (i ? fx : 1.0 - fx) * (j ? fy : 1.0 - fy);
            c->row[ci] = (xc >= 0 && xc < W && yc >= 0 && yc < H) ? start + yc * W + xc : -1;
        }
}

/* Lower corner index floor(p) of a pixel coordinate p on an axis of `size`
 * pixels.  An index below -2 or above size + 1 is clamped there before the
 * conversion to an integer: both neighbours of such a sample lie outside the
 * map either way, so the clamp changes no result. */
static int64_t lower_corner(double p, int64_t size)
{
    double f = floor(p);
    if (f < -2.0) f = -2.0;
    if (f > (double)size + 1.0) f = (double)size + 1.0;
    return (int64_t)f;
}

/* Step a3 from the pixel coordinate (px, py): the cell and the fractions. */
static void cell_of(double px, double py, int64_t H, int64_t W, int64_t start, corners_t *c)
{
    int64_t x0 = lower_corner(px, W);
    int64_t y0 = lower_corner(py, H);
    make_corners(x0, y0, px - (double)x0, py - (double)y0, H, W, start, c);
}

static void corners_unfused(double lx, double ly, int64_t H, int64_t W, int64_t start, int align,
                            corners_t *c)
{
    double px = align ? lx * (double)(W - 1) : lx * (double)W - 0.5;   /* step a3 */
    double py = align ? ly * (double)(H - 1) : ly * (double)H - 0.5;
    cell_of(px, py, H, W, start, c);
}

static void corners_fused(double rx, double ry, double ox, double oy, int64_t H, int64_t W,
                          int64_t start, int align, corners_t *c)
{
    double lx = rx + ox / (double)W;    /* step a1 */
    double ly = ry + oy / (double)H;
    double px = align ? lx * (double)(W - 1) : lx * (double)W - 0.5;   /* step a3 */
    double py = align ? ly * (double)(H - 1) : ly * (double)H - 0.5;
    cell_of(px, py, H, W, start, c);
}

static int check_levels(int64_t Len_in, int64_t n_levels, const int64_t *shapes, const int64_t *starts)
{
    int64_t expect = 0;
    for (int64_t l = 0; l < n_levels; ++l) {
        if (shapes[2 * l] <= 0 || shapes[2 * l + 1] <= 0) return -1;
        if (starts[l] != expect) return -1;
        expect += shapes[2 * l] * shapes[2 * l + 1];
    }
    return expect == Len_in ? 0 : -1;
}

/* sample[d] = sum over in-map corners of w_c * value[n][row_c][m][d] */
static void gather_sample(const double *value, int64_t Len_in, int64_t n_heads, int64_t D,
                          int64_t n, int64_t m, const corners_t *c, double *sample)
{
    for (int64_t d = 0; d < D; ++d) sample[d] = 0.0;
    for (int ci = 0; ci < 4; ++ci) {
        if (c->row[ci] < 0) continue;
        const double *v = value + ((n * Len_in + c->row[ci]) * n_heads + m) * D;
        for (int64_t d = 0; d < D; ++d) sample[d] += c->w[ci] * v[d];
    }
}

/* ------------------------------------------------------------------------- */
/* Steps a3-a5: out[n][q][m*D+d] = sum_{l,k} A[n,q,m,l,k] * sample_{l,k}[d]  */
/* [MSDA-tut] §2.2 (inner sum of the MSDeformAttn formula), §3.2 steps 4-5;   */
/* [DDETR-tut] §3.3.  `fused` selects how the corner is located.              */
/* ------------------------------------------------------------------------- */
static int forward_impl(int fused, int64_t N, int64_t Len_in, int64_t n_heads, int64_t n_groups, int64_t D,
                        int64_t Len_q, int64_t n_levels, int64_t n_points,
                        const double *value, const int64_t *shapes, const int64_t *starts,
                        const double *loc_or_ref, const double *offsets, const double *attn,
                        double *out, int64_t options)
{
    int align = (options & OPT_ALIGN_CORNERS) != 0;
    if (N < 0 || Len_in < 0 || n_heads <= 0 || D <= 0 || Len_q < 0 || n_levels <= 0 || n_points <= 0)
        return -1;
    if (n_groups <= 0 || n_heads % n_groups) return -1;
    int64_t hpg = n_heads / n_groups;           /* heads per group */
    if (check_levels(Len_in, n_levels, shapes, starts)) return -1;
    double *sample = (double *)malloc(sizeof(double) * (size_t)D);
    if (!sample) return -1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t q = 0; q < Len_q; ++q)
            for (int64_t m = 0; m < n_heads; ++m) {
                double *o = out + ((n * Len_q + q) * n_heads + m) * D;
                int64_t gm = m / hpg;               /* the group whose locations head m samples */
                for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
                for (int64_t l = 0; l < n_levels; ++l) {
                    int64_t H = shapes[2 * l], W = shapes[2 * l + 1];
                    for (int64_t k = 0; k < n_points; ++k) {
                        int64_t s = (((n * Len_q + q) * n_groups + gm) * n_levels + l) * n_points + k;
                        corners_t c;
                        if (fused) {
                            const double *ref = loc_or_ref + ((n * Len_q + q) * n_levels + l) * 2;
                            corners_fused(ref[0], ref[1], offsets[2 * s], offsets[2 * s + 1], H, W,
                                          starts[l], align, &c);
                        } else {
                            corners_unfused(loc_or_ref[2 * s], loc_or_ref[2 * s + 1], H, W, starts[l], align, &c);
                        }
                        gather_sample(value, Len_in, n_heads, D, n, m, &c, sample);
                        for (int64_t d = 0; d < D; ++d) o[d] += attn[s] * sample[d];
                    }
                }
            }
    free(sample);
    return 0;
}

int msda_oracle_forward(int64_t N, int64_t Len_in, int64_t n_heads, int64_t D, int64_t Len_q,
                        int64_t n_levels, int64_t n_points, const double *value,
                        const int64_t *spatial_shapes, const int64_t *level_start_index,
                        const double *sampling_locations, const double *attention_weights,
                        double *output, int64_t options)
{
    return forward_impl(0, N, Len_in, n_heads, n_heads, D, Len_q, n_levels, n_points, value, spatial_shapes,
                        level_start_index, sampling_locations, NULL, attention_weights, output, options);
}

int msda_oracle_forward_grouped(int64_t N, int64_t Len_in, int64_t n_heads, int64_t n_groups, int64_t D,
                                int64_t Len_q, int64_t n_levels, int64_t n_points, const double *value,
                                const int64_t *spatial_shapes, const int64_t *level_start_index,
                                const double *sampling_locations, const double *attention_weights,
                                double *output, int64_t options)
{
    return forward_impl(0, N, Len_in, n_heads, n_groups, D, Len_q, n_levels, n_points, value, spatial_shapes,
                        level_start_index, sampling_locations, NULL, attention_weights, output, options);
}

/* The softmax of step a2 with the grouping the options select: all
 * n_levels*n_points logits of a (query, head), or each level's n_points. */
static int softmax_groups(int64_t rows, int64_t n_levels, int64_t n_points, const double *logits,
                          double *weights, int64_t options)
{
    if (options & OPT_PER_LEVEL_SOFTMAX)
        return msda_oracle_softmax(rows * n_levels, n_points, logits, weights);
    return msda_oracle_softmax(rows, n_levels * n_points, logits, weights);
}

/* Steps a1-a5: softmax (a2) of the raw logits, then the sampling with the
 * location taken from the reference point and the pixel offset (a1). */
int msda_oracle_forward_fused_grouped(int64_t N, int64_t Len_in, int64_t n_heads, int64_t n_groups, int64_t D,
                                      int64_t Len_q, int64_t n_levels, int64_t n_points, const double *value,
                                      const int64_t *spatial_shapes, const int64_t *level_start_index,
                                      const double *reference_points, const double *sampling_offsets,
                                      const double *attention_logits, double *output, int64_t options)
{
    if (n_groups <= 0) return -1;
    int64_t rows = N * Len_q * n_groups, cols = n_levels * n_points;
    if (rows < 0 || cols <= 0) return -1;
    double *attn = (double *)malloc(sizeof(double) * (size_t)(rows * cols + 1));
    if (!attn) return -1;
    int rc = softmax_groups(rows, n_levels, n_points, attention_logits, attn, options);
    if (!rc)
        rc = forward_impl(1, N, Len_in, n_heads, n_groups, D, Len_q, n_levels, n_points, value, spatial_shapes,
                          level_start_index, reference_points, sampling_offsets, attn, output, options);
    free(attn);
    return rc;
}

int msda_oracle_forward_fused(int64_t N, int64_t Len_in, int64_t n_heads, int64_t D, int64_t Len_q,
                              int64_t n_levels, int64_t n_points, const double *value,
                              const int64_t *spatial_shapes, const int64_t *level_start_index,
                              const double *reference_points, const double *sampling_offsets,
                              const double *attention_logits, double *output, int64_t options)
{
    return msda_oracle_forward_fused_grouped(N, Len_in, n_heads, n_heads, D, Len_q, n_levels, n_points, value,
                                             spatial_shapes, level_start_index, reference_points, sampling_offsets,
                                             attention_logits, output, options);
}

/* ------------------------------------------------------------------------- */
/* Steps a6-a8: the backward of a3-a5, derived from the bilinear formula of   */
/* [MSDA-tut] §2.3 (continuous and differentiable, so the gradient reaches    */
/* the offset branch).  For one sample s with corners c and weights w_c:      */
/*   grad_attn[s]   = sum_d g[d] * sample_s[d]                                */
/*   d sample/d px  = (1-fy)(v1-v0) + fy(v3-v2)      (corner order above)      */
/*   d sample/d py  = (1-fx)(v2-v0) + fx(v3-v1)                                */
/*   grad_loc_x     = A * sum_d g[d] d sample[d]/d px * W   (px = x*W - 0.5)   */
/*   grad_value[row_c] += A * w_c * g                    (in-map corners only) */
/* A corner outside the map has value 0 here as in the forward.  grad_value   */
/* is overwritten (zeroed first).                                             */
/* ------------------------------------------------------------------------- */
typedef struct {
    double *grad_value, *grad_loc, *grad_attn;
} grads_t;

static int backward_impl(int fused, int64_t N, int64_t Len_in, int64_t n_heads, int64_t n_groups, int64_t D,
                         int64_t Len_q, int64_t n_levels, int64_t n_points, const double *value,
                         const int64_t *shapes, const int64_t *starts, const double *loc_or_ref,
                         const double *offsets, const double *attn, const double *grad_out,
                         grads_t *gr, int64_t options)
{
    int align = (options & OPT_ALIGN_CORNERS) != 0;
    if (N < 0 || Len_in < 0 || n_heads <= 0 || D <= 0 || Len_q < 0 || n_levels <= 0 || n_points <= 0)
        return -1;
    if (n_groups <= 0 || n_heads % n_groups) return -1;
    if (check_levels(Len_in, n_levels, shapes, starts)) return -1;
    int64_t hpg = n_heads / n_groups;           /* heads per group */
    double *v = (double *)malloc(sizeof(double) * (size_t)(4 * D));
    if (!v) return -1;
    for (int64_t i = 0; i < N * Len_in * n_heads * D; ++i) gr->grad_value[i] = 0.0;
    /* a group's location and weight gradients sum over its heads */
    for (int64_t i = 0; i < N * Len_q * n_groups * n_levels * n_points; ++i) {
        gr->grad_attn[i] = 0.0;
        gr->grad_loc[2 * i] = gr->grad_loc[2 * i + 1] = 0.0;
    }
    for (int64_t n = 0; n < N; ++n)
        for (int64_t q = 0; q < Len_q; ++q)
            for (int64_t m = 0; m < n_heads; ++m) {
                const double *g = grad_out + ((n * Len_q + q) * n_heads + m) * D;
                int64_t gm = m / hpg;               /* the group whose locations head m samples */
                for (int64_t l = 0; l < n_levels; ++l) {
                    int64_t H = shapes[2 * l], W = shapes[2 * l + 1];
                    for (int64_t k = 0; k < n_points; ++k) {
                        int64_t s = (((n * Len_q + q) * n_groups + gm) * n_levels + l) * n_points + k;
                        corners_t c;
                        if (fused) {
                            const double *ref = loc_or_ref + ((n * Len_q + q) * n_levels + l) * 2;
                            corners_fused(ref[0], ref[1], offsets[2 * s], offsets[2 * s + 1], H, W,
                                          starts[l], align, &c);
                        } else {
                            corners_unfused(loc_or_ref[2 * s], loc_or_ref[2 * s + 1], H, W, starts[l], align, &c);
                        }
                        for (int ci = 0; ci < 4; ++ci)
                            for (int64_t d = 0; d < D; ++d)
                                v[ci * D + d] = c.row[ci] < 0 ? 0.0
                                    : value[((n * Len_in + c.row[ci]) * n_heads + m) * D + d];
                        double ga = 0.0, gx = 0.0, gy = 0.0;
                        for (int64_t d = 0; d < D; ++d) {
                            double smp = c.w[0] * v[d] + c.w[1] * v[D + d] + c.w[2] * v[2 * D + d]
                                       + c.w[3] * v[3 * D + d];
                            double dsx = (1.0 - c.fy) * (v[D + d] - v[d]) + c.fy * (v[3 * D + d] - v[2 * D + d]);
                            double dsy = (1.0 - c.fx) * (v[2 * D + d] - v[d]) + c.fx * (v[3 * D + d] - v[D + d]);
                            ga += g[d] * smp;
                            gx += g[d] * dsx;
                            gy += g[d] * dsy;
                        }
                        gr->grad_attn[s] += ga;
                        /* d px / d loc_x = W (W - 1 with align_corners) */
                        gr->grad_loc[2 * s + 0] += attn[s] * gx * (double)(align ? W - 1 : W);
                        gr->grad_loc[2 * s + 1] += attn[s] * gy * (double)(align ? H - 1 : H);
                        for (int ci = 0; ci < 4; ++ci) {
                            if (c.row[ci] < 0) continue;
                            double *gv = gr->grad_value + ((n * Len_in + c.row[ci]) * n_heads + m) * D;
                            for (int64_t d = 0; d < D; ++d) gv[d] += attn[s] * c.w[ci] * g[d];
                        }
                    }
                }
            }
    free(v);
    return 0;
}

int msda_oracle_backward(int64_t N, int64_t Len_in, int64_t n_heads, int64_t D, int64_t Len_q,
                         int64_t n_levels, int64_t n_points, const double *value,
                         const int64_t *spatial_shapes, const int64_t *level_start_index,
                         const double *sampling_locations, const double *attention_weights,
                         const double *grad_output, double *grad_value,
                         double *grad_sampling_locations, double *grad_attention_weights, int64_t options)
{
    grads_t gr = {grad_value, grad_sampling_locations, grad_attention_weights};
    return backward_impl(0, N, Len_in, n_heads, n_heads, D, Len_q, n_levels, n_points, value, spatial_shapes,
                         level_start_index, sampling_locations, NULL, attention_weights,
                         grad_output, &gr, options);
}

int msda_oracle_backward_grouped(int64_t N, int64_t Len_in, int64_t n_heads, int64_t n_groups, int64_t D,
                                 int64_t Len_q, int64_t n_levels, int64_t n_points, const double *value,
                                 const int64_t *spatial_shapes, const int64_t *level_start_index,
                                 const double *sampling_locations, const double *attention_weights,
                                 const double *grad_output, double *grad_value,
                                 double *grad_sampling_locations, double *grad_attention_weights, int64_t options)
{
    grads_t gr = {grad_value, grad_sampling_locations, grad_attention_weights};
    return backward_impl(0, N, Len_in, n_heads, n_groups, D, Len_q, n_levels, n_points, value, spatial_shapes,
                         level_start_index, sampling_locations, NULL, attention_weights,
                         grad_output, &gr, options);
}

/* ------------------------------------------------------------------------- */
/* Step a9: backward of the fused call, by the chain rule through a1 and a2.  */
/*   loc = ref + off / W            => grad_off_x = grad_loc_x / W,            */
/*                                     grad_ref_x[n,q,l] = sum_{m,k} grad_loc_x */
/*   A = softmax(logit) over j      => grad_logit_j = A_j (gA_j - sum_i A_i gA_i) */
/* ------------------------------------------------------------------------- */
int msda_oracle_backward_fused_grouped(int64_t N, int64_t Len_in, int64_t n_heads, int64_t n_groups, int64_t D,
                                       int64_t Len_q, int64_t n_levels, int64_t n_points, const double *value,
                                       const int64_t *spatial_shapes, const int64_t *level_start_index,
                                       const double *reference_points, const double *sampling_offsets,
                                       const double *attention_logits, const double *grad_output,
                                       double *grad_value, double *grad_reference_points,
                                       double *grad_sampling_offsets, double *grad_attention_logits, int64_t options)
{
    if (n_groups <= 0) return -1;
    int64_t rows = N * Len_q * n_groups, cols = n_levels * n_points;
    if (rows < 0 || cols <= 0) return -1;
    size_t ns = (size_t)(rows * cols + 1);
    double *attn = (double *)malloc(sizeof(double) * ns);
    double *gloc = (double *)malloc(sizeof(double) * 2 * ns);
    double *gattn = (double *)malloc(sizeof(double) * ns);
    int rc = -1;
    if (!attn || !gloc || !gattn) goto done;
    rc = softmax_groups(rows, n_levels, n_points, attention_logits, attn, options);
    if (rc) goto done;
    grads_t gr = {grad_value, gloc, gattn};
    rc = backward_impl(1, N, Len_in, n_heads, n_groups, D, Len_q, n_levels, n_points, value, spatial_shapes,
                       level_start_index, reference_points, sampling_offsets, attn, grad_output, &gr, options);
    if (rc) goto done;
    for (int64_t i = 0; i < N * Len_q * n_levels * 2; ++i) grad_reference_points[i] = 0.0;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t q = 0; q < Len_q; ++q)
            for (int64_t m = 0; m < n_groups; ++m) {        /* a row: one (n, q, group) */
                int64_t r = (n * Len_q + q) * n_groups + m;
                for (int64_t l = 0; l < n_levels; ++l) {
                    double H = (double)spatial_shapes[2 * l], W = (double)spatial_shapes[2 * l + 1];
                    double *gref = grad_reference_points + ((n * Len_q + q) * n_levels + l) * 2;
                    for (int64_t k = 0; k < n_points; ++k) {
                        int64_t s = r * cols + l * n_points + k;
                        grad_sampling_offsets[2 * s + 0] = gloc[2 * s + 0] / W;
                        grad_sampling_offsets[2 * s + 1] = gloc[2 * s + 1] / H;
                        gref[0] += gloc[2 * s + 0];
                        gref[1] += gloc[2 * s + 1];
                    }
                }
                /* the softmax's groups: the whole row, or each level's n_points */
                int64_t g = (options & OPT_PER_LEVEL_SOFTMAX) ? n_points : cols;
                for (int64_t j0 = 0; j0 < cols; j0 += g) {
                    double dot = 0.0;
                    for (int64_t j = j0; j < j0 + g; ++j) dot += attn[r * cols + j] * gattn[r * cols + j];
                    for (int64_t j = j0; j < j0 + g; ++j)
                        grad_attention_logits[r * cols + j] = attn[r * cols + j] * (gattn[r * cols + j] - dot);
                }
            }
done:
    free(attn);
    free(gloc);
    free(gattn);
    return rc;
}

int msda_oracle_backward_fused(int64_t N, int64_t Len_in, int64_t n_heads, int64_t D, int64_t Len_q,
                               int64_t n_levels, int64_t n_points, const double *value,
                               const int64_t *spatial_shapes, const int64_t *level_start_index,
                               const double *reference_points, const double *sampling_offsets,
                               const double *attention_logits, const double *grad_output,
                               double *grad_value, double *grad_reference_points,
                               double *grad_sampling_offsets, double *grad_attention_logits, int64_t options)
{
    return msda_oracle_backward_fused_grouped(N, Len_in, n_heads, n_heads, D, Len_q, n_levels, n_points, value,
                                              spatial_shapes, level_start_index, reference_points, sampling_offsets,
                                              attention_logits, grad_output, grad_value, grad_reference_points,
                                              grad_sampling_offsets, grad_attention_logits, options);
}

/* ========================================================================= */
/* The 3-D (volumetric / temporal) variant: "可变形注意力…" §5.3 -- on voxel */
/* or video features the offsets gain a z (or time) component and bilinear   */
/* interpolation becomes trilinear; everything else is as in 2-D.  Readings: */
/* a level is a volume (D_l, H_l, W_l) flattened as start + (z*H + y)*W + x; */
/* locations are (x, y, z) in [0,1]; pz = z*D - 0.5 (z*(D-1) with            */
/* align_corners); a corner outside the volume contributes 0.                */
/*   value [N][Len_in][n_heads][head_dim], spatial_shapes [L][3] = (D, H, W), */
/*   sampling_locations [N][Len_q][n_heads][L][K][3], output as in 2-D.       */
/* ========================================================================= */
typedef struct {
    int64_t row[8];     /* value row of corner c (or -1 outside); c = 4*k + 2*j + i */
    double w[8];        /* trilinear weight of corner c */
    double f[3];        /* fx, fy, fz */
} corners3_t;

static void corners3(const double *loc, int64_t Dd, int64_t H, int64_t W, int64_t start, int align, corners3_t *c)
{
    int64_t size[3] = {W, H, Dd};
    int64_t i0[3];
    double p[3];
    for (int a = 0; a < 3; ++a) {
        p[a] = align ? loc[a] * (double)(size[a] - 1) : loc[a] * (double)size[a] - 0.5;
        i0[a] = lower_corner(p[a], size[a]);
        c->f[a] = p[a] - (double)i0[a];
    }
    for (int k = 0; k < 2; ++k)
        for (int j = 0; j < 2; ++j)
            for (int i = 0; i < 2; ++i) {
                int ci = 4 * k + 2 * j + i;
                int64_t xc = i0[0] + i, yc = i0[1] + j, zc = i0[2] + k;
                c->w[ci] = (i ? c->f[0] : 1.0 - c->f[0]) * (j ? c->f[1] : 1.0 - c->f[1]) * (k ? c->f[2] : 1.0 - c->f[2]);
                c->row[ci] = (xc >= 0 && xc < W && yc >= 0 && yc < H && zc >= 0 && zc < Dd)
                                 ? start + (zc * H + yc) * W + xc : -1;
            }
}

static int check_levels3(int64_t Len_in, int64_t n_levels, const int64_t *shapes, const int64_t *starts)
{
    int64_t expect = 0;
    for (int64_t l = 0; l < n_levels; ++l) {
        if (shapes[3 * l] <= 0 || shapes[3 * l + 1] <= 0 || shapes[3 * l + 2] <= 0) return -1;
        if (starts[l] != expect) return -1;
        expect += shapes[3 * l] * shapes[3 * l + 1] * shapes[3 * l + 2];
    }
    return expect == Len_in ? 0 : -1;
}

int msda_oracle_forward3d(int64_t N, int64_t Len_in, int64_t n_heads, int64_t D, int64_t Len_q,
                          int64_t n_levels, int64_t n_points, const double *value,
                          const int64_t *spatial_shapes, const int64_t *level_start_index,
                          const double *sampling_locations, const double *attention_weights,
                          double *output, int64_t options)
{
    if (N < 0 || Len_in < 0 || n_heads <= 0 || D <= 0 || Len_q < 0 || n_levels <= 0 || n_points <= 0)
        return -1;
    if (check_levels3(Len_in, n_levels, spatial_shapes, level_start_index)) return -1;
    int align = (options & OPT_ALIGN_CORNERS) != 0;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t q = 0; q < Len_q; ++q)
            for (int64_t m = 0; m < n_heads; ++m) {
                double *o = output + ((n * Len_q + q) * n_heads + m) * D;
                for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
                for (int64_t l = 0; l < n_levels; ++l) {
                    const int64_t *sh = spatial_shapes + 3 * l;
                    for (int64_t k = 0; k < n_points; ++k) {
                        int64_t s = (((n * Len_q + q) * n_heads + m) * n_levels + l) * n_points + k;
                        corners3_t c;
                        corners3(sampling_locations + 3 * s, sh[0], sh[1], sh[2], level_start_index[l], align, &c);
                        for (int ci = 0; ci < 8; ++ci) {
                            if (c.row[ci] < 0) continue;
                            const double *v = value + ((n * Len_in + c.row[ci]) * n_heads + m) * D;
                            for (int64_t d = 0; d < D; ++d) o[d] += attention_weights[s] * c.w[ci] * v[d];
                        }
                    }
                }
            }
    return 0;
}

/* Backward of the 3-D forward.  For corner c = (i, j, k) the weight is
 * u_x(i) u_y(j) u_z(k) with u(0) = 1 - f, u(1) = f, so d w_c / d f_x =
 * (i ? 1 : -1) u_y(j) u_z(k), and likewise for y and z. */
int msda_oracle_backward3d(int64_t N, int64_t Len_in, int64_t n_heads, int64_t D, int64_t Len_q,
                           int64_t n_levels, int64_t n_points, const double *value,
                           const int64_t *spatial_shapes, const int64_t *level_start_index,
                           const double *sampling_locations, const double *attention_weights,
                           const double *grad_output, double *grad_value,
                           double *grad_sampling_locations, double *grad_attention_weights, int64_t options)
{
    if (N < 0 || Len_in < 0 || n_heads <= 0 || D <= 0 || Len_q < 0 || n_levels <= 0 || n_points <= 0)
        return -1;
    if (check_levels3(Len_in, n_levels, spatial_shapes, level_start_index)) return -1;
    int align = (options & OPT_ALIGN_CORNERS) != 0;
    for (int64_t i = 0; i < N * Len_in * n_heads * D; ++i) grad_value[i] = 0.0;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t q = 0; q < Len_q; ++q)
            for (int64_t m = 0; m < n_heads; ++m) {
                const double *g = grad_output + ((n * Len_q + q) * n_heads + m) * D;
                for (int64_t l = 0; l < n_levels; ++l) {
                    const int64_t *sh = spatial_shapes + 3 * l;
                    double scale[3] = {(double)(align ? sh[2] - 1 : sh[2]), (double)(align ? sh[1] - 1 : sh[1]),
                                       (double)(align ? sh[0] - 1 : sh[0])};
                    for (int64_t k = 0; k < n_points; ++k) {
                        int64_t s = (((n * Len_q + q) * n_heads + m) * n_levels + l) * n_points + k;
                        corners3_t c;
                        corners3(sampling_locations + 3 * s, sh[0], sh[1], sh[2], level_start_index[l], align, &c);
                        double ga = 0.0, gd[3] = {0.0, 0.0, 0.0};
                        for (int ci = 0; ci < 8; ++ci) {
                            if (c.row[ci] < 0) continue;     /* outside: value 0 */
                            const double *v = value + ((n * Len_in + c.row[ci]) * n_heads + m) * D;
                            double gv = 0.0;
                            for (int64_t d = 0; d < D; ++d) gv += g[d] * v[d];
                            int bit[3] = {ci & 1, (ci >> 1) & 1, (ci >> 2) & 1};
                            ga += c.w[ci] * gv;
                            for (int a = 0; a < 3; ++a) {
                                double dw = bit[a] ? 1.0 : -1.0;
                                for (int b = 0; b < 3; ++b)
                                    if (b != a) dw *= bit[b] ? c.f[b] : 1.0 - c.f[b];
                                gd[a] += dw * gv;
                            }
                            double *gvp = grad_value + ((n * Len_in + c.row[ci]) * n_heads + m) * D;
                            for (int64_t d = 0; d < D; ++d) gvp[d] += attention_weights[s] * c.w[ci] * g[d];
                        }
                        grad_attention_weights[s] = ga;
                        for (int a = 0; a < 3; ++a)
                            grad_sampling_locations[3 * s + a] = attention_weights[s] * gd[a] * scale[a];
                    }
                }
            }
    return 0;
}
