// msda_backward.cu -- backward kernels of the MSDeformAttn core.
//
// For one sample s of row (n, q, m) with corners c, bilinear weights w_c
// (zero outside the map), attention weight A and g = grad_output[n][q][m*D..]:
//   grad_attention_weights[s]  = sum_c w_c <g, v_c>
//   d/dpx = sum_c (d w_c / d fx) <g, v_c>,  d/dpy likewise,  px = x * W - 0.5
//   grad_sampling_locations[s] = A * (W * d/dpx, H * d/dpy)
//   grad_value[n][corner c][m] += A * w_c * g            (corners inside the map)
// derived from the bilinear form of "可变形注意力：多尺度稀疏采样与视觉检测实战
// 解析" §2.3 (continuous, so the gradient reaches the offset branch).
//
// Work decomposition follows the forward (msda_forward.cu): a warp owns HW
// rows with R lanes per row; phase 1 stages corner records in shared memory,
// phase 2 gathers the four corner vectors of each sample, forms the per-corner
// dot products <g, v_c> over the lane's channels, reduces them over the R
// lanes of the row with shuffles, and scatters A * w_c * g into grad_value with
// one vector reduction (red.global.add.v4.f32) per corner and 4 channels;
// phase 3 writes the chunk's grad_attention_weights / grad_sampling_locations
// coalesced.
//
// Deterministic mode replaces the fp32 reductions by 64-bit integer ones in
// fixed point (integer addition is associative, so the order in which the
// atomics land does not matter), with a scale chosen from a bound on the total
// |contribution| so that no sum can overflow, then converts to fp32.
#include "msda_device.cuh"
#include "msda_launch.h"

namespace msda {

struct BwdArgs {
    const void *value;
    const float *loc;
    const float *attn;
    const void *grad_out;
    float *grad_value;
    float *grad_loc;
    float *grad_attn;
    unsigned long long *fixed;     // deterministic: [N*Len_in*M*D] accumulators
    const unsigned *bound_bits;    // deterministic: bits of max row bound (a float)
    Dims d;
    LevelTable lv;
    unsigned char level_of[kMaxSamples];
};

__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ void red_add_u64(unsigned long long *p, long long v) {
    asm volatile("red.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Power-of-two scale of the fixed-point sums: every partial sum is at most
// rows * max_row_bound < 2^62 after scaling.
__device__ __forceinline__ int fixed_shift(unsigned bits, int rows) {
    const double bound = (double)__uint_as_float(bits) * (double)rows;
    if (!(bound > 0.0)) return 0;
    int e;
    frexp(bound, &e);          // bound < 2^e
    int shift = 62 - e;
    return shift < -60 ? -60 : (shift > 100 ? 100 : shift);
}

template <typename T, int D, bool DET>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
msda_backward_kernel(const __grid_constant__ BwdArgs a) {
    using Lay = Layout<T, D>;
    constexpr int V = Lay::V, R = Lay::R, HW = Lay::HW;
    constexpr int JC = kRecordsPerWarp / HW;

    __shared__ int4 s_off[kWarpsPerBlock][kRecordsPerWarp];
    __shared__ float4 s_w[kWarpsPerBlock][kRecordsPerWarp];    // bilinear * mask
    __shared__ float4 s_aux[kWarpsPerBlock][kRecordsPerWarp];  // fx, fy, A, mask bits
    __shared__ float4 s_res[kWarpsPerBlock][kRecordsPerWarp];  // gA, A*d/dpx, A*d/dpy

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = (blockIdx.x * kWarpsPerBlock + warp) * HW;
    const Dims &dm = a.d;
    if (row0 >= dm.rows) return;
    const int P = dm.P;

    const int h = lane / R, ch = lane % R;
    const int row = row0 + h;
    const bool row_ok = row < dm.rows;
    const int rowc = row_ok ? row : dm.rows - 1;
    const int n = rowc / dm.qm;
    const int m = rowc % dm.M;
    const size_t vrow = ((size_t)n * dm.Len_in * dm.M + m) * D + ch * V;
    const T *vbase = static_cast<const T *>(a.value) + vrow;
    const uint64_t pol = l2_keep_policy();

    float g[V];
    load_row_f32<T, V>(static_cast<const T *>(a.grad_out) + (size_t)rowc * D + ch * V, g);
    if (!row_ok) {
#pragma unroll
        for (int i = 0; i < V; ++i) g[i] = 0.f;
    }
    float scale = 1.f;
    if constexpr (DET) scale = ldexpf(1.f, fixed_shift(*a.bound_bits, dm.rows));

    for (int s0 = 0; s0 < P; s0 += JC) {
        const int J = min(JC, P - s0);
        // ---- phase 1: corner records
        for (int i = lane; i < HW * J; i += 32) {
            const int hh = i % HW, j = i / HW;
            const int r = row0 + hh, s = s0 + j;
            int4 off = make_int4(0, 0, 0, 0);
            float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
            float4 aux = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < dm.rows) {
                const int l = a.level_of[s];
                const float Wf = a.lv.Wf[l], Hf = a.lv.Hf[l];
                const size_t si = (size_t)r * P + s;
                const float2 lc = load_stream2(a.loc + 2 * si);
                float x0, fx, y0, fy;
                pixel_coord(lc.x, Wf, x0, fx);
                pixel_coord(lc.y, Hf, y0, fy);
                const float A = load_stream1(a.attn + si);
                Corners c = make_corners(x0, fx, y0, fy, a.lv.W[l], a.lv.H[l], Wf, Hf, a.lv.start[l], dm.pix);
                off = c.off;
                w = c.w;
                aux = make_float4(fx, fy, A, __uint_as_float(c.mask));
            }
            s_off[warp][i] = off;
            s_w[warp][i] = w;
            s_aux[warp][i] = aux;
        }
        __syncwarp();
        // ---- phase 2: gather, dot products, scatter into grad_value
        for (int j = 0; j < J; ++j) {
            const int rec = j * HW + h;
            const int4 o = s_off[warp][rec];
            const float4 w = s_w[warp][rec];
            const float4 ax = s_aux[warp][rec];
            const unsigned mask = __float_as_uint(ax.w);
            const Vec<T> v0 = load_value(vbase + o.x, pol);
            const Vec<T> v1 = load_value(vbase + o.y, pol);
            const Vec<T> v2 = load_value(vbase + o.z, pol);
            const Vec<T> v3 = load_value(vbase + o.w, pol);
            float t0 = 0.f, t1 = 0.f, t2 = 0.f, t3 = 0.f;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                t0 = __fmaf_rn(g[i], v0.get(i), t0);
                t1 = __fmaf_rn(g[i], v1.get(i), t1);
                t2 = __fmaf_rn(g[i], v2.get(i), t2);
                t3 = __fmaf_rn(g[i], v3.get(i), t3);
            }
#pragma unroll
            for (int o2 = R / 2; o2 > 0; o2 >>= 1) {
                t0 += __shfl_xor_sync(0xffffffffu, t0, o2);
                t1 += __shfl_xor_sync(0xffffffffu, t1, o2);
                t2 += __shfl_xor_sync(0xffffffffu, t2, o2);
                t3 += __shfl_xor_sync(0xffffffffu, t3, o2);
            }
            // corners outside the map read as zero in the gradient formulas
            t0 = (mask & 1u) ? t0 : 0.f;
            t1 = (mask & 2u) ? t1 : 0.f;
            t2 = (mask & 4u) ? t2 : 0.f;
            t3 = (mask & 8u) ? t3 : 0.f;
            const float fx = ax.x, fy = ax.y, A = ax.z;
            if (ch == 0) {
                const float ga = w.x * t0 + w.y * t1 + w.z * t2 + w.w * t3;
                const float dx = (1.f - fy) * (t1 - t0) + fy * (t3 - t2);
                const float dy = (1.f - fx) * (t2 - t0) + fx * (t3 - t1);
                s_res[warp][rec] = make_float4(ga, A * dx, A * dy, 0.f);
            }
            if (row_ok) {
                const float cw[4] = {A * w.x, A * w.y, A * w.z, A * w.w};
                const int co[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (!(mask & (1u << c))) continue;
                    if constexpr (DET) {
                        unsigned long long *dst = a.fixed + vrow + co[c];
#pragma unroll
                        for (int i = 0; i < V; ++i) red_add_u64(dst + i, __float2ll_rn(cw[c] * g[i] * scale));
                    } else {
                        float *dst = a.grad_value + vrow + co[c];
#pragma unroll
                        for (int i = 0; i < V; i += 4)
                            red_add_v4(dst + i, cw[c] * g[i], cw[c] * g[i + 1], cw[c] * g[i + 2], cw[c] * g[i + 3]);
                    }
                }
            }
        }
        __syncwarp();
        // ---- phase 3: per-sample gradients, coalesced
        for (int i = lane; i < HW * J; i += 32) {
            const int hh = i % HW, j = i / HW;
            const int r = row0 + hh, s = s0 + j;
            if (r < dm.rows) {
                const int l = a.level_of[s];
                const float4 res = s_res[warp][i];
                const size_t si = (size_t)r * P + s;
                __stcs(a.grad_attn + si, res.x);
                __stcs(reinterpret_cast<float2 *>(a.grad_loc) + si, make_float2(res.y * a.lv.Wf[l], res.z * a.lv.Hf[l]));
            }
        }
        __syncwarp();
    }
}

// ---- helpers of the backward -----------------------------------------------
__global__ void zero_f32_kernel(float4 *p, size_t n4) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
        p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void zero_u64_kernel(ulonglong2 *p, size_t n2) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n2; i += (size_t)gridDim.x * blockDim.x)
        p[i] = make_ulonglong2(0ull, 0ull);
}

// max over rows of (sum_s |A_s|) * (max_d |g_d|), as float bits (non-negative
// floats order like their bit patterns, so an integer max is exact and
// independent of the order of the atomics).
template <typename T, int D>
__global__ void row_bound_kernel(const float *attn, const T *grad_out, int rows, int P, unsigned *bound_bits) {
    float best = 0.f;
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += gridDim.x * blockDim.x) {
        float sa = 0.f;
        for (int s = 0; s < P; ++s) sa += fabsf(attn[(size_t)r * P + s]);
        float gm = 0.f;
        const T *g = grad_out + (size_t)r * D;
        for (int d = 0; d < D; ++d) gm = fmaxf(gm, fabsf((float)g[d]));
        // round the product up a little so the bound stays an upper bound
        best = fmaxf(best, sa * gm * 1.0001f);
    }
    best = warp_max(best);
    if ((threadIdx.x & 31) == 0) atomicMax(bound_bits, __float_as_uint(best));
}

__global__ void fixed_to_f32_kernel(const unsigned long long *fixed, const unsigned *bound_bits, int rows,
                                    float *grad_value, size_t n, int accumulate) {
    const int shift = fixed_shift(*bound_bits, rows);
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const float v = (float)ldexp((double)(long long)fixed[i], -shift);
        grad_value[i] = accumulate ? grad_value[i] + v : v;
    }
}

static unsigned grid_for(size_t work, int threads) {
    size_t b = (work + threads - 1) / threads;
    if (b > 148u * 32u) b = 148u * 32u;
    return (unsigned)(b ? b : 1);
}

size_t backward_workspace_bytes(const LaunchGeometry &g, int D, bool deterministic) {
    if (!deterministic) return 0;
    const size_t n = (size_t)g.d.N * g.d.Len_in * g.d.M * D;
    return 256 + n * sizeof(unsigned long long);
}

template <typename T, int D>
static cudaError_t launch_bwd_t(const LaunchGeometry &g, const void *value, const float *loc, const float *attn,
                                const void *grad_out, float *grad_value, float *grad_loc, float *grad_attn,
                                bool det, bool accumulate, void *workspace, cudaStream_t stream) {
    constexpr int HW = Layout<T, D>::HW;
    const size_t nval = (size_t)g.d.N * g.d.Len_in * g.d.M * D;
    BwdArgs a{};
    a.value = value;
    a.loc = loc;
    a.attn = attn;
    a.grad_out = grad_out;
    a.grad_value = grad_value;
    a.grad_loc = grad_loc;
    a.grad_attn = grad_attn;
    a.d = g.d;
    a.lv = g.lv;
    for (int s = 0; s < kMaxSamples; ++s) a.level_of[s] = g.level_of[s];
    if (det) {
        unsigned *hdr = static_cast<unsigned *>(workspace);
        unsigned long long *fixed = reinterpret_cast<unsigned long long *>(static_cast<char *>(workspace) + 256);
        a.fixed = fixed;
        a.bound_bits = hdr;
        // header (256 bytes) and accumulators are contiguous: zero both
        zero_u64_kernel<<<grid_for((nval * 8 + 256) / 16, 256), 256, 0, stream>>>(
            static_cast<ulonglong2 *>(workspace), (nval * 8 + 256) / 16);
        if (g.d.rows > 0)
            row_bound_kernel<T, D><<<grid_for(g.d.rows, 256), 256, 0, stream>>>(
                attn, static_cast<const T *>(grad_out), g.d.rows, g.d.P, hdr);
    } else if (!accumulate && nval > 0) {
        zero_f32_kernel<<<grid_for(nval / 4, 256), 256, 0, stream>>>(reinterpret_cast<float4 *>(grad_value), nval / 4);
    }
    if (g.d.rows > 0) {
        const long long warps = ((long long)g.d.rows + HW - 1) / HW;
        const unsigned blocks = (unsigned)((warps + kWarpsPerBlock - 1) / kWarpsPerBlock);
        if (det)
            msda_backward_kernel<T, D, true><<<blocks, kWarpsPerBlock * 32, 0, stream>>>(a);
        else
            msda_backward_kernel<T, D, false><<<blocks, kWarpsPerBlock * 32, 0, stream>>>(a);
    }
    if (det && nval > 0)
        fixed_to_f32_kernel<<<grid_for(nval, 256), 256, 0, stream>>>(a.fixed, a.bound_bits, g.d.rows, grad_value,
                                                                      nval, accumulate ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_backward(const LaunchGeometry &g, int dtype, int D, const void *value, const float *loc,
                            const float *attn, const void *grad_out, float *grad_value, float *grad_loc,
                            float *grad_attn, bool det, bool accumulate, void *workspace, cudaStream_t stream) {
#define MSDA_BWD(T, DD) \
    return launch_bwd_t<T, DD>(g, value, loc, attn, grad_out, grad_value, grad_loc, grad_attn, det, accumulate, \
                               workspace, stream)
    if (dtype == 0) {
        switch (D) {
            case 8: MSDA_BWD(float, 8);
            case 16: MSDA_BWD(float, 16);
            case 32: MSDA_BWD(float, 32);
            case 64: MSDA_BWD(float, 64);
        }
    } else {
        switch (D) {
            case 8: MSDA_BWD(__nv_bfloat16, 8);
            case 16: MSDA_BWD(__nv_bfloat16, 16);
            case 32: MSDA_BWD(__nv_bfloat16, 32);
            case 64: MSDA_BWD(__nv_bfloat16, 64);
        }
    }
#undef MSDA_BWD
    return cudaErrorInvalidValue;
}

}  // namespace msda
