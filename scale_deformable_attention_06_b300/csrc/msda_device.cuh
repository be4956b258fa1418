// msda_device.cuh -- device-side building blocks shared by the MSDeformAttn
// kernels: the per-level table passed as a kernel parameter, 16-byte vector
// loads of value rows in fp32 or bf16, and the corner-record computation
// (pixel coordinate, floor, bilinear weights, zero padding).
//
// Bilinear sampling follows "可变形注意力：多尺度稀疏采样与视觉检测实战解析"
// §2.3 and the grid_sample module of its §3.2: px = x * W - 0.5 (align_corners
// = False), corners (x0,y0), (x0+1,y0), (x0,y0+1), (x0+1,y0+1) weighted
// (1-fx)(1-fy), fx(1-fy), (1-fx)fy, fx*fy, a corner outside the map reads 0.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace msda {

constexpr int kMaxLevels = 16;
constexpr int kMaxSamples = 256;     // n_levels * n_points per (query, head)
constexpr int kWarpsPerBlock = 8;
constexpr int kRecordsPerWarp = 64;  // corner records staged per warp and chunk

// Per-level geometry, a kernel parameter (constant bank, stream-ordered).
struct LevelTable {
    int H[kMaxLevels];
    int W[kMaxLevels];
    int start[kMaxLevels];     // first value row of the level
    float Hf[kMaxLevels];
    float Wf[kMaxLevels];
};

struct Dims {
    int N, Len_in, M, Len_q, L, K;
    int P;          // L * K samples per row
    int rows;       // N * Len_q * M rows (one row = one (n, q, m))
    int qm;         // Len_q * M rows per batch element
    int pix;        // M * D elements per value pixel
};

// Elements of T carried by one 16-byte load, and the lane layout that follows:
// R lanes cover the D channels of one row, a warp covers HW = 32 / R rows.
template <typename T, int D>
struct Layout {
    static constexpr int V = 16 / (int)sizeof(T);
    static constexpr int R = D / V;
    static constexpr int HW = 32 / R;
    static_assert(D % V == 0 && R >= 1 && R <= 32 && (R & (R - 1)) == 0, "unsupported head_dim");
};

// ---- 16-byte vectors ------------------------------------------------------
template <typename T> struct Vec;
template <> struct Vec<float> {
    float4 v;
    __device__ __forceinline__ float get(int i) const { return (&v.x)[i]; }
};
template <> struct Vec<__nv_bfloat16> {
    uint4 v;
    __device__ __forceinline__ float get(int i) const {
        uint32_t w = (&v.x)[i >> 1];
        return (i & 1) ? __uint_as_float(w & 0xffff0000u) : __uint_as_float(w << 16);
    }
};

// value rows: read-only path, kept in L2 (evict_last) since every row is
// gathered by many queries.
__device__ __forceinline__ uint64_t l2_keep_policy() {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

template <typename T>
__device__ __forceinline__ Vec<T> load_value(const T *p, uint64_t pol) {
    Vec<T> r;
    uint32_t a, b, c, d;
    asm("ld.global.nc.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "l"(p), "l"(pol));
    if constexpr (sizeof(T) == 4) {
        r.v = make_float4(__uint_as_float(a), __uint_as_float(b), __uint_as_float(c), __uint_as_float(d));
    } else {
        r.v = make_uint4(a, b, c, d);
    }
    return r;
}

// Streamed tensors (read or written once): evict-first.
__device__ __forceinline__ float2 load_stream2(const float *p) { return __ldcs(reinterpret_cast<const float2 *>(p)); }
__device__ __forceinline__ float load_stream1(const float *p) { return __ldcs(p); }

template <typename T, int V>
__device__ __forceinline__ void store_row(T *p, const float (&acc)[V]) {
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int i = 0; i < V; i += 4)
            __stcs(reinterpret_cast<float4 *>(p) + i / 4, make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]));
    } else {
        uint32_t w[V / 2];
#pragma unroll
        for (int i = 0; i < V; i += 2) {
            __nv_bfloat162 h = __floats2bfloat162_rn(acc[i], acc[i + 1]);
            w[i / 2] = *reinterpret_cast<uint32_t *>(&h);
        }
#pragma unroll
        for (int i = 0; i < V / 2; i += 4)
            __stcs(reinterpret_cast<uint4 *>(p) + i / 4, make_uint4(w[i], w[i + 1], w[i + 2], w[i + 3]));
    }
}

// Load the V channels of a row of grad_output (or any row) as fp32.
template <typename T, int V>
__device__ __forceinline__ void load_row_f32(const T *p, float (&g)[V]) {
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int i = 0; i < V; i += 4) {
            float4 t = __ldcs(reinterpret_cast<const float4 *>(p) + i / 4);
            g[i] = t.x; g[i + 1] = t.y; g[i + 2] = t.z; g[i + 3] = t.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < V; i += 8) {
            uint4 t = __ldcs(reinterpret_cast<const uint4 *>(p) + i / 8);
            uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                g[i + 2 * j] = __uint_as_float(w[j] << 16);
                g[i + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
            }
        }
    }
}

// ---- pixel coordinates ------------------------------------------------------
// Unfused: px = x * size - 0.5.  The floor is taken of RN(RN(x*size) - 0.5);
// the fraction adds back the exact rounding error of the product (fma), so it
// is accurate to about 1e-7 px instead of half an ulp of px.
__device__ __forceinline__ void pixel_coord(float x, float size, float &fl, float &frac) {
    float p = __fmul_rn(x, size);
    float e = __fmaf_rn(x, size, -p);          // x*size = p + e exactly
    float ph = __fsub_rn(p, 0.5f);
    fl = floorf(ph);
    frac = __fadd_rn(__fsub_rn(ph, fl), e);
}

// Fused: px = ref * size + off - 0.5 (= (ref + off/size) * size - 0.5).  The
// floor is taken of RN(RN(ref*size) + RN(off - 0.5)); the fraction carries the
// rounding errors of all three operations (fma and two-sum).
__device__ __forceinline__ float two_sum_err(float a, float b, float s) {
    float bb = __fsub_rn(s, a);
    return __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ void pixel_coord_fused(float ref, float off, float size, float &fl, float &frac) {
    float p = __fmul_rn(ref, size);
    float e1 = __fmaf_rn(ref, size, -p);
    float t = __fsub_rn(off, 0.5f);
    float e2 = two_sum_err(off, -0.5f, t);
    float s = __fadd_rn(p, t);
    float e3 = two_sum_err(p, t, s);
    fl = floorf(s);
    frac = __fadd_rn(__fsub_rn(s, fl), __fadd_rn(e1, __fadd_rn(e2, e3)));
}

// One sample's four corners: element offsets (relative to the row's value
// base) and bilinear weights, zero for corners outside the map.  An outside
// corner gets offset 0 (a valid address) so that its load needs no predicate.
struct Corners {
    int4 off;
    float4 w;        // bilinear weight * mask (no attention weight)
    unsigned mask;   // bit c set if corner c is inside the map
};

__device__ __forceinline__ Corners make_corners(float x0f, float fx, float y0f, float fy, int W, int H, float Wf,
                                                float Hf, int start, int pix) {
    // clamp far-away samples so the integer arithmetic cannot overflow
    int x0 = (int)fminf(fmaxf(x0f, -2.f), Wf + 1.f);
    int y0 = (int)fminf(fmaxf(y0f, -2.f), Hf + 1.f);
    bool vx0 = (unsigned)x0 < (unsigned)W, vx1 = (unsigned)(x0 + 1) < (unsigned)W;
    bool vy0 = (unsigned)y0 < (unsigned)H, vy1 = (unsigned)(y0 + 1) < (unsigned)H;
    float wx1 = fx, wx0 = 1.f - fx, wy1 = fy, wy0 = 1.f - fy;
    int base = (start + y0 * W + x0) * pix;
    Corners c;
    bool v0 = vx0 && vy0, v1 = vx1 && vy0, v2 = vx0 && vy1, v3 = vx1 && vy1;
    c.off.x = v0 ? base : 0;
    c.off.y = v1 ? base + pix : 0;
    c.off.z = v2 ? base + W * pix : 0;
    c.off.w = v3 ? base + (W + 1) * pix : 0;
    c.w.x = v0 ? wx0 * wy0 : 0.f;
    c.w.y = v1 ? wx1 * wy0 : 0.f;
    c.w.z = v2 ? wx0 * wy1 : 0.f;
    c.w.w = v3 ? wx1 * wy1 : 0.f;
    c.mask = (v0 ? 1u : 0u) | (v1 ? 2u : 0u) | (v2 ? 4u : 0u) | (v3 ? 8u : 0u);
    return c;
}

// acc[0..V) += w * v
template <typename T, int V>
__device__ __forceinline__ void fma_row(float (&acc)[V], float w, const Vec<T> &v) {
    if constexpr (sizeof(T) == 4) {
        float2 ww = make_float2(w, w);
#pragma unroll
        for (int i = 0; i < V; i += 2) {
            float2 a = make_float2(acc[i], acc[i + 1]);
            float2 x = make_float2(v.get(i), v.get(i + 1));
            a = __ffma2_rn(ww, x, a);
            acc[i] = a.x;
            acc[i + 1] = a.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = __fmaf_rn(w, v.get(i), acc[i]);
    }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace msda
