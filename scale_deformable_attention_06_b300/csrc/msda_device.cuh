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

// ---- the debug build (compiled with -DMSDA_DEBUG into libmsda_debug.so) ------
// Every value gather, grad_output load and grad_value / fixed-point reduction
// is checked against the extent of its tensor (and the 16-byte alignment of
// vector accesses).  A bad access is counted in the translation unit's
// counter and skipped: a load reads the tensor's first elements instead, a
// reduction is dropped.  Nothing traps.  Release builds compile the checks
// away (MSDA_ADDR is the pointer itself, MSDA_IN is true).
#ifdef MSDA_DEBUG
static __device__ unsigned long long g_debug_violations;

// p (inside or outside [base, base + total)) if its `width` elements lie in
// the tensor and a 16-byte access there is aligned, else base.
template <typename T>
__device__ __forceinline__ T *debug_addr(T *base, T *p, long long total, int width) {
    const long long i = (long long)(p - base);
    const bool ok = i >= 0 && i + width <= total && (width * sizeof(T) < 16 || ((i * (long long)sizeof(T)) & 15) == 0);
    if (!ok) atomicAdd(&g_debug_violations, 1ull);
    return ok ? p : base;
}
template <typename T>
__device__ __forceinline__ bool debug_in(const T *base, const T *p, long long total, int width) {
    const long long i = (long long)(p - base);
    const bool ok = i >= 0 && i + width <= total;
    if (!ok) atomicAdd(&g_debug_violations, 1ull);
    return ok;
}
#define MSDA_ADDR(base, p, total, width) ::msda::debug_addr((base), (p), (long long)(total), (width))
#define MSDA_IN(base, p, total, width) ::msda::debug_in((base), (p), (long long)(total), (width))
// the host side of a translation unit's counter: read it, and zero it if asked
#define MSDA_DEBUG_COUNTER(fn)                                                               \
    unsigned long long fn(bool reset) {                                                      \
        unsigned long long v = 0;                                                            \
        cudaMemcpyFromSymbol(&v, g_debug_violations, sizeof(v));                             \
        if (reset) {                                                                         \
            const unsigned long long z = 0;                                                  \
            cudaMemcpyToSymbol(g_debug_violations, &z, sizeof(z));                           \
        }                                                                                    \
        return v;                                                                            \
    }
#else
#define MSDA_ADDR(base, p, total, width) (p)
#define MSDA_IN(base, p, total, width) true
#endif

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
    float Sx[kMaxLevels];      // pixel scale: W (W - 1 with align_corners)
    float Sy[kMaxLevels];      // H (H - 1 with align_corners)
    float Rx[kMaxLevels];      // offset pixels to pixel coordinate: Sx / W (fp32)
    float Ry[kMaxLevels];      // Sy / H
    float shift;               // 0.5 (0 with align_corners)
};

struct Dims {
    int N, Len_in, M, Len_q, L, K;
    int per_level_softmax;     // fused calls: softmax over each level's K logits
    int P;          // L * K samples per row
    int rows;       // N * Len_q * M rows (one row = one (n, q, m))
    int qm;         // Len_q * M rows per batch element
    int pix;        // M * D elements per value pixel
};

// Elements of T carried by one 16-byte load, and the lane layout that follows:
// R lanes cover the D channels of one row, NV 16-byte vectors a lane (vector
// k of lane ch holds channels (k * R + ch) * V ..), a warp covers HW = 32 / R
// rows.
template <typename T, int D>
struct Layout {
    static constexpr int V = 16 / (int)sizeof(T);
    static constexpr int R = D / V < 32 ? D / V : 32;
    static constexpr int NV = D / (V * R);
    static constexpr int HW = 32 / R;
    static_assert(D % V == 0 && R >= 1 && (R & (R - 1)) == 0 && NV * V * R == D, "unsupported head_dim");
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
// The pixel coordinate is carried as an unevaluated sum hi + lo of two floats
// (lo holds the exact rounding errors of the operations that formed hi), and
// the corner is floor() of that exact sum, as the method defines it (x0 =
// floor(px)), not floor() of the rounded hi: a coordinate a rounding below an
// integer stays in the lower cell with a fraction near 1.
__device__ __forceinline__ float two_sum_err(float a, float b, float s) {
    float bb = __fsub_rn(s, a);
    return __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// fl = floor(hi + lo), frac = hi + lo - fl in [0, 1] (rounded once).
__device__ __forceinline__ void floor_frac(float hi, float lo, float &fl, float &frac) {
    const float f0 = floorf(hi);
    const float t = __fsub_rn(hi, f0);             // hi - floor(hi), exact for |hi| >= 1
    // -1: the exact sum lies below f0; +1: at or above f0 + 1
    const float c = lo < -t ? -1.f : (lo >= __fsub_rn(1.f, t) ? 1.f : 0.f);
    fl = __fadd_rn(f0, c);
    frac = __fadd_rn(__fsub_rn(t, c), lo);
}

// Unfused: px = x * S - shift (S = W, shift = 0.5; with align_corners S = W - 1,
// shift = 0), with the exact errors of the product (fma) and the subtraction.
__device__ __forceinline__ void pixel_coord(float x, float S, float shift, float &fl, float &frac) {
    const float p = __fmul_rn(x, S);
    const float e1 = __fmaf_rn(x, S, -p);          // x*S = p + e1 exactly
    const float ph = __fsub_rn(p, shift);
    const float e2 = two_sum_err(p, -shift, ph);   // p - shift = ph + e2 exactly
    floor_frac(ph, __fadd_rn(e1, e2), fl, frac);
}

// Fused: px = ref * S + off * Rr - shift, the same point as (ref + off / W) * S
// - shift with Rr = S / W (1 without align_corners), formed without the
// division, with the errors of every operation (fma and two-sum).
// Default convention (S = size, Rr = 1, shift = 0.5).
__device__ __forceinline__ void pixel_coord_fused(float ref, float off, float size, float &fl, float &frac) {
    const float p = __fmul_rn(ref, size);
    const float e1 = __fmaf_rn(ref, size, -p);
    const float t = __fsub_rn(off, 0.5f);
    const float e2 = two_sum_err(off, -0.5f, t);
    const float s = __fadd_rn(p, t);
    const float e3 = two_sum_err(p, t, s);
    floor_frac(s, __fadd_rn(e1, __fadd_rn(e2, e3)), fl, frac);
}

// Any convention; for the default one it gives the same floor and fraction as
// the function above (off * 1 and its error term 0 are exact).
__device__ __forceinline__ void pixel_coord_fused(float ref, float off, float S, float Rr, float shift, float &fl,
                                                  float &frac) {
    const float p = __fmul_rn(ref, S);
    const float e1 = __fmaf_rn(ref, S, -p);
    const float t0 = __fmul_rn(off, Rr);
    const float ea = __fmaf_rn(off, Rr, -t0);
    const float t = __fsub_rn(t0, shift);
    const float eb = two_sum_err(t0, -shift, t);
    const float s = __fadd_rn(p, t);
    const float e3 = two_sum_err(p, t, s);
    floor_frac(s, __fadd_rn(e1, __fadd_rn(ea, __fadd_rn(eb, e3))), fl, frac);
}

// Attention weight of sample k of a softmax group of n logits at lg (max
// subtracted, then a multiply by 1/sum): one fixed order, so every kernel that
// calls it gets the same value.
__device__ __forceinline__ void group_softmax_stats(const float *lg, int n, float &mx, float &inv) {
    mx = -INFINITY;
    for (int i = 0; i < n; ++i) mx = fmaxf(mx, __ldg(lg + i));
    float sum = 0.f;
    for (int i = 0; i < n; ++i) sum += expf(__ldg(lg + i) - mx);
    inv = 1.f / sum;
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

// ---- 16-byte corner records -------------------------------------------------
// One sample's four corners in 16 bytes, written once per sample and read by
// every lane of its row:
//   .x  value row (pixel index, < 2^28) of corner 00 clamped into the map, with
//       four validity bits above it: bit 28 column x0 inside, 29 column x0+1,
//       30 row y0, 31 row y0+1;
//   .y  fx,  .z  fy  (fractions of the pixel coordinate);
//   .w  the sample's attention weight.
// A corner is inside the map when its column and its row are.  Corners 10/01/11
// step from the clamped corner 00 by one column / one row only when both
// columns / both rows are inside; otherwise the step is 0, which keeps every
// address inside the map and, since then one of the two neighbours has weight
// 0, leaves the inside neighbour at its true address.
constexpr uint32_t kPixMask = 0x0fffffffu;

__device__ __forceinline__ uint4 pack_record(float x0f, float fx, float y0f, float fy, float A, int W, int H,
                                             float Wf, float Hf, int start) {
    // clamp far-away samples so the integer arithmetic cannot overflow
    const int x0 = (int)fminf(fmaxf(x0f, -2.f), Wf + 1.f);
    const int y0 = (int)fminf(fmaxf(y0f, -2.f), Hf + 1.f);
    const uint32_t fl = ((unsigned)x0 < (unsigned)W ? 1u : 0u) | ((unsigned)(x0 + 1) < (unsigned)W ? 2u : 0u) |
                        ((unsigned)y0 < (unsigned)H ? 4u : 0u) | ((unsigned)(y0 + 1) < (unsigned)H ? 8u : 0u);
    const int cx = min(max(x0, 0), W - 1), cy = min(max(y0, 0), H - 1);
    const uint32_t p = (uint32_t)(start + cy * W + cx);
    return make_uint4(p | (fl << 28), __float_as_uint(fx), __float_as_uint(fy), __float_as_uint(A));
}

struct Unpacked {
    uint32_t pix[4];    // value row of corners 00, 10, 01, 11 (always inside the map)
    float w[4];         // bilinear weights, 0 for corners outside the map
    bool in[4];         // corner inside the map
    float fx, fy, A;
};

// W: width of the sample's level (pixels per row of the map)
__device__ __forceinline__ Unpacked unpack_record(uint4 rc, int W) {
    Unpacked u;
    const uint32_t fl = rc.x >> 28;
    const uint32_t p = rc.x & kPixMask;
    const uint32_t dx = ((fl & 3u) == 3u) ? 1u : 0u;
    const uint32_t dy = ((fl & 12u) == 12u) ? (uint32_t)W : 0u;
    u.pix[0] = p; u.pix[1] = p + dx; u.pix[2] = p + dy; u.pix[3] = p + dy + dx;
    u.fx = __uint_as_float(rc.y); u.fy = __uint_as_float(rc.z); u.A = __uint_as_float(rc.w);
    const float wx0 = (fl & 1u) ? 1.f - u.fx : 0.f, wx1 = (fl & 2u) ? u.fx : 0.f;
    const float wy0 = (fl & 4u) ? 1.f - u.fy : 0.f, wy1 = (fl & 8u) ? u.fy : 0.f;
    u.w[0] = wx0 * wy0; u.w[1] = wx1 * wy0; u.w[2] = wx0 * wy1; u.w[3] = wx1 * wy1;
    u.in[0] = (fl & 5u) == 5u; u.in[1] = (fl & 6u) == 6u; u.in[2] = (fl & 9u) == 9u; u.in[3] = (fl & 10u) == 10u;
    return u;
}

// ---- 4-channel lane vectors (any storage type) ------------------------------
template <typename T>
__device__ __forceinline__ float4 load4_value(const T *p, uint64_t pol) {
    uint32_t a, b, c, d;
    if constexpr (sizeof(T) == 4) {
        asm("ld.global.nc.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
            : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "l"(p), "l"(pol));
        return make_float4(__uint_as_float(a), __uint_as_float(b), __uint_as_float(c), __uint_as_float(d));
    } else {
        asm("ld.global.nc.L2::cache_hint.v2.u32 {%0,%1}, [%2], %3;" : "=r"(a), "=r"(b) : "l"(p), "l"(pol));
        return make_float4(__uint_as_float(a << 16), __uint_as_float(a & 0xffff0000u), __uint_as_float(b << 16),
                           __uint_as_float(b & 0xffff0000u));
    }
}

template <typename T>
__device__ __forceinline__ float4 load4_stream(const T *p) {
    if constexpr (sizeof(T) == 4) {
        return __ldcs(reinterpret_cast<const float4 *>(p));
    } else {
        const uint2 u = __ldcs(reinterpret_cast<const uint2 *>(p));
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                           __uint_as_float(u.y & 0xffff0000u));
    }
}

// y + a * x, two packed fp32 FMAs
__device__ __forceinline__ float4 ffma4(float a, float4 x, float4 y) {
    const float2 aa = make_float2(a, a);
    const float2 lo = __ffma2_rn(aa, make_float2(x.x, x.y), make_float2(y.x, y.y));
    const float2 hi = __ffma2_rn(aa, make_float2(x.z, x.w), make_float2(y.z, y.w));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// Sums four per-lane partials over the R lanes of a row group (lanes h*R ..
// h*R+R-1 of the warp) with 2 + log2(R/4) shuffles.  Afterwards the lane holds
// in out[0] the total of value `first` (0: x0, 1: x1, 2: x2, 3: x3) and, for
// R == 2, in out[1] the total of value first + 1.  All 32 lanes must call it.
template <int R>
__device__ __forceinline__ void reduce_scatter4(float x0, float x1, float x2, float x3, int ch, float (&out)[2],
                                                int &first) {
    const bool hb = (ch & (R / 2)) != 0;
    const float s0 = __shfl_xor_sync(0xffffffffu, hb ? x0 : x2, R / 2);
    const float s1 = __shfl_xor_sync(0xffffffffu, hb ? x1 : x3, R / 2);
    const float y0 = (hb ? x2 : x0) + s0, y1 = (hb ? x3 : x1) + s1;
    if constexpr (R == 2) {
        out[0] = y0;
        out[1] = y1;
        first = hb ? 2 : 0;
    } else {
        const bool lb = (ch & (R / 4)) != 0;
        float z = (lb ? y1 : y0) + __shfl_xor_sync(0xffffffffu, lb ? y0 : y1, R / 4);
#pragma unroll
        for (int o = R / 8; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        out[0] = z;
        out[1] = 0.f;
        first = (hb ? 2 : 0) + (lb ? 1 : 0);
    }
}

// ---- grad_value reductions ----------------------------------------------------
__device__ __forceinline__ void red_add_v4(float *p, float4 v) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

__device__ __forceinline__ void red_add_u64(unsigned long long *p, long long v) {
    asm volatile("red.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Fixed-point accumulators of the deterministic backward.  Within each
// (pixel, head) block of D = 4R words the channels are permuted: channel
// 4*ch + i, the i-th of lane ch's four, sits at word i*R + ch.  Each of a
// lane's four 64-bit reductions then covers, over the R lanes of one query,
// R consecutive words, not R words 32 bytes apart (a quarter of the sectors).
// dst: element offset of channel 4*ch of the block, as for the fp32 buffer.
template <int R>
__device__ __forceinline__ void red_fixed4(unsigned long long *fixed, size_t dst, int ch, float4 v, float scale) {
    unsigned long long *p = fixed + (dst - 3 * (size_t)ch);
    red_add_u64(p, __float2ll_rn(v.x * scale));
    red_add_u64(p + R, __float2ll_rn(v.y * scale));
    red_add_u64(p + 2 * R, __float2ll_rn(v.z * scale));
    red_add_u64(p + 3 * R, __float2ll_rn(v.w * scale));
}

// Power-of-two scale of the fixed-point sums: every partial sum is at most
// rows * max_row_bound < 2^62 after scaling (rows: those that can add into one
// accumulator, the rows of one batch element).
__device__ __forceinline__ int fixed_shift(unsigned bits, int rows) {
    const double bound = (double)__uint_as_float(bits) * (double)rows;
    if (!(bound > 0.0)) return 0;
    int e;
    frexp(bound, &e);          // bound < 2^e
    int shift = 62 - e;
    return shift < -60 ? -60 : (shift > 100 ? 100 : shift);
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

// ---- softmax statistics of whole rows -----------------------------------------
// For rows of at most 32 logits every kernel sums exp(logit - max) in one tree,
// pairwise by sample index and zero padded to the next power of two, whichever
// lane layout holds the logits: the record phase of the fused forward (rows
// fastest), that of the fused backward (samples fastest), or the separate pass
// below.  So A is bitwise the same in the fused forward and the fused backward
// whichever path each takes.  Longer rows use a strided warp reduction, the
// same code in both kernels.

// stats[hh] = (max, 1 / sum of exp(logit - max)) of the P logits of row hh,
// rows lg0 + hh * stride for hh < nvalid <= NR (warp-uniform arguments; all
// lanes).  P <= 32: a row takes P2 (P rounded up to a power of two) lanes, a
// pass 32 / P2 rows, and the max and the sum are xor trees over the row's
// lanes.  The logits of up to four passes are loaded before their trees, so a
// warp waits for one round of loads per four passes, not one per pass.
template <int NR>
__device__ __forceinline__ void row_softmax_stats(const float *lg0, size_t stride, int P, int nvalid, int lane,
                                                  float2 *stats) {
    if (P <= 32) {
        constexpr int G = NR < 4 ? NR : 4;
        int P2 = 1;
        while (P2 < P) P2 <<= 1;
        const int per_pass = 32 / P2;
        const int j = lane % P2, hl = lane / P2;
        for (int p0 = 0; p0 * per_pass < nvalid; p0 += G) {
            float x[G];                 // pass p0 + u: row (p0 + u) * per_pass + hl
#pragma unroll
            for (int u = 0; u < G; ++u) {
                const int hh = (p0 + u) * per_pass + hl;
                x[u] = (hh < nvalid && j < P) ? __ldg(lg0 + hh * stride + j) : -INFINITY;
            }
#pragma unroll
            for (int u = 0; u < G; ++u) {
                if ((p0 + u) * per_pass >= nvalid) break;   // warp-uniform
                const int hh = (p0 + u) * per_pass + hl;
                const bool valid = hh < nvalid && j < P;
                float mx = x[u];
                for (int o = 1; o < P2; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float e = valid ? expf(x[u] - mx) : 0.f;
                float sum = e;
                for (int o = 1; o < P2; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                if (j == 0 && hh < nvalid) stats[hh] = make_float2(mx, 1.f / sum);
            }
        }
    } else {
        for (int hh = 0; hh < nvalid; ++hh) {
            const float *lg = lg0 + hh * stride;
            float mx = -INFINITY;
            for (int s = lane; s < P; s += 32) mx = fmaxf(mx, __ldg(lg + s));
            mx = warp_max(mx);
            float sum = 0.f;
            for (int s = lane; s < P; s += 32) sum += expf(__ldg(lg + s) - mx);
            sum = warp_sum(sum);
            if (lane == 0) stats[hh] = make_float2(mx, 1.f / sum);
        }
    }
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

}  // namespace msda
