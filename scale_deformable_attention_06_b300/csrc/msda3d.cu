// msda3d.cu -- the 3-D (volumetric / temporal) variant of the MSDeformAttn
// core.  "可变形注意力：多尺度稀疏采样与视觉检测实战解析" §5.3: on voxel or video
// features the sampling offsets gain a z (time) component and bilinear
// interpolation becomes trilinear; the rest is the 2-D method.
//
//   out[n][q][m*D+d] = sum_{l,k} A[n,q,m,l,k] * trilinear_l(value[n,:,m,d], loc[n,q,m,l,k])
//
// A level is a volume (Dz_l, H_l, W_l) flattened z-major: value row
// start_l + (z*H_l + y)*W_l + x.  The pixel coordinate is px = x*W - shift
// (likewise y, z; W - 1 and shift 0 with align_corners); the eight integer
// neighbours are weighted u_x(i) u_y(j) u_z(k), u(0) = 1 - f, u(1) = f, and a
// neighbour outside the volume contributes zero.
//
// Forward: the 2-D forward's decomposition (msda_forward.cu): a warp owns HW
// rows (n, q, m), R lanes per row with 16 bytes of channels each; phase 1
// stages one 32-byte corner record per (row, sample); phase 2 issues eight
// 16-byte gathers per sample.  Backward: the 2-D backward's (msda_backward.cu):
// a warp owns HW consecutive queries of one head, 4 channels per lane; per
// sample the lane's partial grad_attn and d/dpx, d/dpy, d/dpz are summed over
// the query's lanes by one reduce-scatter (the fourth slot carries d/dpz), and
// A * w_c * g goes into grad_value by one vector reduction per corner.
#include "msda_device.cuh"
#include "msda_launch.h"

namespace msda {

// ---- 32-byte corner record ----------------------------------------------------
// a.x  value row of corner 000 clamped into the volume (< 2^28)
// a.y  validity bits: 1 x0, 2 x0+1, 4 y0, 8 y0+1, 16 z0, 32 z0+1 inside
// a.z  fx   a.w  fy   b.x  fz   b.y  attention weight
// Corners step from the clamped corner 000 by one column / row / slice only
// when both neighbours along that axis are inside, so every address is
// inside the volume and an inside corner keeps its true address.
struct Rec3 {
    uint4 a, b;
};

__device__ __forceinline__ Rec3 pack_record3(const float (&f0)[3], const float (&fr)[3], float A, int W, int H,
                                             int Dz, float Wf, float Hf, float Dzf, int start) {
    const int x0 = (int)fminf(fmaxf(f0[0], -2.f), Wf + 1.f);
    const int y0 = (int)fminf(fmaxf(f0[1], -2.f), Hf + 1.f);
    const int z0 = (int)fminf(fmaxf(f0[2], -2.f), Dzf + 1.f);
    const uint32_t fl = ((unsigned)x0 < (unsigned)W ? 1u : 0u) | ((unsigned)(x0 + 1) < (unsigned)W ? 2u : 0u) |
                        ((unsigned)y0 < (unsigned)H ? 4u : 0u) | ((unsigned)(y0 + 1) < (unsigned)H ? 8u : 0u) |
                        ((unsigned)z0 < (unsigned)Dz ? 16u : 0u) | ((unsigned)(z0 + 1) < (unsigned)Dz ? 32u : 0u);
    const int cx = min(max(x0, 0), W - 1), cy = min(max(y0, 0), H - 1), cz = min(max(z0, 0), Dz - 1);
    Rec3 r;
    r.a = make_uint4((uint32_t)(start + (cz * H + cy) * W + cx), fl, __float_as_uint(fr[0]), __float_as_uint(fr[1]));
    r.b = make_uint4(__float_as_uint(fr[2]), __float_as_uint(A), 0u, 0u);
    return r;
}

struct Unpacked3 {
    uint32_t pix[8];    // corner c = 4k + 2j + i: (x0+i, y0+j, z0+k), always inside the volume
    float w[8];         // trilinear weights, 0 outside
    bool in[8];
    float f[3], A;
    float u[3][2];      // masked axis factors u_a(0), u_a(1)
};

__device__ __forceinline__ Unpacked3 unpack_record3(const Rec3 &r, int W, int HW) {
    Unpacked3 u;
    const uint32_t fl = r.a.y;
    const uint32_t p = r.a.x;
    const uint32_t dx = ((fl & 3u) == 3u) ? 1u : 0u;
    const uint32_t dy = ((fl & 12u) == 12u) ? (uint32_t)W : 0u;
    const uint32_t dz = ((fl & 48u) == 48u) ? (uint32_t)HW : 0u;
    u.f[0] = __uint_as_float(r.a.z);
    u.f[1] = __uint_as_float(r.a.w);
    u.f[2] = __uint_as_float(r.b.x);
    u.A = __uint_as_float(r.b.y);
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        u.u[a][0] = (fl & (1u << (2 * a))) ? 1.f - u.f[a] : 0.f;
        u.u[a][1] = (fl & (2u << (2 * a))) ? u.f[a] : 0.f;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const int i = c & 1, j = (c >> 1) & 1, k = (c >> 2) & 1;
        u.pix[c] = p + (i ? dx : 0u) + (j ? dy : 0u) + (k ? dz : 0u);
        u.w[c] = u.u[0][i] * u.u[1][j] * u.u[2][k];
        u.in[c] = (fl & (1u << i)) && (fl & (4u << j)) && (fl & (16u << k));
    }
    return u;
}

struct Args3 {
    const void *value;
    const float *loc;      // [N][Len_q][M][L][K][3]
    const float *attn;
    void *out;             // forward
    const void *grad_out;  // backward
    float *grad_value;
    float *grad_loc;
    float *grad_attn;
    unsigned long long *fixed;
    const unsigned *bound_bits;
    Dims d;
    LevelTable3 lv;
    unsigned char level_of[kMaxSamples];
    int qblocks;
};

// corner record of sample s of row r
__device__ __forceinline__ Rec3 record3(const Args3 &a, int r, int s) {
    const int l = a.level_of[s];
    const size_t si = (size_t)r * a.d.P + s;
    const float *lp = a.loc + 3 * si;
    const float S[3] = {a.lv.Sx[l], a.lv.Sy[l], a.lv.Sz[l]};
    float f0[3], fr[3];
#pragma unroll
    for (int c = 0; c < 3; ++c) pixel_coord(load_stream1(lp + c), S[c], a.lv.shift, f0[c], fr[c]);
    return pack_record3(f0, fr, load_stream1(a.attn + si), a.lv.W[l], a.lv.H[l], a.lv.Dz[l], a.lv.Wf[l], a.lv.Hf[l],
                        a.lv.Dzf[l], a.lv.start[l]);
}

// ---- expanded records --------------------------------------------------------
// Phase 1 expands a sample once, for all the lanes of its row: the eight
// corners' element offsets (relative to the row's value head; always inside
// the volume) with the corner's inside bit in bit 0 (offsets are multiples of
// n_heads * head_dim >= 8), and the forward's weights (A folded in) or the
// backward's fractions and A.
struct Exp3 {
    int4 o0, o1;       // offsets | inside bit, corners 0-3 and 4-7
    float4 a, b;       // forward: A*w_c, corners 0-3 and 4-7; backward: (fx, fy, fz, A), unused
};

__device__ __forceinline__ Exp3 expand3(const Rec3 &r, int W, int HW, int pix, bool forward) {
    const Unpacked3 u = unpack_record3(r, W, HW);
    int o[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) o[c] = (int)u.pix[c] * pix | (u.in[c] ? 1 : 0);
    Exp3 e;
    e.o0 = make_int4(o[0], o[1], o[2], o[3]);
    e.o1 = make_int4(o[4], o[5], o[6], o[7]);
    if (forward) {
        e.a = make_float4(u.A * u.w[0], u.A * u.w[1], u.A * u.w[2], u.A * u.w[3]);
        e.b = make_float4(u.A * u.w[4], u.A * u.w[5], u.A * u.w[6], u.A * u.w[7]);
    } else {
        e.a = make_float4(u.f[0], u.f[1], u.f[2], u.A);
        e.b = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return e;
}

// ---- forward ------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
msda3d_forward_kernel(const __grid_constant__ Args3 a) {
    using Lay = Layout<T, D>;
    constexpr int V = Lay::V, R = Lay::R, HW = Lay::HW;
    constexpr int JC = kRecordsPerWarp / HW;
    __shared__ Exp3 s_rec[kWarpsPerBlock][HW][JC + 1];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = (blockIdx.x * kWarpsPerBlock + warp) * HW;
    const Dims &dm = a.d;
    if (row0 >= dm.rows) return;
    const int P = dm.P;
    const int h = lane / R, ch = lane % R;
    const int row = row0 + h;
    const bool row_ok = row < dm.rows;
    const int rowc = row_ok ? row : dm.rows - 1;
    const int n = rowc / dm.qm, m = rowc % dm.M;
    const T *vbase = static_cast<const T *>(a.value) + ((size_t)n * dm.Len_in * dm.M + m) * D + ch * V;
    [[maybe_unused]] const T *vten = static_cast<const T *>(a.value);          // debug build: extent checks
    [[maybe_unused]] const long long vtotal = (long long)dm.N * dm.Len_in * dm.pix;
    const uint64_t pol = l2_keep_policy();

    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;

    for (int s0 = 0; s0 < P; s0 += JC) {
        const int J = min(JC, P - s0);
        for (int i = lane; i < HW * JC; i += 32) {
            const int j = i % JC, hh = i / JC;
            if (j >= J) continue;
            Exp3 e;
            e.o0 = e.o1 = make_int4(0, 0, 0, 0);      // outside every volume: offset 0, weight 0
            e.a = e.b = make_float4(0.f, 0.f, 0.f, 0.f);
            if (row0 + hh < dm.rows) {
                const int l = a.level_of[s0 + j];
                e = expand3(record3(a, row0 + hh, s0 + j), a.lv.W[l], a.lv.H[l] * a.lv.W[l], dm.pix, true);
            }
            s_rec[warp][hh][j] = e;
        }
        __syncwarp();
#pragma unroll 2
        for (int j = 0; j < J; ++j) {
            const Exp3 &e = s_rec[warp][h][j];
            const int4 o0 = e.o0, o1 = e.o1;
            const float4 wa = e.a, wb = e.b;
            const int o[8] = {o0.x & ~1, o0.y & ~1, o0.z & ~1, o0.w & ~1, o1.x & ~1, o1.y & ~1, o1.z & ~1, o1.w & ~1};
            const float wt[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
            Vec<T> v[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) v[c] = load_value(MSDA_ADDR(vten, vbase + o[c], vtotal, V), pol);
#pragma unroll
            for (int c = 0; c < 8; ++c) fma_row<T, V>(acc, wt[c], v[c]);
        }
        __syncwarp();
    }
    if (row_ok) store_row<T, V>(static_cast<T *>(a.out) + (size_t)row * D + ch * V, acc);
}

// ---- backward -----------------------------------------------------------------
// Four warps a block (video backward 500 -> 486 us against eight; the forward
// keeps eight: 205 against 233 us)
constexpr int k3dBwdWarps = 4;

template <typename T, int D, bool DET>
__global__ void __launch_bounds__(k3dBwdWarps * 32, 6)
msda3d_backward_kernel(const __grid_constant__ Args3 a) {
    constexpr int R = D / 4, HW = 32 / R;
    constexpr int RC = kRecordsPerWarp / HW;
    static_assert(HW * RC == 64, "phase 1 and 3 give every lane two (query, sample) slots");
    __shared__ int4 s_o0[k3dBwdWarps][HW][RC + 1];        // corner offsets | inside bit, corners 0-3
    __shared__ int4 s_o1[k3dBwdWarps][HW][RC + 1];        // corners 4-7
    __shared__ float4 s_f[k3dBwdWarps][HW][RC + 1];       // fx, fy, fz, A
    __shared__ float4 s_res[k3dBwdWarps][HW][RC + 1];     // grad_attn, A*d/dpx, A*d/dpy, A*d/dpz

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Dims &dm = a.d;
    const int task = blockIdx.x * k3dBwdWarps + warp;
    if (task >= dm.N * a.qblocks * dm.M) return;       // warp-uniform
    // query blocks fastest: neighbouring warps take neighbouring queries of one
    // head, whose samples share value rows in L1 (video backward 486 -> 473 us
    // against heads fastest)
    const int qb = task % a.qblocks, t2 = task / a.qblocks;
    const int m = t2 % dm.M, n = t2 / dm.M;
    const int P = dm.P;
    const int h = lane / R, ch = lane % R;
    const int q = qb * HW + h;
    const bool row_ok = q < dm.Len_q;
    const int row = (n * dm.Len_q + (row_ok ? q : qb * HW)) * dm.M + m;
    const size_t vhead = ((size_t)n * dm.Len_in * dm.M + m) * D + ch * 4;
    const T *vbase = static_cast<const T *>(a.value) + vhead;
    const uint64_t pol = l2_keep_policy();
    [[maybe_unused]] const T *vten = static_cast<const T *>(a.value);          // debug build: extent checks
    [[maybe_unused]] const T *gten = static_cast<const T *>(a.grad_out);
    [[maybe_unused]] const long long vtotal = (long long)dm.N * dm.Len_in * dm.pix;
    [[maybe_unused]] const long long gtotal = (long long)dm.N * dm.Len_q * dm.pix;

    float4 g = load4_stream<T>(MSDA_ADDR(gten, gten + (size_t)row * D + ch * 4, gtotal, 4));
    if (!row_ok) g = make_float4(0.f, 0.f, 0.f, 0.f);
    float scale = 1.f;
    if constexpr (DET) scale = ldexpf(1.f, fixed_shift(a.bound_bits[n], dm.qm));   // this batch element's scale

    for (int r0 = 0; r0 < P; r0 += RC) {
        const int RJ = min(RC, P - r0);
        // ---- phase 1: corner records
        for (int i = lane; i < HW * RC; i += 32) {
            const int j = i % RC, hh = i / RC;
            if (j >= RJ) continue;
            const int qq = qb * HW + hh;
            Exp3 e;
            e.o0 = e.o1 = make_int4(0, 0, 0, 0);
            e.a = e.b = make_float4(0.f, 0.f, 0.f, 0.f);
            if (qq < dm.Len_q) {
                const int l = a.level_of[r0 + j];
                e = expand3(record3(a, (n * dm.Len_q + qq) * dm.M + m, r0 + j), a.lv.W[l], a.lv.H[l] * a.lv.W[l],
                            dm.pix, false);
            }
            s_o0[warp][hh][j] = e.o0;
            s_o1[warp][hh][j] = e.o1;
            s_f[warp][hh][j] = e.a;
        }
        __syncwarp();
        // ---- phase 2: gather, partial sums, reduce-scatter, grad_value
#pragma unroll 1
        for (int j = 0; j < RJ; ++j) {
            const int4 o0 = s_o0[warp][h][j], o1 = s_o1[warp][h][j];
            const float4 fr = s_f[warp][h][j];
            const int oc[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
            const float f[3] = {fr.x, fr.y, fr.z};
            const float A = fr.w;
            float t[8];
            bool in[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                in[c] = (oc[c] & 1) != 0;
                const float4 v = load4_value(MSDA_ADDR(vten, vbase + (oc[c] & ~1), vtotal, 4), pol);
                float2 pr = __fmul2_rn(make_float2(g.x, g.y), make_float2(v.x, v.y));
                pr = __ffma2_rn(make_float2(g.z, g.w), make_float2(v.z, v.w), pr);
                t[c] = in[c] ? pr.x + pr.y : 0.f;     // outside corners read as zero
            }
            // partial grad_attn and d/dp along each axis (unmasked factors: outside
            // corners have t = 0 and are not scattered)
            float pga = 0.f, pd[3] = {0.f, 0.f, 0.f};
            float w[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int i = c & 1, jj = (c >> 1) & 1, k = (c >> 2) & 1;
                const float ux = i ? f[0] : 1.f - f[0], uy = jj ? f[1] : 1.f - f[1], uz = k ? f[2] : 1.f - f[2];
                w[c] = ux * uy * uz;
                pga = __fmaf_rn(w[c], t[c], pga);
                // d w_c / d f_x = (i ? 1 : -1) u_y(j) u_z(k), and likewise
                pd[0] = __fmaf_rn(i ? uy * uz : -(uy * uz), t[c], pd[0]);
                pd[1] = __fmaf_rn(jj ? ux * uz : -(ux * uz), t[c], pd[1]);
                pd[2] = __fmaf_rn(k ? ux * uy : -(ux * uy), t[c], pd[2]);
            }
            float tot[2];
            int first;
            reduce_scatter4<R>(pga, pd[0], pd[1], pd[2], ch, tot, first);
            if (R <= 4 || (ch & (R / 4 - 1)) == 0) {
                float *rs = reinterpret_cast<float *>(&s_res[warp][h][j]);
                rs[first] = first == 0 ? tot[0] : A * tot[0];
                if (R == 2) rs[first + 1] = A * tot[1];
            }
            if (row_ok) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    if (!in[c]) continue;
                    const float cw = A * w[c];
                    const size_t dst = vhead + (oc[c] & ~1);
                    if constexpr (DET) {
                        if (MSDA_IN(a.fixed, a.fixed + (dst - 3 * (size_t)ch), vtotal, 3 * R + 1))
                            red_fixed4<R>(a.fixed, dst, ch, make_float4(cw * g.x, cw * g.y, cw * g.z, cw * g.w),
                                          scale);
                    } else {
                        if (MSDA_IN(a.grad_value, a.grad_value + dst, vtotal, 4))
                            red_add_v4(a.grad_value + dst, make_float4(cw * g.x, cw * g.y, cw * g.z, cw * g.w));
                    }
                }
            }
            __syncwarp();
        }
        // ---- phase 3: per-sample gradients
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int i = lane + 32 * it;
            const int j = i % RC, hh = i / RC;
            const int qq = qb * HW + hh;
            if (j < RJ && qq < dm.Len_q) {
                const int l = a.level_of[r0 + j];
                const size_t si = ((size_t)(n * dm.Len_q + qq) * dm.M + m) * P + r0 + j;
                const float4 res = s_res[warp][hh][j];
                __stcs(a.grad_attn + si, res.x);
                // d px / d loc = S (size, or size - 1 with align_corners)
                __stcs(a.grad_loc + 3 * si + 0, res.y * a.lv.Sx[l]);
                __stcs(a.grad_loc + 3 * si + 1, res.z * a.lv.Sy[l]);
                __stcs(a.grad_loc + 3 * si + 2, res.w * a.lv.Sz[l]);
            }
        }
        __syncwarp();
    }
}

// ---- launchers ------------------------------------------------------------------
static void fill3(Args3 &a, const LaunchGeometry3 &g) {
    a.d = g.g.d;
    a.lv = g.lv;
    for (int s = 0; s < kMaxSamples; ++s) a.level_of[s] = g.g.level_of[s];
}

template <typename T, int D>
static cudaError_t fwd3_t(const Args3 &a, cudaStream_t stream) {
    constexpr int HW = Layout<T, D>::HW;
    const long long warps = ((long long)a.d.rows + HW - 1) / HW;
    msda3d_forward_kernel<T, D><<<(unsigned)((warps + kWarpsPerBlock - 1) / kWarpsPerBlock), kWarpsPerBlock * 32, 0,
                                  stream>>>(a);
    return cudaGetLastError();
}

#ifdef MSDA_DEBUG
MSDA_DEBUG_COUNTER(debug_count_3d)
#endif

cudaError_t launch_forward3d(const LaunchGeometry3 &g, int dtype, int D, const void *value, const float *loc,
                             const float *attn, void *out, cudaStream_t stream) {
    Args3 a{};
    fill3(a, g);
    a.value = value;
    a.loc = loc;
    a.attn = attn;
    a.out = out;
    if (dtype == 0) {
        switch (D) {
            case 8: return fwd3_t<float, 8>(a, stream);
            case 16: return fwd3_t<float, 16>(a, stream);
            case 32: return fwd3_t<float, 32>(a, stream);
            case 64: return fwd3_t<float, 64>(a, stream);
        }
    } else {
        switch (D) {
            case 8: return fwd3_t<__nv_bfloat16, 8>(a, stream);
            case 16: return fwd3_t<__nv_bfloat16, 16>(a, stream);
            case 32: return fwd3_t<__nv_bfloat16, 32>(a, stream);
            case 64: return fwd3_t<__nv_bfloat16, 64>(a, stream);
        }
    }
    return cudaErrorInvalidValue;
}

template <typename T, int D>
static cudaError_t bwd3_t(Args3 &a, bool det, cudaStream_t stream) {
    constexpr int HW = 32 / (D / 4);
    a.qblocks = (a.d.Len_q + HW - 1) / HW;
    const long long tasks = (long long)a.d.N * a.qblocks * a.d.M;
    const unsigned blocks = (unsigned)((tasks + k3dBwdWarps - 1) / k3dBwdWarps);
    if (det) msda3d_backward_kernel<T, D, true><<<blocks, k3dBwdWarps * 32, 0, stream>>>(a);
    else msda3d_backward_kernel<T, D, false><<<blocks, k3dBwdWarps * 32, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_backward3d(const LaunchGeometry3 &g, int dtype, int D, const void *value, const float *loc,
                              const float *attn, const void *grad_out, float *grad_value, float *grad_loc,
                              float *grad_attn, bool det, bool accumulate, void *workspace, cudaStream_t stream) {
    Args3 a{};
    fill3(a, g);
    a.value = value;
    a.loc = loc;
    a.attn = attn;
    a.grad_out = grad_out;
    a.grad_value = grad_value;
    a.grad_loc = grad_loc;
    a.grad_attn = grad_attn;
    unsigned long long *fixed = nullptr;
    const unsigned *bound = nullptr;
    cudaError_t e = backward_prepare(g.g, dtype, D, attn, 1.f, grad_out, grad_value, det, accumulate, workspace,
                                     &fixed, &bound, stream);
    if (e != cudaSuccess) return e;
    a.fixed = fixed;
    a.bound_bits = bound;
    if (g.g.d.rows > 0) {
        if (dtype == 0) {
            switch (D) {
                case 8: e = bwd3_t<float, 8>(a, det, stream); break;
                case 16: e = bwd3_t<float, 16>(a, det, stream); break;
                case 32: e = bwd3_t<float, 32>(a, det, stream); break;
                case 64: e = bwd3_t<float, 64>(a, det, stream); break;
                default: return cudaErrorInvalidValue;
            }
        } else {
            switch (D) {
                case 8: e = bwd3_t<__nv_bfloat16, 8>(a, det, stream); break;
                case 16: e = bwd3_t<__nv_bfloat16, 16>(a, det, stream); break;
                case 32: e = bwd3_t<__nv_bfloat16, 32>(a, det, stream); break;
                case 64: e = bwd3_t<__nv_bfloat16, 64>(a, det, stream); break;
                default: return cudaErrorInvalidValue;
            }
        }
        if (e != cudaSuccess) return e;
    }
    return backward_finish(g.g, D, grad_value, det, accumulate, fixed, bound, stream);
}

}  // namespace msda
