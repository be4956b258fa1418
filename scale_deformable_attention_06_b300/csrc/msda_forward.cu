// msda_forward.cu -- forward kernels of the MSDeformAttn core.
//
//   out[n][q][m*D+d] = sum_{l,k} A[n,q,m,l,k] * bilinear_l(value[n,:,m,d], loc[n,q,m,l,k])
//
// ("可变形注意力：多尺度稀疏采样与视觉检测实战解析" §2.2 formula, §2.3 bilinear
// sampling, §3.2 steps 4-5; "可变形 DETR：加速收敛的稀疏注意力检测器" §3.3.)
// The fused variant also forms loc = ref + off / (W_l, H_l) ("可变形 DETR…" §6)
// and A = softmax over the L*K logits of the row (the tutorial module, §3.2).
//
// Work decomposition.  A "row" is one (n, q, m).  A warp owns HW = 32 / R
// consecutive rows (head-major order for fp32 rows of a 128-byte line or
// more, query-major otherwise), R lanes per row, each lane holding 16 bytes of the row's
// D channels (4 fp32 or 8 bf16), NV such vectors where a row is wider than 32
// of them (head_dim 256 fp32).  Per chunk of samples:
//   phase 1: each lane computes the corner records (four element offsets and
//            four weights, attention weight folded in) of one or two samples,
//            coalesced over the warp's rows, into warp-private shared memory;
//   phase 2: each lane walks the chunk's samples of its own row and issues four
//            independent 16-byte gathers per sample, accumulating in fp32.
// Every corner fetch is a full 16-byte vector per lane and R lanes cover one
// contiguous D-channel row segment, so a warp-wide gather touches HW value
// rows, each fully used.
#include "msda_device.cuh"
#include "msda_launch.h"

namespace msda {

struct FwdArgs {
    const void *value;
    const float *loc;      // unfused
    const float *attn;     // unfused
    const float *ref;      // fused
    const float *off;      // fused
    const float *logits;   // fused
    void *out;
    Dims d;
    LevelTable lv;
    unsigned char level_of[kMaxSamples];   // level of sample s = l*K + k
    int opts;                              // any option bit set
};

// Query order where the queries are the value pixels.
// In encoder self-attention Len_q == Len_in and query i sits at value pixel i
// of the flattened levels.  The head-major forward then takes the queries of
// one head in band order: each level cut into bands of four rows (the last
// band of a level may be shorter), each band walked column by column.  A
// warp's four consecutive positions are then a column of four pixels and a
// block's 32 an 8 x 4 patch, instead of a 32 x 1 strip, so the value rows a
// block gathers overlap more in L1 (encoder forward 158 -> 152 us).  The order
// only decides which queries run together: it maps [0, Len_in) one to one
// onto itself, for any query layout.  It relies on the levels tiling
// [0, Len_in) exactly (start[l] the running sum of H * W, the sum Len_in,
// every side at least 1), which the host checks before any launch.  The
// backward keeps raster order: there the extra overlap makes concurrent
// grad_value reductions meet on the same lines, and it measured slower
// (405 -> 412 us; 391 -> 399 us with its lean shared memory).
__device__ __forceinline__ int band_query(int p, const LevelTable &lv, int L) {
    int l = 0;
    while (l + 1 < L && p >= lv.start[l + 1]) ++l;
    const int W = lv.W[l], H = lv.H[l];
    const int i = p - lv.start[l];
    const int band = i / (4 * W);
    const int rem = i - band * 4 * W;
    const int bh = min(4, H - 4 * band);            // rows of this band
    const int x = bh == 4 ? rem >> 2 : rem / bh;    // only a level's last band is shorter
    return lv.start[l] + (4 * band + (rem - x * bh)) * W + x;
}

// Resident blocks per SM the fp32 kernels are compiled for: six (at most 40
// registers a thread) up to head width 64, faster on the gathers than five
// (encoder forward 152 -> 145 us, fused 167 -> 158 us) or seven (which
// spills: 166 us); five (48 registers) at width 128, where the fused kernel
// with option code would spill at 40; three at 256.  The unfused bf16 kernel
// is held to the same 40 registers (twelve of its four-warp blocks; decoder
// forward 24.6 -> 22.5 us, large unchanged); the fused bf16 kernel keeps the
// compiler's choice, the 40-register bound made it spill (decoder fused
// forward 24.6 -> 27.2 us).
constexpr int kFwdMinBlocksF32 = 6;
// Warps a forward block: eight for fp32 values, whose band-ordered blocks
// then cover an 8 x 4 patch (four warps measured slower: encoder 143 ->
// 150 us); four for bf16 (large forward 391 -> 387 us, fused 440 -> 432 us).
template <typename T>
constexpr int fwd_warps() { return sizeof(T) == 4 ? kWarpsPerBlock : 4; }
template <int D>
constexpr int fwd_min_blocks_f32() { return D > 128 ? 3 : D == 128 ? 5 : kFwdMinBlocksF32; }
constexpr int kFwdMinBlocksBf16Unfused = 12;     // of four warps: 40 registers

// The kernel body.  OPTS: the problem sets option bits (fused calls); without
// them the kernel carries none of the option code.  SEG: a fused call with
// the whole-row softmax whose rows are one record chunk each (the host checks
// L * K <= JC): the kernel carries only that softmax path, no online one.
template <typename T, int D, bool FUSED, bool OPTS, bool SEG>
__device__ __forceinline__ void forward_body(const FwdArgs &a) {
    using Lay = Layout<T, D>;
    constexpr int V = Lay::V, R = Lay::R, HW = Lay::HW, NV = Lay::NV;
    constexpr int JC = kRecordsPerWarp / HW;     // samples of each row per chunk
    static_assert(!SEG || (FUSED && JC >= 16), "one-chunk rows: fused calls where a chunk holds 16 logits");

    constexpr int WB = fwd_warps<T>();           // warps a block
    __shared__ int4 s_off[WB][kRecordsPerWarp];
    __shared__ float4 s_w[WB][kRecordsPerWarp];
    __shared__ float2 s_stat[WB][HW];               // fused: (row max, 1 / row sum)
    __shared__ int s_row[WB][32];                    // each lane's record-phase row (below)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // fp32 rows of a 128-byte line or more are taken head-major: a warp (and a
    // block) then holds consecutive queries of one head, whose samples share
    // value rows in L1 (encoder forward 164 -> 158 us).  Narrower rows stay
    // query-major, so that a warp's output rows are one contiguous span (64-byte
    // bf16 rows taken head-major measured 19% slower), and so do bf16 rows.
    constexpr bool HEAD_MAJOR = sizeof(T) == 4 && D * (int)sizeof(T) >= 128;
    const int row0 = (blockIdx.x * WB + warp) * HW;                  // in the order above
    // the (n, q, m) row of position vr in that order
    auto row_of = [&](int vr) {
        if constexpr (!HEAD_MAJOR) return vr;
        int q = vr % a.d.Len_q;
        const int t = vr / a.d.Len_q;
        if (a.d.Len_q == a.d.Len_in) q = band_query(q, a.lv, a.d.L);   // queries are the value pixels
        return (t / a.d.M * a.d.Len_q + q) * a.d.M + t % a.d.M;
    };
    const Dims &dm = a.d;
    if (row0 >= dm.rows) return;
    const int P = dm.P;
    // a lane's row in the record and softmax phases: that of position
    // row0 + lane % HW (HW divides 32, so every slot of the lane falls on it),
    // dm.rows or more past the end.  Head-major, it is looked up once; with
    // several rows a warp it is kept in shared memory between chunks (in a
    // register it made the fused kernels spill), with one row a warp it is
    // also the phase-2 row and stays in a register.
    constexpr bool SROW = HEAD_MAJOR && HW > 1;
    int r_mine = row0 + lane % HW;
    if constexpr (HEAD_MAJOR) r_mine = r_mine < dm.rows ? row_of(r_mine) : dm.rows;
    if constexpr (SROW) s_row[warp][lane] = r_mine;
    auto my_row = [&]() -> int {
        if constexpr (SROW) return s_row[warp][lane];
        if constexpr (HEAD_MAJOR) return r_mine;
        return row0 + lane % HW;
    };

    // fused, whole-row softmax.  A row that is one record chunk (the SEG
    // kernels) gets its statistics in the record phase and normalised
    // weights.  A row of several chunks (the other fused kernels) is summed
    // online: each
    // chunk's record phase updates the row's running max and sum and keeps the
    // weights relative to that max, the gather phase first rescales the
    // accumulator by exp(old max - new max), and the output is divided by the
    // sum at the end, so no pass over the logits precedes the gathers.
    const bool row_softmax = FUSED && !(OPTS && a.d.per_level_softmax);
    constexpr bool seg_stats = SEG;
    const bool online = !SEG && row_softmax;
    float run_max = -INFINITY, run_sum = 0.f;      // online: of row lane % HW (phase-1 role)

    // phase-2 lane role
    const int h = lane / R, ch = lane % R;
    const bool row_ok = row0 + h < dm.rows;
    const int row_qm = row0 + h;                    // query-major: the phase-2 row
    // lane h holds the row of position row0 + h (one row a warp: every lane)
    const int rowc = !HEAD_MAJOR ? (row_ok ? row_qm : dm.rows - 1)
                     : HW == 1   ? r_mine
                                 : __shfl_sync(0xffffffffu, r_mine, row_ok ? h : 0);
    const int n = rowc / dm.qm;
    const int m = rowc % dm.M;
    const T *vbase = static_cast<const T *>(a.value) + ((size_t)n * dm.Len_in * dm.M + m) * D + ch * V;
    [[maybe_unused]] const T *vten = static_cast<const T *>(a.value);          // debug build: extent checks
    [[maybe_unused]] const long long vtotal = (long long)dm.N * dm.Len_in * dm.pix;
    const uint64_t pol = l2_keep_policy();

    float acc[NV][V];
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int i = 0; i < V; ++i) acc[k][i] = 0.f;

    // seg_stats: the attention weight of each of this lane's two record slots
    // (slot it = record lane + 32 it, one row: HW divides 32)
    float A_seg[2] = {0.f, 0.f};
    if constexpr (FUSED) {
        if (seg_stats) {                                // warp-uniform; the row is one chunk
            float lg[2];
            bool valid[2];
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const int i = lane + 32 * it, j = i / HW;       // row i % HW = lane % HW
                valid[it] = j < P && my_row() < dm.rows;
                lg[it] = valid[it] ? __ldg(a.logits + (size_t)my_row() * P + j) : -INFINITY;
            }
            float mx = fmaxf(lg[0], lg[1]);
#pragma unroll
            for (int o = HW; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            float e[2], sm[2];
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                e[it] = valid[it] ? expf(lg[it] - mx) : 0.f;
                sm[it] = e[it];
#pragma unroll
                for (int o = HW; o < 32; o <<= 1) sm[it] += __shfl_xor_sync(0xffffffffu, sm[it], o);
            }
            const float inv = 1.f / (sm[0] + sm[1]);
            A_seg[0] = e[0] * inv;
            A_seg[1] = e[1] * inv;
        }
    }

    for (int s0 = 0; s0 < P; s0 += JC) {
        const int J = min(JC, P - s0);
        // online softmax: exp(logit - running max) of this lane's two record
        // slots (slot it = record lane + 32 it, row lane % HW, sample its / HW);
        // the row's lanes are those with the same lane % HW
        float e_slot[2] = {0.f, 0.f};
        if constexpr (FUSED) {
            if (online) {                                   // warp-uniform
                const int r = my_row();                         // >= dm.rows: past the end
                float lg[2];
#pragma unroll
                for (int it = 0; it < 2; ++it) {
                    const int j = (lane + 32 * it) / HW;
                    lg[it] = (j < J && r < dm.rows) ? __ldg(a.logits + (size_t)r * P + s0 + j) : -INFINITY;
                }
                float cm = fmaxf(lg[0], lg[1]);
#pragma unroll
                for (int o = HW; o < 32; o <<= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
                const float m_new = fmaxf(run_max, cm);
                // first chunk: exp(-inf) = 0; a row outside the problem keeps scale 1
                const float scale = m_new == -INFINITY ? 1.f : expf(run_max - m_new);
#pragma unroll
                for (int it = 0; it < 2; ++it) e_slot[it] = lg[it] == -INFINITY ? 0.f : expf(lg[it] - m_new);
                float cs = e_slot[0] + e_slot[1];
#pragma unroll
                for (int o = HW; o < 32; o <<= 1) cs += __shfl_xor_sync(0xffffffffu, cs, o);
                run_sum = __fmaf_rn(run_sum, scale, cs);
                run_max = m_new;
                if (lane < HW) s_stat[warp][lane] = make_float2(scale, run_sum);
            }
        }
        // ---- phase 1: corner records, record i = j * HW + hh
        for (int i = lane; i < HW * J; i += 32) {
            const int j = i / HW, s = s0 + j;                  // row i % HW = lane % HW
            const int r = my_row();                             // >= dm.rows: past the end
            int4 off = make_int4(0, 0, 0, 0);
            float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < dm.rows) {
                const int l = a.level_of[s];
                const float Wf = a.lv.Wf[l], Hf = a.lv.Hf[l];
                float x0, fx, y0, fy, A;
                const size_t si = (size_t)r * P + s;
                if constexpr (FUSED) {
                    const int nq = r / dm.M;            // (n, q) of this row
                    const float2 rf = __ldg(reinterpret_cast<const float2 *>(a.ref) + (size_t)nq * dm.L + l);
                    const float2 of = load_stream2(a.off + 2 * si);
                    float2 st = make_float2(0.f, 1.f);      // per-level groups only
                    if constexpr (OPTS) {
                        pixel_coord_fused(rf.x, of.x, a.lv.Sx[l], a.lv.Rx[l], a.lv.shift, x0, fx);
                        pixel_coord_fused(rf.y, of.y, a.lv.Sy[l], a.lv.Ry[l], a.lv.shift, y0, fy);
                        if (dm.per_level_softmax)       // the level's K logits are this sample's group
                            group_softmax_stats(a.logits + (size_t)r * P + l * dm.K, dm.K, st.x, st.y);
                    } else {
                        pixel_coord_fused(rf.x, of.x, Wf, x0, fx);
                        pixel_coord_fused(rf.y, of.y, Hf, y0, fy);
                    }
                    if (!row_softmax)                   // per-level groups
                        A = expf(load_stream1(a.logits + si) - st.x) * st.y;
                    else if (seg_stats)
                        A = A_seg[(i - lane) >> 5];     // this iteration's slot
                    else
                        A = e_slot[(i - lane) >> 5];    // relative to the running max
                } else {
                    const float2 lc = load_stream2(a.loc + 2 * si);
                    pixel_coord(lc.x, a.lv.Sx[l], a.lv.shift, x0, fx);
                    pixel_coord(lc.y, a.lv.Sy[l], a.lv.shift, y0, fy);
                    A = load_stream1(a.attn + si);
                }
                Corners c = make_corners(x0, fx, y0, fy, a.lv.W[l], a.lv.H[l], Wf, Hf, a.lv.start[l], dm.pix);
                off = c.off;
                w = make_float4(c.w.x * A, c.w.y * A, c.w.z * A, c.w.w * A);
            }
            s_off[warp][i] = off;
            s_w[warp][i] = w;
        }
        __syncwarp();
        // ---- phase 2: gathers of this lane's row
        if constexpr (FUSED) {
            if (online) {                                   // rescale to the row's new running max
                const float sc = s_stat[warp][h].x;
#pragma unroll
                for (int k = 0; k < NV; ++k)
#pragma unroll
                    for (int v = 0; v < V; ++v) acc[k][v] *= sc;
            }
        }
        // samples in flight per lane: eight from head width 32 in the unfused
        // kernels (encoder forward 145 -> 143 us, large 395 -> 389 us; four
        // measured the same as two, eight spills at width 16) and in the fused
        // bf16 ones up to width 128 (no register cap there: large fused forward
        // 432 -> 414 us), two in the fused fp32 ones and at width 256 (four or
        // eight spill there)
#pragma unroll((FUSED && (sizeof(T) == 4 || D > 128)) || D < 32 ? 2 : 8)
        for (int j = 0; j < J; ++j) {
            const int4 o = s_off[warp][j * HW + h];
            const float4 w = s_w[warp][j * HW + h];
#pragma unroll
            for (int k = 0; k < NV; ++k) {         // vector k: channels (k * R + ch) * V ..
                const T *vb = vbase + k * R * V;
                const Vec<T> v0 = load_value(MSDA_ADDR(vten, vb + o.x, vtotal, V), pol);
                const Vec<T> v1 = load_value(MSDA_ADDR(vten, vb + o.y, vtotal, V), pol);
                const Vec<T> v2 = load_value(MSDA_ADDR(vten, vb + o.z, vtotal, V), pol);
                const Vec<T> v3 = load_value(MSDA_ADDR(vten, vb + o.w, vtotal, V), pol);
                fma_row<T, V>(acc[k], w.x, v0);
                fma_row<T, V>(acc[k], w.y, v1);
                fma_row<T, V>(acc[k], w.z, v2);
                fma_row<T, V>(acc[k], w.w, v3);
            }
        }
        __syncwarp();
    }
    if constexpr (FUSED) {
        if (online) {                                       // divide by the row's sum
            const float inv = 1.f / s_stat[warp][h].y;
#pragma unroll
            for (int k = 0; k < NV; ++k)
#pragma unroll
                for (int v = 0; v < V; ++v) acc[k][v] *= inv;
        }
    }
    if (row_ok) {
        // the row again (not held through the gathers): lane h's record-phase
        // row, written before the chunk loop's warp barriers
        const int row = SROW ? s_row[warp][h] : HEAD_MAJOR ? r_mine : row_qm;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            store_row<T, V>(static_cast<T *>(a.out) + (size_t)row * D + (k * R + ch) * V, acc[k]);
    }
}

template <typename T, int D, bool FUSED, bool OPTS, bool SEG>
__global__ void __launch_bounds__(fwd_warps<T>() * 32, fwd_min_blocks_f32<D>())
msda_forward_kernel(const __grid_constant__ FwdArgs a) {       // fp32 value (two vectors a lane at D = 256: three blocks)
    forward_body<T, D, FUSED, OPTS, SEG>(a);
}

template <typename T, int D, bool FUSED, bool OPTS, bool SEG>
__global__ void __launch_bounds__(fwd_warps<T>() * 32)
msda_forward_kernel_bf16(const __grid_constant__ FwdArgs a) {  // bf16 value, fused
    forward_body<T, D, FUSED, OPTS, SEG>(a);
}

template <typename T, int D>
__global__ void __launch_bounds__(fwd_warps<T>() * 32, kFwdMinBlocksBf16Unfused)
msda_forward_kernel_bf16_unfused(const __grid_constant__ FwdArgs a) {  // bf16 value, unfused
    forward_body<T, D, false, false, false>(a);
}

template <typename T, int D, bool OPTS, bool SEG>
static void launch_fwd_fused(const FwdArgs &args, unsigned blocks, cudaStream_t stream) {
    if constexpr (sizeof(T) == 4)
        msda_forward_kernel<T, D, true, OPTS, SEG><<<blocks, fwd_warps<T>() * 32, 0, stream>>>(args);
    else
        msda_forward_kernel_bf16<T, D, true, OPTS, SEG><<<blocks, fwd_warps<T>() * 32, 0, stream>>>(args);
}

template <typename T, int D, bool FUSED>
static cudaError_t launch_fwd(const FwdArgs &args, cudaStream_t stream) {
    constexpr int HW = Layout<T, D>::HW;
    constexpr int JC = kRecordsPerWarp / HW;
    const long long warps = ((long long)args.d.rows + HW - 1) / HW;
    constexpr int WB = fwd_warps<T>();
    const unsigned blocks = (unsigned)((warps + WB - 1) / WB);
    if constexpr (!FUSED) {
        if constexpr (sizeof(T) == 4)
            msda_forward_kernel<T, D, false, false, false><<<blocks, WB * 32, 0, stream>>>(args);
        else
            msda_forward_kernel_bf16_unfused<T, D><<<blocks, WB * 32, 0, stream>>>(args);
    } else {
        const bool opts = args.opts != 0;
        // rows of one record chunk under the whole-row softmax: the one-chunk kernels
        bool seg = false;
        if constexpr (JC >= 16) seg = !(opts && args.d.per_level_softmax) && args.d.P <= JC;
        if constexpr (JC >= 16) {
            if (seg) {
                if (opts) launch_fwd_fused<T, D, true, true>(args, blocks, stream);
                else launch_fwd_fused<T, D, false, true>(args, blocks, stream);
                return cudaGetLastError();
            }
        }
        if (opts) launch_fwd_fused<T, D, true, false>(args, blocks, stream);
        else launch_fwd_fused<T, D, false, false>(args, blocks, stream);
    }
    return cudaGetLastError();
}

template <bool FUSED>
static cudaError_t dispatch_fwd(const FwdArgs &args, int dtype, int D, cudaStream_t stream) {
    if (dtype == 0) {
        switch (D) {
            case 8: return launch_fwd<float, 8, FUSED>(args, stream);
            case 16: return launch_fwd<float, 16, FUSED>(args, stream);
            case 32: return launch_fwd<float, 32, FUSED>(args, stream);
            case 64: return launch_fwd<float, 64, FUSED>(args, stream);
            case 128: return launch_fwd<float, 128, FUSED>(args, stream);
            case 256: return launch_fwd<float, 256, FUSED>(args, stream);
        }
    } else {
        switch (D) {
            case 8: return launch_fwd<__nv_bfloat16, 8, FUSED>(args, stream);
            case 16: return launch_fwd<__nv_bfloat16, 16, FUSED>(args, stream);
            case 32: return launch_fwd<__nv_bfloat16, 32, FUSED>(args, stream);
            case 64: return launch_fwd<__nv_bfloat16, 64, FUSED>(args, stream);
            case 128: return launch_fwd<__nv_bfloat16, 128, FUSED>(args, stream);
            case 256: return launch_fwd<__nv_bfloat16, 256, FUSED>(args, stream);
        }
    }
    return cudaErrorInvalidValue;
}

static void fill_common(FwdArgs &fa, const LaunchGeometry &g) {
    fa.d = g.d;
    fa.lv = g.lv;
    fa.opts = g.d.per_level_softmax || g.lv.shift != 0.5f;
    for (int s = 0; s < kMaxSamples; ++s) fa.level_of[s] = g.level_of[s];
}

#ifdef MSDA_DEBUG
MSDA_DEBUG_COUNTER(debug_count_forward)
#endif

cudaError_t launch_forward(const LaunchGeometry &g, int dtype, int D, const void *value, const float *loc,
                           const float *attn, void *out, cudaStream_t stream) {
    FwdArgs fa{};
    fill_common(fa, g);
    fa.value = value;
    fa.loc = loc;
    fa.attn = attn;
    fa.out = out;
    return dispatch_fwd<false>(fa, dtype, D, stream);
}

cudaError_t launch_forward_fused(const LaunchGeometry &g, int dtype, int D, const void *value, const float *ref,
                                 const float *off, const float *logits, void *out, cudaStream_t stream) {
    FwdArgs fa{};
    fill_common(fa, g);
    fa.value = value;
    fa.ref = ref;
    fa.off = off;
    fa.logits = logits;
    fa.out = out;
    return dispatch_fwd<true>(fa, dtype, D, stream);
}

}  // namespace msda
