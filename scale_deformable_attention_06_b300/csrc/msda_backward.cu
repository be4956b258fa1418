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
// Work decomposition.  A warp owns HW consecutive queries of one (n, head m)
// ("head-major"), every lane NV vectors of 4 channels of one of them
// (R = min(D / 4, 32) lanes per query, HW = 32 / R); the warps of a block own
// consecutive query groups of the same head.  Per chunk of up to RC samples:
//   phase 1: one 32-byte corner record per (query, sample) into warp-private
//            shared memory: the four corners' element offsets (clamped inside
//            the map, see pack_record), fx, fy, A and the inside-mask; reads
//            contiguous along the samples;
//   phase 2: per sample, four gathers of the lane's channels; the lane forms
//            its partial <g, v_c> and from them its partial grad_attn, d/dpx,
//            d/dpy (all linear in the dot products), which a reduce-scatter
//            over the R lanes sums with 2 + log2(R/4) shuffles instead of
//            3 * log2(R); then the grad_value contributions A * w_c * g;
//   phase 3: the chunk's per-sample gradients, written contiguously.
// grad_value contributions go out as one vector reduction (red.global.add.v4
// .f32) per corner and lane, or through a per-warp merge table: on densely
// sampled levels of problems of 32 or 64 channels a set the HW = 4 or 2
// queries of a warp are neighbours, so on a coarse level their corners often
// coincide; where a warp holds one query of 128 or 256 channels, that query's
// own samples coincide too, and a merged entry saves a whole row of
// reductions.  The table sums, per distinct corner pixel, one coefficient per
// query, and one reduction per distinct pixel carries sum_h alpha_h * g_h.
// Either way every contribution is added exactly once.
//
// Deterministic mode replaces the fp32 reductions by 64-bit integer ones in
// fixed point (integer addition is associative, so the order in which the
// atomics land does not matter), with a scale chosen from a bound on the total
// |contribution| so that no sum can overflow, then converts to fp32.  The
// merge table's fp32 coefficient sums are formed in a fixed order (program
// order of the samples), so they too are the same from run to run.
#include <type_traits>

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
    const float *ref;              // fused: reference points [N][Len_q][L][2]
    const float *off;              // fused: sampling offsets (pixels of the level)
    const float *logits;           // fused: attention logits [N][Len_q][M][L*K]
    unsigned long long *fixed;     // deterministic: [N*Len_in*M*D] accumulators
    const unsigned *bound_bits;    // deterministic: per batch element, bits of its max row bound (a float)
    Dims d;
    LevelTable lv;
    unsigned char level_of[kMaxSamples];
    int qblocks;                   // ceil(Len_q / HW) query blocks per (n, head)
    unsigned merge_mask;           // bit l: merge grad_value contributions on level l
};

// grad_value[dst .. dst + 4) += v, lane ch of R (fp32 reduction, or fixed point)
template <bool DET, int R>
__device__ __forceinline__ void scatter4(const BwdArgs &a, size_t dst, int ch, float4 v, float scale) {
    [[maybe_unused]] const long long total = (long long)a.d.N * a.d.Len_in * a.d.pix;   // debug build
    if constexpr (DET) {
        // words dst - 3 ch + i R, i < 4: the block's first and last word in range
        if (MSDA_IN(a.fixed, a.fixed + (dst - 3 * (size_t)ch), total, 3 * R + 1))
            red_fixed4<R>(a.fixed, dst, ch, v, scale);
    } else {
        if (MSDA_IN(a.grad_value, a.grad_value + dst, total, 4)) red_add_v4(a.grad_value + dst, v);
    }
}

// Warps a backward block: four.  Smaller blocks balance the SMs better
// (finer blocks to place) and keep fewer concurrent reductions on shared
// lines: encoder backward 392 -> 383 us, large 1.60 -> 1.55 ms, decoder
// 57 -> 51 us, deterministic mode 4-5% faster, against eight.
constexpr int kBwdWarpsPerBlock = 4;

constexpr unsigned kEmptyKey = 0xffffffffu;
// Merge-table slots per warp; a merge chunk has at most 64 entries (16 with
// one query a warp).  fp32 mode merges the coarse levels (a quarter or less
// of a chunk's entries distinct), every level only with one query a warp:
// 64 slots, whose smaller footprint leaves the SM more L1 (encoder backward
// 405 -> 392 us).  Deterministic mode merges every level, up to three
// quarters distinct on the finest: 128 slots keep its probe chains short (64
// measured 1-2% slower there).
template <bool DET>
constexpr int merge_slots() { return DET ? 128 : 64; }
constexpr int kMergeSamples = 4;       // samples per merge chunk (4 queries x 4 x 4 corners = 64 entries)

// Warp-private shared memory.  The fused calls' arrays have one element in
// the unfused kernels, the per-level softmax's in kernels without option code
// (never read there), and the merge table exists only where it is compiled
// in: less shared memory a block leaves the SM more L1.
template <int HW, int RC, bool FUSED, bool OPTS>
struct BwdWarpSmem {
    int4 roff[HW][RC + 1];             // corner records: element offsets of the 4 corners (padded rows)
    float4 raux[HW][RC + 1];           //   fx, fy, A, inside-mask bits
    float4 res[HW][RC + 1];            // per sample: grad_attn, A*d/dpx, A*d/dpy
    float2 stat[FUSED ? HW : 1];       // fused: softmax max and 1 / sum of each query
    float gdot[FUSED && OPTS ? HW : 1][FUSED && OPTS ? kMaxLevels : 1];   // per-level softmax: sum_k A_k grad_A_k
    float dotp[FUSED ? 64 : 1];        // fused: per (query, sample) slot, sum of A * grad_A
};

template <int HW, int RC, bool FUSED, bool OPTS, int SLOTS>
struct BwdWarpSmemMerge {
    int4 roff[HW][RC + 1];
    float4 raux[HW][RC + 1];
    float4 res[HW][RC + 1];
    float2 stat[FUSED ? HW : 1];
    float gdot[FUSED && OPTS ? HW : 1][FUSED && OPTS ? kMaxLevels : 1];
    float dotp[FUSED ? 64 : 1];
    unsigned key[SLOTS];               // corner pixel of the slot, kEmptyKey if free
    std::conditional_t<HW == 4, float4, std::conditional_t<HW == 2, float2, float>> alpha[SLOTS];   // per query of the warp: summed A * w_c
    unsigned short list[SLOTS];        // occupied slots in order of first use
    int count;
};

// Lanes of the backward for head_dim D: R lanes a query, 4 channels a vector,
// NV vectors a lane (vector k of lane ch: channels 4 * (k * R + ch) ..), HW
// queries a warp.
template <int D>
struct BwdLanes {
    static constexpr int R = D / 4 < 32 ? D / 4 : 32;
    static constexpr int NV = D / (4 * R);
    static constexpr int HW = 32 / R;
};

// OPTS: the problem sets option bits (fused calls); without them the kernel
// carries none of the option code.  Launch bounds: eight blocks of four warps
// per SM up to head width 64 in deterministic mode and in the fused calls
// (64 registers; fused kernels at 66-67 fell to seven blocks: large fused
// backward 1.73 -> 1.70 ms, decoder 64 -> 62 us with the cap), except the
// fp32 fused kernels with the merge table, and six otherwise (85: these use
// 62-64, so eight fit, and the cap made them slower: encoder fused backward
// 429 -> 436 us, unfused 383 -> 403 us; head widths above 64 need the
// registers for two vectors a lane).
template <typename T, int D, bool DET, bool MERGE, bool FUSED, bool OPTS>
__global__ void __launch_bounds__(kBwdWarpsPerBlock * 32,
                                  (D <= 64 && (DET || (FUSED && (sizeof(T) == 2 || !MERGE)))) ? 8 : 6)
msda_backward_kernel(const __grid_constant__ BwdArgs a) {
    constexpr int R = BwdLanes<D>::R, HW = BwdLanes<D>::HW, NV = BwdLanes<D>::NV;
    constexpr int RC = kRecordsPerWarp / HW;      // samples per record chunk
    static_assert(HW * RC == 64, "phase 1 and 3 give every lane two (query, sample) slots");
    static_assert(!MERGE || HW == 4 || HW == 2 || HW == 1, "the merge table holds four, two or one queries a slot");
    static_assert(!MERGE || HW == 1 || NV == 1, "several queries a warp: one vector a lane");
    constexpr int kMergeSlots = merge_slots<DET>();
    using WS = std::conditional_t<MERGE, BwdWarpSmemMerge<HW, RC, FUSED, OPTS, kMergeSlots>,
                                  BwdWarpSmem<HW, RC, FUSED, OPTS>>;
    __shared__ WS smem[kBwdWarpsPerBlock];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WS &sm = smem[warp];
    const Dims &dm = a.d;
    // query blocks fastest: the warps of a block (and blocks launched together)
    // take consecutive queries of one head, whose samples share value rows
    const int task = blockIdx.x * kBwdWarpsPerBlock + warp;
    if (task >= dm.N * a.qblocks * dm.M) return;       // warp-uniform
    const int qb = task % a.qblocks, t2 = task / a.qblocks;
    const int m = t2 % dm.M, n = t2 / dm.M;
    const int P = dm.P;
    const int h = lane / R, ch = lane % R;
    const int q = qb * HW + h;
    const bool row_ok = q < dm.Len_q;
    const int row = (n * dm.Len_q + (row_ok ? q : qb * HW)) * dm.M + m;
    const size_t vhead = ((size_t)n * dm.Len_in * dm.M + m) * D + ch * 4;   // (n, pixel 0, m, lane channels)
    const T *vbase = static_cast<const T *>(a.value) + vhead;
    const uint64_t pol = l2_keep_policy();
    [[maybe_unused]] const T *vten = static_cast<const T *>(a.value);          // debug build: extent checks
    [[maybe_unused]] const T *gten = static_cast<const T *>(a.grad_out);
    [[maybe_unused]] const long long vtotal = (long long)dm.N * dm.Len_in * dm.pix;
    [[maybe_unused]] const long long gtotal = (long long)dm.N * dm.Len_q * dm.pix;

    float4 gv[NV];                               // this lane's channels of grad_output
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        gv[k] = load4_stream<T>(MSDA_ADDR(gten, gten + (size_t)row * D + (k * R + ch) * 4, gtotal, 4));
        if (!row_ok) gv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float4 &g = gv[0];
    float scale = 1.f;
    if constexpr (DET) scale = ldexpf(1.f, fixed_shift(a.bound_bits[n], dm.qm));   // this batch element's scale

    if constexpr (MERGE) {
        for (int i = lane; i < kMergeSlots; i += 32) {
            sm.key[i] = kEmptyKey;
            sm.alpha[i] = {};
        }
        if (lane == 0) sm.count = 0;
        __syncwarp();
    }
    // fused, whole-row softmax: statistics in the record phase when the row is
    // one record chunk (compiled in where a chunk holds 16 logits), else in a
    // pass of their own before the records, since every sample's gradient
    // needs its normalised weight
    const bool row_softmax = FUSED && !(OPTS && dm.per_level_softmax);
    const bool seg_stats = (RC >= 16 && RC <= 32) && row_softmax && P <= RC;
    if (row_softmax && !seg_stats) {
        row_softmax_stats<HW>(a.logits + ((size_t)(n * dm.Len_q + qb * HW) * dm.M + m) * P, (size_t)dm.M * P, P,
                          min(HW, dm.Len_q - qb * HW), lane, sm.stat);
        __syncwarp();
    }
    // fused: slot it of lane i is query (lane + 32 it) / RC, sample its
    // remainder (a query's samples are RC consecutive slots); each lane alone
    // reads and writes its two slots' partial sums of A * grad_A
    if constexpr (FUSED) {
        sm.dotp[lane] = 0.f;
        sm.dotp[lane + 32] = 0.f;
    }

    for (int r0 = 0; r0 < P; r0 += RC) {
        const int RJ = min(RC, P - r0);
        // ---- phase 1: corner records of samples r0 .. r0 + RJ
        for (int i = lane; i < HW * RC; i += 32) {    // two iterations on every lane
            const int j = i % RC, hh = i / RC;
            float A_slot = 0.f;
            if constexpr (FUSED) {
                if (seg_stats) {    // warp-uniform: the row is this one chunk; its softmax, a slot per lane
                    const int qq = qb * HW + hh;
                    const bool valid = j < P && qq < dm.Len_q;
                    const float lg = valid ? __ldg(a.logits + ((size_t)(n * dm.Len_q + qq) * dm.M + m) * P + j)
                                           : -INFINITY;
                    float mx = lg;
#pragma unroll
                    for (int o = 1; o < RC && o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    const float e = valid ? expf(lg - mx) : 0.f;
                    float sum = e;
#pragma unroll
                    for (int o = 1; o < RC && o < 32; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                    A_slot = e * (1.f / sum);
                }
            }
            if (j >= RJ) continue;
            const int qq = qb * HW + hh;
            int4 ro = make_int4(0, 0, 0, 0);                   // outside every map: offset 0, mask 0
            float4 ra = make_float4(0.f, 0.f, 0.f, 0.f);
            if (qq < dm.Len_q) {
                const int l = a.level_of[r0 + j];
                const float Wf = a.lv.Wf[l], Hf = a.lv.Hf[l];
                const size_t si = ((size_t)(n * dm.Len_q + qq) * dm.M + m) * P + r0 + j;
                float x0, fx, y0, fy, A;
                if constexpr (FUSED) {
                    const float2 rf = __ldg(reinterpret_cast<const float2 *>(a.ref) + (size_t)(n * dm.Len_q + qq) * dm.L + l);
                    const float2 of = load_stream2(a.off + 2 * si);
                    if constexpr (OPTS) {
                        pixel_coord_fused(rf.x, of.x, a.lv.Sx[l], a.lv.Rx[l], a.lv.shift, x0, fx);
                        pixel_coord_fused(rf.y, of.y, a.lv.Sy[l], a.lv.Ry[l], a.lv.shift, y0, fy);
                    } else {
                        pixel_coord_fused(rf.x, of.x, Wf, x0, fx);
                        pixel_coord_fused(rf.y, of.y, Hf, y0, fy);
                    }
                    if (seg_stats) {
                        A = A_slot;
                    } else {
                        float2 st;
                        if (OPTS && dm.per_level_softmax)
                            group_softmax_stats(a.logits + (si - (r0 + j)) + l * dm.K, dm.K, st.x, st.y);
                        else
                            st = sm.stat[hh];
                        A = expf(load_stream1(a.logits + si) - st.x) * st.y;
                    }
                } else {
                    const float2 lc = load_stream2(a.loc + 2 * si);
                    pixel_coord(lc.x, a.lv.Sx[l], a.lv.shift, x0, fx);
                    pixel_coord(lc.y, a.lv.Sy[l], a.lv.shift, y0, fy);
                    A = load_stream1(a.attn + si);
                }
                // four element offsets (relative to this lane group's value head),
                // always inside the map, and the inside-mask; computed once here
                // instead of by every lane of the query in phase 2
                const uint4 pk = pack_record(x0, fx, y0, fy, A, a.lv.W[l], a.lv.H[l], Wf, Hf, a.lv.start[l]);
                const Unpacked u = unpack_record(pk, a.lv.W[l]);
                ro = make_int4((int)u.pix[0] * dm.pix, (int)u.pix[1] * dm.pix, (int)u.pix[2] * dm.pix,
                               (int)u.pix[3] * dm.pix);
                const unsigned mask = (u.in[0] ? 1u : 0u) | (u.in[1] ? 2u : 0u) | (u.in[2] ? 4u : 0u) | (u.in[3] ? 8u : 0u);
                ra = make_float4(fx, fy, A, __uint_as_float(mask));
            }
            sm.roff[hh][j] = ro;
            sm.raux[hh][j] = ra;
        }
        __syncwarp();
        // ---- phase 2, one level (or merge chunk) at a time
        for (int s0 = r0; s0 < r0 + RJ;) {
            const int l = a.level_of[s0];
            const bool merge = MERGE && ((a.merge_mask >> l) & 1u);
            int J = r0 + RJ - s0;
            if (merge && J > kMergeSamples) J = kMergeSamples;
            for (int jj = 1; jj < J; ++jj)
                if (a.level_of[s0 + jj] != l) { J = jj; break; }
            // one sample at a time: unrolled by two (no spills at 64 registers)
            // it measured 4% slower
#pragma unroll 1
            for (int j = s0 - r0; j < s0 - r0 + J; ++j) {
                const int4 ro = sm.roff[h][j];
                const float4 ra = sm.raux[h][j];
                const int off[4] = {ro.x, ro.y, ro.z, ro.w};
                const float fx = ra.x, fy = ra.y, A = ra.z;
                const unsigned mask = __float_as_uint(ra.w);
                const bool in[4] = {(mask & 1u) != 0, (mask & 2u) != 0, (mask & 4u) != 0, (mask & 8u) != 0};
                // bilinear weights; an outside corner's weight is never used (its
                // dot product is zeroed and it is not scattered)
                const float w[4] = {(1.f - fx) * (1.f - fy), fx * (1.f - fy), (1.f - fx) * fy, fx * fy};
                // partial <g, v_c> over this lane's channels (two packed products
                // per corner and vector); corners outside the map read as zero
                float t[4];
                {
                    float2 pr[4];
#pragma unroll
                    for (int k = 0; k < NV; ++k) {
                        float4 v[4];
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            v[c] = load4_value(MSDA_ADDR(vten, vbase + off[c] + k * 4 * R, vtotal, 4), pol);
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            pr[c] = k == 0 ? __fmul2_rn(make_float2(gv[k].x, gv[k].y), make_float2(v[c].x, v[c].y))
                                           : __ffma2_rn(make_float2(gv[k].x, gv[k].y), make_float2(v[c].x, v[c].y),
                                                        pr[c]);
                            pr[c] = __ffma2_rn(make_float2(gv[k].z, gv[k].w), make_float2(v[c].z, v[c].w), pr[c]);
                        }
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) t[c] = in[c] ? pr[c].x + pr[c].y : 0.f;
                }
                // partial grad_attn, d/dpx, d/dpy
                const float pga = w[0] * t[0] + w[1] * t[1] + w[2] * t[2] + w[3] * t[3];
                const float pdx = (1.f - fy) * (t[1] - t[0]) + fy * (t[3] - t[2]);
                const float pdy = (1.f - fx) * (t[2] - t[0]) + fx * (t[3] - t[1]);
                float tot[2];
                int first;
                reduce_scatter4<R>(pga, pdx, pdy, 0.f, ch, tot, first);
                if (R <= 4 || (ch & (R / 4 - 1)) == 0) {
                    float *rs = reinterpret_cast<float *>(&sm.res[h][j]);
                    if (first < 3) rs[first] = first == 0 ? tot[0] : A * tot[0];
                    if (R == 2 && first == 0) rs[1] = A * tot[1];
                }
                if (row_ok) {
                    if (!merge) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            if (!in[c]) continue;
                            const float cw = A * w[c];
#pragma unroll
                            for (int k = 0; k < NV; ++k) {
                                const float2 lo = __fmul2_rn(make_float2(cw, cw), make_float2(gv[k].x, gv[k].y));
                                const float2 hi = __fmul2_rn(make_float2(cw, cw), make_float2(gv[k].z, gv[k].w));
                                scatter4<DET, R>(a, vhead + off[c] + k * 4 * R, ch, make_float4(lo.x, lo.y, hi.x, hi.y),
                                                 scale);
                            }
                        }
                    } else if constexpr (MERGE) {
                        // lanes ch < 4 insert corner c = ch of their query; the valid
                        // corners of one sample are distinct pixels, so no two lanes of
                        // one step touch the same (slot, query) coefficient
                        if (ch < 4) {
                            const int c = ch;
                            const bool inside = (mask >> c) & 1u;
                            if (inside) {
                                // the corner's element offset is the key (< 2^31, never kEmptyKey)
                                const unsigned key = (unsigned)(c == 0 ? off[0] : c == 1 ? off[1] : c == 2 ? off[2] : off[3]);
                                const float coef = A * (c == 0 ? w[0] : c == 1 ? w[1] : c == 2 ? w[2] : w[3]);
                                // at most 64 keys per chunk in 64 or 128 slots: a probe of
                                // every slot finds a free or matching one
                                // offsets are multiples of n_heads * head_dim: hash, do not mask
                                static_assert((kMergeSlots == 64 || kMergeSlots == 128) &&
                                                  kMergeSamples * 4 * 4 <= kMergeSlots,
                                              "the hash below yields log2(slots) bits; a chunk's entries fit");
                                unsigned slot = (key * 2654435761u) >> (kMergeSlots == 64 ? 26 : 25);
                                for (int probe = 0; probe < kMergeSlots; ++probe) {
                                    const unsigned old = atomicCAS(&sm.key[slot], kEmptyKey, key);
                                    if (old == kEmptyKey) sm.list[atomicAdd(&sm.count, 1)] = (unsigned short)slot;
                                    if (old == kEmptyKey || old == key) {
                                        reinterpret_cast<float *>(&sm.alpha[slot])[h] += coef;
                                        break;
                                    }
                                    slot = (slot + 1) & (kMergeSlots - 1);
                                }
                            }
                        }
                    }
                }
                __syncwarp();
            }
            if constexpr (MERGE) {
                if (merge) {
                    // one reduction per distinct corner pixel and lane: sum_h alpha_h * g_h
                    const int U = sm.count;
                    if constexpr (HW > 1) {
                        // this lane's channels of grad_output of each of the warp's queries,
                        // reloaded here rather than held in registers through the sample loop
                        float4 gq[HW];
#pragma unroll
                        for (int hh = 0; hh < HW; ++hh) {
                            const int qq = qb * HW + hh;
                            gq[hh] = qq < dm.Len_q
                                         ? load4_value<T>(MSDA_ADDR(gten, gten + ((size_t)(n * dm.Len_q + qq) * dm.M + m) *
                                                                              D + ch * 4, gtotal, 4),
                                                          pol)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                        for (int u0 = 0; u0 < U; u0 += HW) {
                            const int ui = u0 + h;
                            if (ui < U) {
                                const int slot = sm.list[ui];
                                const auto al = sm.alpha[slot];
                                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                                acc = ffma4(al.x, gq[0], acc);
                                acc = ffma4(al.y, gq[1], acc);
                                if constexpr (HW == 4) {
                                    acc = ffma4(al.z, gq[2], acc);
                                    acc = ffma4(al.w, gq[3], acc);
                                }
                                scatter4<DET, R>(a, vhead + sm.key[slot], ch, acc, scale);
                            }
                        }
                    } else {
                        // one query a warp: every lane takes every distinct pixel, its
                        // NV vectors of the query's grad_output already in registers
                        for (int ui = 0; ui < U; ++ui) {
                            const int slot = sm.list[ui];
                            const float al = sm.alpha[slot];
                            const size_t base = vhead + sm.key[slot];
#pragma unroll
                            for (int k = 0; k < NV; ++k)
                                scatter4<DET, R>(a, base + k * 4 * R, ch, ffma4(al, gv[k], make_float4(0.f, 0.f, 0.f, 0.f)),
                                                 scale);
                        }
                    }
                    __syncwarp();
                    for (int ui = lane; ui < U; ui += 32) {
                        const int slot = sm.list[ui];
                        sm.key[slot] = kEmptyKey;
                        sm.alpha[slot] = {};
                    }
                    if (lane == 0) sm.count = 0;
                    __syncwarp();
                }
            }
            s0 += J;
        }
        // ---- phase 3: per-sample gradients of the chunk
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int i = lane + 32 * it;
            const int j = i % RC, hh = i / RC;
            const int qq = qb * HW + hh;
            if (j < RJ && qq < dm.Len_q) {
                const int l = a.level_of[r0 + j];
                const size_t si = ((size_t)(n * dm.Len_q + qq) * dm.M + m) * P + r0 + j;
                const float4 res = sm.res[hh][j];
                if constexpr (FUSED) {
                    // offsets are pixels of the level: d px / d off = S / W = Rx
                    if constexpr (OPTS)
                        __stcs(reinterpret_cast<float2 *>(a.grad_loc) + si,
                               make_float2(res.y * a.lv.Rx[l], res.z * a.lv.Ry[l]));
                    else
                        __stcs(reinterpret_cast<float2 *>(a.grad_loc) + si, make_float2(res.y, res.z));
                    // one chunk (seg_stats): A and grad_A stay in raux and res for the
                    // closing pass; else grad_A goes to grad_attn, read back below by
                    // this lane, and the slot's A * grad_A to its partial sum
                    if (!seg_stats) {
                        a.grad_attn[si] = res.x;
                        sm.dotp[i] = __fmaf_rn(sm.raux[hh][j].z, res.x, sm.dotp[i]);
                    }
                } else {
                    __stcs(a.grad_attn + si, res.x);
                    // d px / d loc = S (W, or W - 1 with align_corners)
                    __stcs(reinterpret_cast<float2 *>(a.grad_loc) + si,
                           make_float2(res.y * a.lv.Sx[l], res.z * a.lv.Sy[l]));
                }
            }
        }
        __syncwarp();
    }
    if constexpr (FUSED) {
        // softmax backward: grad_logit_s = A_s * (grad_A_s - sum_t A_t grad_A_t).
        // Slot it of lane i covers query (lane + 32 it) / RC; the lanes of one
        // query form an aligned group of min(RC, 32), summed in a fixed order.
        constexpr int G = RC < 32 ? RC : 32;
        if (seg_stats) {
            // one chunk: A and grad_A of every sample are still in raux and res
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const int i = lane + 32 * it;
                const int j = i % RC, hh = i / RC;
                const int qq = qb * HW + hh;
                const bool ok = j < P && qq < dm.Len_q;
                const float A = ok ? sm.raux[hh][j].z : 0.f, gA = ok ? sm.res[hh][j].x : 0.f;
                float v = __fmaf_rn(A, gA, 0.f);
#pragma unroll
                for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (ok)
                    __stcs(a.grad_attn + ((size_t)(n * dm.Len_q + qq) * dm.M + m) * P + j, A * (gA - v));
            }
            return;
        }
        float tot[2];
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            float v = sm.dotp[lane + 32 * it];
#pragma unroll
            for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            tot[it] = v;
        }
        if constexpr (RC > 32) {          // one query a warp: both of a lane's slots are its samples
            tot[0] += tot[1];
            tot[1] = tot[0];
        }
        if (OPTS && dm.per_level_softmax) {
            // groups are the levels.  Their K grad_A were written by several
            // lanes (and a level may straddle two record chunks), so first every
            // (query, level) dot sum_k A_k grad_A_k, one lane each in a fixed
            // order, while all grad_A are still in place.
            __syncwarp();
            for (int u = lane; u < HW * dm.L; u += 32) {
                const int hh = u / dm.L, l = u % dm.L;
                const int qq = qb * HW + hh;
                float dot = 0.f;
                if (qq < dm.Len_q) {
                    const size_t g0 = ((size_t)(n * dm.Len_q + qq) * dm.M + m) * P + (size_t)l * dm.K;
                    float mx, inv;
                    group_softmax_stats(a.logits + g0, dm.K, mx, inv);
                    for (int k = 0; k < dm.K; ++k)
                        dot = __fmaf_rn(expf(__ldg(a.logits + g0 + k) - mx) * inv, __ldcg(a.grad_attn + g0 + k), dot);
                }
                sm.gdot[hh][l] = dot;
            }
            __syncwarp();
        }
        // grad_logit = A * (grad_A - dot); each lane rewrites only the samples it wrote
        for (int r0 = 0; r0 < P; r0 += RC) {
            const int RJ = min(RC, P - r0);
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const int i = lane + 32 * it;
                const int j = i % RC, hh = i / RC;
                const int qq = qb * HW + hh;
                if (j < RJ && qq < dm.Len_q) {
                    const size_t si = ((size_t)(n * dm.Len_q + qq) * dm.M + m) * P + r0 + j;
                    float A, dot;
                    if (OPTS && dm.per_level_softmax) {
                        const int l = a.level_of[r0 + j];
                        float mx, inv;
                        group_softmax_stats(a.logits + (si - (r0 + j)) + (size_t)l * dm.K, dm.K, mx, inv);
                        A = expf(__ldg(a.logits + si) - mx) * inv;
                        dot = sm.gdot[hh][l];
                    } else {
                        const float2 st = sm.stat[hh];
                        A = expf(__ldg(a.logits + si) - st.x) * st.y;
                        dot = tot[it];
                    }
                    // own write: the plain load sees it (per-level groups read L2 above)
                    __stcs(a.grad_attn + si, A * (a.grad_attn[si] - dot));
                }
            }
        }
    }
}

#ifdef MSDA_DEBUG
MSDA_DEBUG_COUNTER(debug_count_backward)
#endif

// grad_reference_points[n][q][l] = sum over heads and points of the location
// gradient = (W_l, H_l) * sum of the offset gradients (loc = ref + off / (W, H)).
// One thread per (n, q, l), summed in a fixed order.
__global__ void ref_grad_kernel(const float *grad_off, float *grad_ref, int nql, int M, int L, int K, LevelTable lv) {
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < nql; t += gridDim.x * blockDim.x) {
        const int l = t % L, nq = t / L;
        float sx = 0.f, sy = 0.f;
        for (int m = 0; m < M; ++m) {
            const float2 *g = reinterpret_cast<const float2 *>(grad_off) + (((size_t)nq * M + m) * L + l) * K;
            for (int k = 0; k < K; ++k) {
                const float2 v = g[k];
                sx += v.x;
                sy += v.y;
            }
        }
        reinterpret_cast<float2 *>(grad_ref)[t] = make_float2(sx * lv.Wf[l], sy * lv.Hf[l]);
    }
}

// The same sums for small problems where n_heads * n_levels divides 32: one
// thread per (n, q, m, l) in memory order reads its K offset gradients (K * 8
// contiguous bytes, so a warp reads whole rows), and an xor tree over the
// lanes of the heads (lane bits log2(L) and up, a fixed order) sums the
// heads; the thread of head 0 writes.  M times the threads of the kernel
// above: decoder fused backward 61.6 -> 57.5 us; on the encoder and larger
// problems the kernel above is as fast or faster (428.6 against 430.5 us).
__global__ void ref_grad_kernel_rows(const float *grad_off, float *grad_ref, int nqml, int M, int L, int K,
                                     LevelTable lv) {
    const int lane = threadIdx.x & 31;
    for (int t0 = blockIdx.x * blockDim.x; t0 < nqml; t0 += gridDim.x * blockDim.x) {
        const int t = t0 + (threadIdx.x & ~31) + lane;                 // whole warps in range together
        const bool ok = t < nqml;
        const int l = t % L, m = (t / L) % M, nq = t / (L * M);
        float sx = 0.f, sy = 0.f;
        if (ok) {
            const float2 *g = reinterpret_cast<const float2 *>(grad_off) + (size_t)t * K;   // ((nq*M + m)*L + l)*K
            for (int k = 0; k < K; ++k) {
                const float2 v = g[k];
                sx += v.x;
                sy += v.y;
            }
        }
        for (int o = L; o < L * M; o <<= 1) {           // the heads' lanes: bits log2(L) .. log2(L*M)-1
            sx += __shfl_xor_sync(0xffffffffu, sx, o);
            sy += __shfl_xor_sync(0xffffffffu, sy, o);
        }
        if (ok && m == 0)
            reinterpret_cast<float2 *>(grad_ref)[(size_t)nq * L + l] = make_float2(sx * lv.Wf[l], sy * lv.Hf[l]);
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

// Bound of batch element n's fixed-point sums: max over its rows of
// (sum_s |A_s|) * (max_d |g_d|), as float bits in bound_bits[n] (non-negative
// floats order like their bit patterns, so an integer max is exact and
// independent of the order of the atomics).  Every grad_value element of batch
// element n sums at most rows_per_batch such row totals (bilinear weights lie in
// [0, 1] and sum to at most 1).  attn == nullptr (fused calls): the weights of
// a row are softmax outputs summing to row_sum (1, or n_levels with the
// per-level softmax).  Blocks (x, y): y walks the batch elements.
template <typename T, int D>
__global__ void row_bound_kernel(const float *attn, const T *grad_out, int N, int rows_per_batch, int P,
                                 float row_sum, unsigned *bound_bits) {
    __shared__ float s_max[32];
    for (int n = blockIdx.y; n < N; n += gridDim.y) {
        float best = 0.f;
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < rows_per_batch; i += gridDim.x * blockDim.x) {
            const size_t r = (size_t)n * rows_per_batch + i;
            float sa = row_sum * 1.001f;
            if (attn) {
                sa = 0.f;
                for (int s = 0; s < P; ++s) sa += fabsf(attn[r * P + s]);
            }
            float gm = 0.f;
            const T *g = grad_out + r * D;
            for (int d = 0; d < D; ++d) gm = fmaxf(gm, fabsf((float)g[d]));
            // round the product up a little so the bound stays an upper bound
            best = fmaxf(best, sa * gm * 1.0001f);
        }
        best = warp_max(best);
        if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = best;
        __syncthreads();
        if (threadIdx.x < 32) {
            float v = threadIdx.x < (blockDim.x >> 5) ? s_max[threadIdx.x] : 0.f;
            v = warp_max(v);
            if (threadIdx.x == 0) atomicMax(bound_bits + n, __float_as_uint(v));
        }
        __syncthreads();
    }
}

// grad_value = fixed * 2^-shift_n, batch element n's own scale, undoing the
// channel permutation of each block of D = 4R words (red_fixed4): thread t
// writes the 4 channels of lane ch = t mod R of its block, words ch, R + ch,
// 2R + ch, 3R + ch (consecutive threads read consecutive words).  The sums are
// below 2^62 and shift lies in [-60, 100], so the scaled value is a normal
// float: one rounding, in the int64 -> fp32 conversion; the power-of-two
// scaling is exact.  Blocks (x, y): y walks the batch elements.
__global__ void fixed_to_f32_kernel(const unsigned long long *fixed, const unsigned *bound_bits, int N,
                                    int rows_per_batch, float4 *grad_value, size_t n4_per_batch, int D,
                                    int accumulate) {
    const size_t R = (size_t)((D >> 2) < 32 ? (D >> 2) : 32);    // lanes of a query: blocks of 4R words
    for (int n = blockIdx.y; n < N; n += gridDim.y) {
        const int shift = fixed_shift(bound_bits[n], rows_per_batch);
        const unsigned long long *fx = fixed + (size_t)n * n4_per_batch * 4;
        float4 *gv = grad_value + (size_t)n * n4_per_batch;
        for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < n4_per_batch;
             t += (size_t)gridDim.x * blockDim.x) {
            const size_t ch = t & (R - 1);
            const unsigned long long *w = fx + (t - ch) * 4 + ch;
            float4 v = make_float4(ldexpf(__ll2float_rn((long long)__ldcs(w)), -shift),
                                   ldexpf(__ll2float_rn((long long)__ldcs(w + R)), -shift),
                                   ldexpf(__ll2float_rn((long long)__ldcs(w + 2 * R)), -shift),
                                   ldexpf(__ll2float_rn((long long)__ldcs(w + 3 * R)), -shift));
            if (accumulate) {
                const float4 o = gv[t];
                v = make_float4(o.x + v.x, o.y + v.y, o.z + v.z, o.w + v.w);
            }
            gv[t] = v;
        }
    }
}

static unsigned grid_for(size_t work, int threads) {
    size_t b = (work + threads - 1) / threads;
    if (b > 148u * 32u) b = 148u * 32u;
    return (unsigned)(b ? b : 1);
}

// Deterministic workspace: a header of one 32-bit bound per batch element,
// padded to a multiple of 256 bytes, then the fixed-point accumulators.
static size_t workspace_header_bytes(int N) { return ((size_t)(N > 0 ? N : 1) * 4 + 255) / 256 * 256; }

size_t backward_workspace_bytes(const LaunchGeometry &g, int D, bool deterministic) {
    if (!deterministic) return 0;
    const size_t n = (size_t)g.d.N * g.d.Len_in * g.d.M * D;
    return workspace_header_bytes(g.d.N) + n * sizeof(unsigned long long);
}

// grid.y of the per-batch helper kernels
static unsigned batch_grid(int N) { return (unsigned)(N < 1 ? 1 : (N > 65535 ? 65535 : N)); }

// Levels whose samples are dense enough that neighbouring queries' corners
// often coincide: Len_q * n_points samples on H*W pixels, at least 32 per pixel.
static unsigned merge_levels(const LaunchGeometry &g) {
    unsigned mask = 0;
    for (int l = 0; l < g.d.L; ++l) {
        const double pixels = (double)g.lv.H[l] * (double)g.lv.W[l];
        if ((double)g.d.Len_q * g.d.K >= 32.0 * pixels) mask |= 1u << l;
    }
    return mask;
}

// grad_value preparation and completion, shared by the 2-D and 3-D
// backward: zeroing (fp32 mode) or the fixed-point accumulators and their
// per-batch scale bounds (deterministic mode); then the conversion back to
// fp32.  attn == nullptr: fused call, whose rows' weights sum to row_sum.
cudaError_t backward_prepare(const LaunchGeometry &g, int dtype, int D, const float *attn, float row_sum,
                             const void *grad_out, float *grad_value, bool det, bool accumulate, void *workspace,
                             unsigned long long **fixed, const unsigned **bound, cudaStream_t stream) {
    const size_t nval = (size_t)g.d.N * g.d.Len_in * g.d.M * D;
    *fixed = nullptr;
    *bound = nullptr;
    if (det) {
        const size_t hdr_bytes = workspace_header_bytes(g.d.N);
        unsigned *hdr = static_cast<unsigned *>(workspace);
        *fixed = reinterpret_cast<unsigned long long *>(static_cast<char *>(workspace) + hdr_bytes);
        *bound = hdr;
        // header and accumulators are contiguous: zero both
        zero_u64_kernel<<<grid_for((nval * 8 + hdr_bytes) / 16, 256), 256, 0, stream>>>(
            static_cast<ulonglong2 *>(workspace), (nval * 8 + hdr_bytes) / 16);
        if (g.d.rows > 0) {
            const dim3 grid(grid_for(g.d.qm, 256) / batch_grid(g.d.N) + 1, batch_grid(g.d.N));
#define MSDA_BOUND(T, DD) row_bound_kernel<T, DD><<<grid, 256, 0, stream>>>( \
        attn, static_cast<const T *>(grad_out), g.d.N, g.d.qm, g.d.P, row_sum, hdr)
            if (dtype == 0) {
                switch (D) {
                    case 8: MSDA_BOUND(float, 8); break;
                    case 16: MSDA_BOUND(float, 16); break;
                    case 32: MSDA_BOUND(float, 32); break;
                    case 64: MSDA_BOUND(float, 64); break;
                    case 128: MSDA_BOUND(float, 128); break;
                    case 256: MSDA_BOUND(float, 256); break;
                }
            } else {
                switch (D) {
                    case 8: MSDA_BOUND(__nv_bfloat16, 8); break;
                    case 16: MSDA_BOUND(__nv_bfloat16, 16); break;
                    case 32: MSDA_BOUND(__nv_bfloat16, 32); break;
                    case 64: MSDA_BOUND(__nv_bfloat16, 64); break;
                    case 128: MSDA_BOUND(__nv_bfloat16, 128); break;
                    case 256: MSDA_BOUND(__nv_bfloat16, 256); break;
                }
            }
#undef MSDA_BOUND
        }
    } else if (!accumulate && nval > 0) {
        zero_f32_kernel<<<grid_for(nval / 4, 256), 256, 0, stream>>>(reinterpret_cast<float4 *>(grad_value), nval / 4);
    }
    return cudaGetLastError();
}

cudaError_t backward_finish(const LaunchGeometry &g, int D, float *grad_value, bool det, bool accumulate,
                            const unsigned long long *fixed, const unsigned *bound, cudaStream_t stream) {
    const size_t per_batch = (size_t)g.d.Len_in * g.d.M * D / 4;
    if (det && per_batch > 0 && g.d.N > 0) {
        const dim3 grid(grid_for(per_batch, 256) / batch_grid(g.d.N) + 1, batch_grid(g.d.N));
        fixed_to_f32_kernel<<<grid, 256, 0, stream>>>(fixed, bound, g.d.N, g.d.qm,
                                                      reinterpret_cast<float4 *>(grad_value), per_batch, D,
                                                      accumulate ? 1 : 0);
    }
    return cudaGetLastError();
}

// Inputs and outputs of one backward launch.  Unfused: loc, attn -> grad_loc,
// grad_attn.  Fused: ref, off, logits -> grad_off (in grad_loc), grad_logits
// (in grad_attn), grad_ref.
struct BwdIO {
    const void *value;
    const float *loc, *attn;              // unfused
    const float *ref, *off, *logits;      // fused
    const void *grad_out;
    float *grad_value, *grad_loc, *grad_attn, *grad_ref;
};

template <typename T, int D, bool FUSED, bool OPTS>
static void launch_bwd_kernel(const BwdArgs &a, bool det, unsigned blocks, cudaStream_t stream) {
    constexpr int HW = BwdLanes<D>::HW;
    constexpr int B = kBwdWarpsPerBlock * 32;
    const bool merge = a.merge_mask != 0;
    if constexpr (HW == 4 || HW == 2 || HW == 1) {
        if (det && merge) msda_backward_kernel<T, D, true, true, FUSED, OPTS><<<blocks, B, 0, stream>>>(a);
        else if (det) msda_backward_kernel<T, D, true, false, FUSED, OPTS><<<blocks, B, 0, stream>>>(a);
        else if (merge) msda_backward_kernel<T, D, false, true, FUSED, OPTS><<<blocks, B, 0, stream>>>(a);
        else msda_backward_kernel<T, D, false, false, FUSED, OPTS><<<blocks, B, 0, stream>>>(a);
    } else {
        if (det) msda_backward_kernel<T, D, true, false, FUSED, OPTS><<<blocks, B, 0, stream>>>(a);
        else msda_backward_kernel<T, D, false, false, FUSED, OPTS><<<blocks, B, 0, stream>>>(a);
    }
}

template <typename T, int D, bool FUSED>
static cudaError_t launch_bwd_t(const LaunchGeometry &g, const BwdIO &io, bool det, bool accumulate, void *workspace,
                                cudaStream_t stream) {
    constexpr int HW = BwdLanes<D>::HW;
    BwdArgs a{};
    a.value = io.value;
    a.loc = io.loc;
    a.attn = io.attn;
    a.ref = io.ref;
    a.off = io.off;
    a.logits = io.logits;
    a.grad_out = io.grad_out;
    a.grad_value = io.grad_value;
    a.grad_loc = io.grad_loc;
    a.grad_attn = io.grad_attn;
    a.d = g.d;
    a.lv = g.lv;
    for (int s = 0; s < kMaxSamples; ++s) a.level_of[s] = g.level_of[s];
    a.qblocks = (g.d.Len_q + HW - 1) / HW;
    // deterministic mode: a fixed-point reduction is four 64-bit atomics per
    // lane and corner, so merging pays on every level
    // Levels merged: every level in deterministic mode (a fixed-point reduction
    // costs four); in fp32 mode the coarse levels, and every level where a
    // warp holds one query of 256 channels, whose merged entry saves two 512-byte
    // rows of reductions.  Measured on the encoder with G sets: 64 channels
    // every level 444 against 383 us coarse; 128 channels 409 against 385 us;
    // 256 channels 373 against 389 us.
    const unsigned all_levels = (1u << g.d.L) - 1u;
    constexpr bool kMergeable = HW == 4 || HW == 2 || HW == 1;
    a.merge_mask = !kMergeable ? 0u : (det || (HW == 1 && BwdLanes<D>::NV == 2)) ? all_levels : merge_levels(g);
    // fused: a row's weights are softmax outputs, summing to 1 (n_levels with
    // the per-level softmax)
    const float row_sum = g.d.per_level_softmax ? (float)g.d.L : 1.f;
    unsigned long long *fixed = nullptr;
    const unsigned *bound = nullptr;
    cudaError_t e = backward_prepare(g, sizeof(T) == 4 ? 0 : 1, D, FUSED ? nullptr : io.attn, row_sum, io.grad_out,
                                     io.grad_value, det, accumulate, workspace, &fixed, &bound, stream);
    if (e != cudaSuccess) return e;
    a.fixed = fixed;
    a.bound_bits = bound;
    if (g.d.rows > 0) {
        const long long tasks = (long long)g.d.N * a.qblocks * g.d.M;
        const unsigned blocks = (unsigned)((tasks + kBwdWarpsPerBlock - 1) / kBwdWarpsPerBlock);
        if (FUSED && (g.d.per_level_softmax || g.lv.shift != 0.5f))
            launch_bwd_kernel<T, D, FUSED, true>(a, det, blocks, stream);
        else
            launch_bwd_kernel<T, D, FUSED, false>(a, det, blocks, stream);
        if (FUSED) {
            const int nql = g.d.N * g.d.Len_q * g.d.L;
            const int ML = g.d.M * g.d.L;
            if (32 % ML == 0 && nql < (1 << 16)) {      // small problems whose heads x levels tile a warp
                const int nqml = nql * g.d.M;
                ref_grad_kernel_rows<<<grid_for(nqml, 256), 256, 0, stream>>>(io.grad_loc, io.grad_ref, nqml, g.d.M,
                                                                            g.d.L, g.d.K, g.lv);
            } else {
                ref_grad_kernel<<<grid_for(nql, 256), 256, 0, stream>>>(io.grad_loc, io.grad_ref, nql, g.d.M, g.d.L,
                                                                       g.d.K, g.lv);
            }
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return backward_finish(g, D, io.grad_value, det, accumulate, fixed, bound, stream);
}

template <bool FUSED>
static cudaError_t dispatch_bwd(const LaunchGeometry &g, int dtype, int D, const BwdIO &io, bool det, bool accumulate,
                                void *workspace, cudaStream_t stream) {
    if (dtype == 0) {
        switch (D) {
            case 8: return launch_bwd_t<float, 8, FUSED>(g, io, det, accumulate, workspace, stream);
            case 16: return launch_bwd_t<float, 16, FUSED>(g, io, det, accumulate, workspace, stream);
            case 32: return launch_bwd_t<float, 32, FUSED>(g, io, det, accumulate, workspace, stream);
            case 64: return launch_bwd_t<float, 64, FUSED>(g, io, det, accumulate, workspace, stream);
            case 128: return launch_bwd_t<float, 128, FUSED>(g, io, det, accumulate, workspace, stream);
            case 256: return launch_bwd_t<float, 256, FUSED>(g, io, det, accumulate, workspace, stream);
        }
    } else {
        switch (D) {
            case 8: return launch_bwd_t<__nv_bfloat16, 8, FUSED>(g, io, det, accumulate, workspace, stream);
            case 16: return launch_bwd_t<__nv_bfloat16, 16, FUSED>(g, io, det, accumulate, workspace, stream);
            case 32: return launch_bwd_t<__nv_bfloat16, 32, FUSED>(g, io, det, accumulate, workspace, stream);
            case 64: return launch_bwd_t<__nv_bfloat16, 64, FUSED>(g, io, det, accumulate, workspace, stream);
            case 128: return launch_bwd_t<__nv_bfloat16, 128, FUSED>(g, io, det, accumulate, workspace, stream);
            case 256: return launch_bwd_t<__nv_bfloat16, 256, FUSED>(g, io, det, accumulate, workspace, stream);
        }
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_backward(const LaunchGeometry &g, int dtype, int D, const void *value, const float *loc,
                            const float *attn, const void *grad_out, float *grad_value, float *grad_loc,
                            float *grad_attn, bool det, bool accumulate, void *workspace, cudaStream_t stream) {
    BwdIO io{};
    io.value = value;
    io.loc = loc;
    io.attn = attn;
    io.grad_out = grad_out;
    io.grad_value = grad_value;
    io.grad_loc = grad_loc;
    io.grad_attn = grad_attn;
    return dispatch_bwd<false>(g, dtype, D, io, det, accumulate, workspace, stream);
}

cudaError_t launch_backward_fused(const LaunchGeometry &g, int dtype, int D, const void *value, const float *ref,
                                  const float *off, const float *logits, const void *grad_out, float *grad_value,
                                  float *grad_ref, float *grad_off, float *grad_logits, bool det, bool accumulate,
                                  void *workspace, cudaStream_t stream) {
    BwdIO io{};
    io.value = value;
    io.ref = ref;
    io.off = off;
    io.logits = logits;
    io.grad_out = grad_out;
    io.grad_value = grad_value;
    io.grad_loc = grad_off;
    io.grad_attn = grad_logits;
    io.grad_ref = grad_ref;
    return dispatch_bwd<true>(g, dtype, D, io, det, accumulate, workspace, stream);
}

}  // namespace msda
