// line_rates.cu -- measurement kernels (libmsda_probes.so, include/msda_probes.h):
// how fast this GPU's SMs gather random 128-byte lines and reduce into them.
//
// A bilinear sample of the MSDeformAttn kernels reads four value rows from
// random places and, in the backward, adds into as many rows of grad_value;
// at head_dim = 32 fp32 a row is one 128-byte line, read or reduced by eight
// lanes of 16 bytes, four rows per warp instruction.  These probes do exactly
// that access and nothing else, so their rates are the ceilings those kernels
// run against.  Line indices come from an integer hash, reduced into
// [0, n_lines) by a multiply-high: every access is inside the buffer.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../../include/msda_probes.h"

namespace {

constexpr int kThreads = 256;
constexpr int kBlocks = 148 * 8;       // eight resident blocks on each of the 148 SMs

// 32-bit integer hash (xorshift-multiply, the "lowbias32" constants)
__device__ __forceinline__ uint32_t mix32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}

// accesses per launch of the probes below (defined after them)
long long rounds_for(int64_t lines);

// uniform in [0, n): (h * n) / 2^32 < n
__device__ __forceinline__ uint32_t pick(uint32_t h, uint32_t n) { return (uint32_t)(((uint64_t)h * n) >> 32); }

// the 32-bit linear congruential step of Numerical Recipes (a = 1664525,
// c = 1013904223): one multiply-add a line, so the probes spend their issue
// slots on the accesses, not on the index arithmetic
__device__ __forceinline__ uint32_t lcg(uint32_t x) { return x * 1664525u + 1013904223u; }

__device__ __forceinline__ float4 ldg_line(const float4 *p) {
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void red_line(float4 *p, float4 v) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

constexpr int kUnroll = 8;             // independent accesses in flight per thread

// A quarter-warp (eight lanes, 16 bytes each) covers one line per access; its
// lines come from its own generator stream, so a warp instruction covers four
// lines.  Every quarter-warp runs the same number of rounds of kUnroll
// accesses: a launch makes msda_probe_accesses(lines) >= lines of them.
__global__ void __launch_bounds__(kThreads) gather_kernel(const float4 *buf, uint32_t n, long long rounds,
                                                          float4 *sink, uint32_t seed) {
    const int sub = threadIdx.x & 7;
    const uint32_t quarter = (blockIdx.x * blockDim.x + threadIdx.x) >> 3;
    uint32_t x = mix32(seed ^ mix32(quarter));
    float acc = 0.f;
    for (long long r = 0; r < rounds; ++r) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            x = lcg(x);
            v[u] = ldg_line(buf + (size_t)pick(x, n) * 8 + sub);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) acc += v[u].x;
    }
    sink[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = make_float4(acc, 0.f, 0.f, 0.f);
}

__global__ void __launch_bounds__(kThreads) reduce_kernel(float4 *buf, uint32_t n, long long rounds, uint32_t seed) {
    const int sub = threadIdx.x & 7;
    const uint32_t quarter = (blockIdx.x * blockDim.x + threadIdx.x) >> 3;
    uint32_t x = mix32(seed ^ mix32(quarter));
    const float4 one = make_float4(1.f, 1.f, 1.f, 1.f);
    for (long long r = 0; r < rounds; ++r) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            x = lcg(x);
            red_line(buf + (size_t)pick(x, n) * 8 + sub, one);
        }
    }
}

// Per round kUnroll gathers, then reds_per_8 (0..8) reductions into other lines.
__global__ void __launch_bounds__(kThreads) mixed_kernel(float4 *buf, uint32_t n, long long rounds, int reds_per_8,
                                                         float4 *sink, uint32_t seed) {
    const int sub = threadIdx.x & 7;
    const uint32_t quarter = (blockIdx.x * blockDim.x + threadIdx.x) >> 3;
    uint32_t x = mix32(seed ^ mix32(quarter)), y = mix32(~seed ^ mix32(quarter));
    float acc = 0.f;
    const float4 one = make_float4(1.f, 1.f, 1.f, 1.f);
    for (long long r = 0; r < rounds; ++r) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            x = lcg(x);
            v[u] = ldg_line(buf + (size_t)pick(x, n) * 8 + sub);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (u < reds_per_8) {
                y = lcg(y);
                red_line(buf + (size_t)pick(y, n) * 8 + sub, one);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) acc += v[u].x;
    }
    sink[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = make_float4(acc, 0.f, 0.f, 0.f);
}

// Bulk (TMA) reductions: each quarter-warp stages its line in one of kSlots
// 128-byte shared-memory slots (its eight lanes write 16 bytes each), fences
// the writes to the async proxy, and its first lane issues one
// cp.reduce.async.bulk .add.f32 of the 128 bytes into the line, so a warp
// step covers four lines as the reductions above do.  A slot is written again
// only after the bulk group that read it has finished reading (wait_group.read
// on the issuing lane, which owns the groups), and every lane's groups are
// complete before the kernel returns.
constexpr int kSlots = 8;

__global__ void __launch_bounds__(kThreads) bulk_reduce_kernel(float4 *buf, uint32_t n, long long rounds,
                                                               uint32_t seed) {
    __shared__ __align__(128) float4 stage[kThreads / 8][kSlots][8];     // [quarter][slot][lane]
    const int sub = threadIdx.x & 7, qw = threadIdx.x >> 3;
    const uint32_t quarter = (blockIdx.x * blockDim.x + threadIdx.x) >> 3;
    uint32_t x = mix32(seed ^ mix32(quarter));
    const float4 one = make_float4(1.f, 1.f, 1.f, 1.f);
    for (long long r = 0; r < rounds; ++r) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int slot = u % kSlots;
            x = lcg(x);
            const uint32_t line = pick(x, n);
            if (sub == 0) asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kSlots - 1) : "memory");
            __syncwarp();
            stage[qw][slot][sub] = one;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (sub == 0) {
                const uint32_t sa = (uint32_t)__cvta_generic_to_shared(&stage[qw][slot][0]);
                asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], 128;"
                             ::"l"(buf + (size_t)line * 8), "r"(sa) : "memory");
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
        }
    }
    if (sub == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
}

// accesses per launch: rounds * kUnroll * quarter-warps
long long rounds_for(int64_t lines) {
    const long long q = (long long)kBlocks * kThreads / 8;
    return (lines + q * kUnroll - 1) / (q * kUnroll);
}

bool lines_ok(int64_t n_lines, int64_t lines) { return n_lines >= 1 && n_lines < (int64_t(1) << 31) && lines >= 0; }

}  // namespace

extern "C" {

size_t msda_probe_sink_bytes(void) { return (size_t)kBlocks * kThreads * sizeof(float4); }

int64_t msda_probe_accesses(int64_t lines) {
    return lines < 0 ? 0 : rounds_for(lines) * kUnroll * ((int64_t)kBlocks * kThreads / 8);
}

int msda_probe_gather(const void *buf, int64_t n_lines, int64_t hot_lines, int64_t lines, void *sink, uint32_t seed,
                      void *stream) {
    if (!buf || !sink || !lines_ok(n_lines, lines) || hot_lines < 0) return (int)cudaErrorInvalidValue;
    const uint32_t n = (uint32_t)(hot_lines > 0 && hot_lines < n_lines ? hot_lines : n_lines);
    gather_kernel<<<kBlocks, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const float4 *>(buf), n, rounds_for(lines), static_cast<float4 *>(sink), seed);
    return (int)cudaGetLastError();
}

int msda_probe_bulk_reduce(void *buf, int64_t n_lines, int64_t lines, uint32_t seed, void *stream) {
    if (!buf || !lines_ok(n_lines, lines) || (reinterpret_cast<uintptr_t>(buf) & 15)) return (int)cudaErrorInvalidValue;
    bulk_reduce_kernel<<<kBlocks, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<float4 *>(buf), (uint32_t)n_lines, rounds_for(lines), seed);
    return (int)cudaGetLastError();
}

int msda_probe_reduce(void *buf, int64_t n_lines, int64_t hot_lines, int64_t lines, uint32_t seed, void *stream) {
    if (!buf || !lines_ok(n_lines, lines) || hot_lines < 0) return (int)cudaErrorInvalidValue;
    const uint32_t n = (uint32_t)(hot_lines > 0 && hot_lines < n_lines ? hot_lines : n_lines);
    reduce_kernel<<<kBlocks, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<float4 *>(buf), n,
                                                                              rounds_for(lines), seed);
    return (int)cudaGetLastError();
}

int msda_probe_mixed(void *buf, int64_t n_lines, int64_t lines, int reds_per_8, void *sink, uint32_t seed,
                     void *stream) {
    if (!buf || !sink || !lines_ok(n_lines, lines) || reds_per_8 < 0 || reds_per_8 > 8)
        return (int)cudaErrorInvalidValue;
    mixed_kernel<<<kBlocks, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<float4 *>(buf), (uint32_t)n_lines, rounds_for(lines), reds_per_8, static_cast<float4 *>(sink),
        seed);
    return (int)cudaGetLastError();
}

}  // extern "C"
