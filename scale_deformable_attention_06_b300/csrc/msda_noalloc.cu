// msda_noalloc.cu -- msda_backward_noalloc: the deterministic backward with
// its scratch memory inside the library, for callers that cannot allocate
// device memory (see include/msda.h).
//
// The scratch is one file-scope device array.  Host code never uses its name
// as an address: the name is a host-side stand-in for the device symbol.  The
// device address is looked up with cudaGetSymbolAddress, once per device, with
// that device current, and passed to the kernels like any caller workspace.
#include <cstdio>
#include <mutex>

#include "../../include/msda.h"
#include "msda_launch.h"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(64) << 20;   // 64 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device; the first call
// per device does the lookup.
cudaError_t scratch_for_current_device(void **out, int *device) {
    cudaError_t e = cudaGetDevice(device);
    if (e != cudaSuccess) return e;
    if (*device < 0 || *device >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[*device]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[*device] = p;
    }
    *out = g_scratch_ptr[*device];
    return cudaSuccess;
}

}  // namespace

namespace msda {
msda_status noalloc_check_and_geometry(const msda_problem *problem, const int64_t *spatial_shapes,
                                       const int64_t *level_start_index, LaunchGeometry &g);
msda_status noalloc_fail(msda_status s, const char *msg);
msda_status noalloc_check_pointers(const msda_problem *problem, const LaunchGeometry &g, const void *value,
                                   const float *loc, const float *attn, const void *grad_out, const float *grad_value,
                                   const float *grad_loc, const float *grad_attn);
}  // namespace msda

extern "C" msda_status msda_backward_noalloc(const msda_problem *problem, const void *value,
                                             const int64_t *spatial_shapes, const int64_t *level_start_index,
                                             const float *sampling_locations, const float *attention_weights,
                                             const void *grad_output, float *grad_value,
                                             float *grad_sampling_locations, float *grad_attention_weights,
                                             unsigned flags, void *stream) {
    msda::LaunchGeometry g;
    msda_status st = msda::noalloc_check_and_geometry(problem, spatial_shapes, level_start_index, g);
    if (st != MSDA_OK) return st;
    if (flags & ~MSDA_ACCUMULATE_GRAD_VALUE)
        return msda::noalloc_fail(MSDA_ERR_INVALID_ARG, "msda_backward_noalloc: only MSDA_ACCUMULATE_GRAD_VALUE is accepted");
    const size_t need = msda::backward_workspace_bytes(g, g.D, true);
    if (need > kNoallocScratchBytes) {
        char msg[400];
        snprintf(msg, sizeof(msg),
                 "msda_backward_noalloc: this problem needs %zu bytes of scratch (8 per grad_value element plus "
                 "4 per batch element, rounded up to 256), above the built-in %zu; use msda_backward with a "
                 "workspace",
                 need, kNoallocScratchBytes);
        return msda::noalloc_fail(MSDA_ERR_UNSUPPORTED, msg);
    }
    st = msda::noalloc_check_pointers(problem, g, value, sampling_locations, attention_weights, grad_output, grad_value,
                                      grad_sampling_locations, grad_attention_weights);
    if (st != MSDA_OK) return st;
    const size_t nval = (size_t)g.d.N * g.d.Len_in * g.d.M * g.D;
    const bool acc = (flags & MSDA_ACCUMULATE_GRAD_VALUE) != 0;
    if (nval == 0 && g.d.rows == 0) return MSDA_OK;
    if (g.d.rows == 0 && acc) return MSDA_OK;

    void *scratch = nullptr;
    int device = -1;
    cudaError_t e = scratch_for_current_device(&scratch, &device);
    if (e != cudaSuccess) {
        char msg[400];
        snprintf(msg, sizeof(msg), "msda_backward_noalloc: scratch lookup on device %d: %s", device,
                 cudaGetErrorString(e));
        return msda::noalloc_fail(MSDA_ERR_CUDA, msg);
    }
    // launch_backward clears the fixed-point accumulators and the bound header
    // in the scratch before it sums into them, so the previous call's contents
    // do not leak into this one.
    e = msda::launch_backward(g, problem->dtype, g.D, value, sampling_locations, attention_weights,
                              grad_output, grad_value, grad_sampling_locations, grad_attention_weights, true, acc,
                              scratch, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        char msg[400];
        snprintf(msg, sizeof(msg), "msda_backward_noalloc launch: %s", cudaGetErrorString(e));
        return msda::noalloc_fail(MSDA_ERR_CUDA, msg);
    }
    return MSDA_OK;
}
