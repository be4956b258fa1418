"""ctypes binding of libmsda (include/msda.h): argument marshalling only.

Every function here checks shapes and dtypes of torch tensors, passes their
device pointers and the current CUDA stream to the C ABI, and raises
MSDAError when the library returns a non-OK status.  No step of the method
runs in Python; there is no CPU fallback.  If libmsda.so has not been built,
importing the package raises ImportError.
"""
import contextlib
import contextvars
import ctypes
import functools
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_HERE, "libmsda.so")
# the same kernels with every access checked against its tensor's extent
# (include/msda_debug.h); for tests, through using_library()
DEBUG_LIBRARY = os.path.join(_HERE, "libmsda_debug.so")

MSDA_OK = 0
MSDA_F32 = 0
MSDA_BF16 = 1
MSDA_DETERMINISTIC = 1
MSDA_ACCUMULATE_GRAD_VALUE = 2
MSDA_OPT_PER_LEVEL_SOFTMAX = 1
MSDA_OPT_ALIGN_CORNERS = 2

EXPORTED = ("msda_forward", "msda_forward_fused", "msda_backward", "msda_backward_fused",
            "msda_backward_workspace_size", "msda_backward_noalloc", "msda3d_forward", "msda3d_backward",
            "msda_status_string", "msda_last_error", "msda_version")


class MSDAError(RuntimeError):
    def __init__(self, status, name, detail):
        super().__init__(f"{name}: {detail}")
        self.status = status
        self.name = name


class msda_problem(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int32), ("Len_in", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("Len_q", ctypes.c_int32), ("n_levels", ctypes.c_int32),
                ("n_points", ctypes.c_int32), ("dtype", ctypes.c_int32), ("options", ctypes.c_uint32),
                ("n_groups", ctypes.c_int32)]


def _load(path=LIBRARY):
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python scale_deformable_attention_06_b300/build.py` (or __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    vp, i64p, fp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.c_void_p
    pp = ctypes.POINTER(msda_problem)
    lib.msda_forward.argtypes = [pp, vp, i64p, i64p, fp, fp, vp, vp]
    lib.msda_forward_fused.argtypes = [pp, vp, i64p, i64p, fp, fp, fp, vp, vp]
    lib.msda_backward.argtypes = [pp, vp, i64p, i64p, fp, fp, vp, fp, fp, fp, ctypes.c_uint, vp, ctypes.c_size_t, vp]
    lib.msda_backward_fused.argtypes = [pp, vp, i64p, i64p, fp, fp, fp, vp, fp, fp, fp, fp, ctypes.c_uint, vp,
                                        ctypes.c_size_t, vp]
    lib.msda_backward_noalloc.argtypes = [pp, vp, i64p, i64p, fp, fp, vp, fp, fp, fp, ctypes.c_uint, vp]
    lib.msda3d_forward.argtypes = [pp, vp, i64p, i64p, fp, fp, vp, vp]
    lib.msda3d_backward.argtypes = [pp, vp, i64p, i64p, fp, fp, vp, fp, fp, fp, ctypes.c_uint, vp, ctypes.c_size_t, vp]
    lib.msda_backward_noalloc.restype = ctypes.c_int
    lib.msda_backward_workspace_size.argtypes = [pp, ctypes.c_uint]
    lib.msda_backward_workspace_size.restype = ctypes.c_size_t
    for f in ("msda_forward", "msda_forward_fused", "msda_backward", "msda_backward_fused", "msda3d_forward",
              "msda3d_backward"):
        getattr(lib, f).restype = ctypes.c_int
    lib.msda_status_string.argtypes = [ctypes.c_int]
    lib.msda_status_string.restype = ctypes.c_char_p
    lib.msda_last_error.argtypes = []
    lib.msda_last_error.restype = ctypes.c_char_p
    lib.msda_version.restype = ctypes.c_int
    if hasattr(lib, "msda_debug_violations"):
        lib.msda_debug_violations.argtypes = [ctypes.c_int]
        lib.msda_debug_violations.restype = ctypes.c_ulonglong
    return lib


_lib = _load()


@contextlib.contextmanager
def using_library(path):
    """Route every call of this module to another build of the library (the
    debug build DEBUG_LIBRARY) inside the with-block; yields that ctypes
    library."""
    global _lib
    saved, _lib = _lib, _load(path)
    try:
        yield _lib
    finally:
        _lib = saved


def lib():
    """The loaded ctypes library (for tests that call the C ABI directly)."""
    return _lib


def _check(status):
    if status != MSDA_OK:
        raise MSDAError(status, _lib.msda_status_string(status).decode(), _lib.msda_last_error().decode())


def _dtype_code(t):
    if t.dtype == torch.float32:
        return MSDA_F32
    if t.dtype == torch.bfloat16:
        return MSDA_BF16
    raise TypeError(f"value dtype {t.dtype} is not float32 or bfloat16")


# the device of the call being marshalled (that of its value tensor)
_CALL_DEVICE = contextvars.ContextVar("msda_call_device", default=None)


def _on_value_device(fn):
    """Runs a call with its value tensor's device current (the library
    launches on the current device); every tensor the call passes must live
    on that device."""
    @functools.wraps(fn)
    def call(value, *args, **kwargs):
        if not isinstance(value, torch.Tensor):
            raise TypeError("value must be a torch.Tensor")
        if not value.is_cuda:
            raise ValueError("value must be on a CUDA device (there is no CPU path)")
        token = _CALL_DEVICE.set(value.device)
        try:
            with torch.cuda.device(value.device):
                return fn(value, *args, **kwargs)
        finally:
            _CALL_DEVICE.reset(token)
    return call


def _dev(t, name, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device (there is no CPU path)")
    device = _CALL_DEVICE.get()
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, value on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


class _HostLevels:
    """spatial_shapes [L,2] and level_start_index [L] as host int64 arrays."""

    def __init__(self, spatial_shapes, level_start_index):
        sh = torch.as_tensor(spatial_shapes).detach().to("cpu", torch.int64).contiguous().reshape(-1, 2)
        st = torch.as_tensor(level_start_index).detach().to("cpu", torch.int64).contiguous().reshape(-1)
        self.sh, self.st = sh, st          # keep alive for the call
        self.L = sh.shape[0]
        self.shp = ctypes.cast(sh.data_ptr(), ctypes.POINTER(ctypes.c_int64))
        self.stp = ctypes.cast(st.data_ptr(), ctypes.POINTER(ctypes.c_int64))


def _stream(stream, device):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))




def _check_out(t, name, shape, dtype):
    """A caller-passed output tensor must have exactly this shape and dtype."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")

def groups_of(value, per_sample):
    """G, the sets of locations of a call: per_sample [N, Len_q, G, ...] holds one
    set per head (G = M) or one per group of M / G heads; G must divide M."""
    M = value.shape[2]
    G = per_sample.shape[2] if per_sample.dim() >= 3 else 0
    if G < 1 or M % G:
        raise ValueError(f"the per-sample tensors have {G} sets, which does not divide n_heads {M}")
    return G


def _check_backward_args(value, n_levels, sampling_locations, attention_weights, grad_output, grad_value=None,
                         grad_sampling_locations=None, grad_attention_weights=None, coords=2):
    """Shapes and dtypes of a backward call, checked before anything reaches
    the library (a wrong size there would be read or written out of bounds).
    value [N,Len_in,M,D]; sampling_locations [N,Len_q,G,L,K,coords] (G = M, or
    G groups of M / G heads); attention_weights [N,Len_q,G,L,K]; grad_output
    [N,Len_q,M*D] with the dtype of value; the optional outputs grad_value
    [N,Len_in,M,D], grad_sampling_locations and grad_attention_weights (shaped
    like the locations and weights), all float32.  Returns (Len_q, L, K)."""
    if value.dim() != 4:
        raise ValueError("value must be [N, Len_in, M, D]")
    N, S, M, D = value.shape
    if sampling_locations.dim() != 6 or sampling_locations.shape[-1] != coords:
        raise ValueError(f"sampling_locations must be [N, Len_q, G, L, K, {coords}]")
    G = groups_of(value, sampling_locations)
    Lq, L, K = sampling_locations.shape[1], sampling_locations.shape[3], sampling_locations.shape[4]
    if tuple(sampling_locations.shape[:5]) != (N, Lq, G, L, K):
        raise ValueError("sampling_locations disagrees with value (N)")
    if tuple(attention_weights.shape) != (N, Lq, G, L, K):
        raise ValueError("attention_weights must be [N, Len_q, G, L, K], like sampling_locations")
    if tuple(grad_output.shape) != (N, Lq, M * D):
        raise ValueError("grad_output must be [N, Len_q, M*D]")
    if grad_output.dtype != value.dtype:
        raise TypeError("grad_output must have the dtype of value")
    if L != n_levels:
        raise ValueError("n_levels of sampling_locations and spatial_shapes disagree")
    for t, name in ((sampling_locations, "sampling_locations"), (attention_weights, "attention_weights")):
        if t.dtype != torch.float32:
            raise TypeError(f"{name} must be torch.float32, got {t.dtype}")
    _check_out(grad_value, "grad_value", (N, S, M, D), torch.float32)
    _check_out(grad_sampling_locations, "grad_sampling_locations", sampling_locations.shape, torch.float32)
    _check_out(grad_attention_weights, "grad_attention_weights", (N, Lq, G, L, K), torch.float32)
    return Lq, L, K

def _grad_value_out(value, grad_value, flags):
    """The grad_value the backward writes: the caller's, else a new one.  With
    MSDA_ACCUMULATE_GRAD_VALUE the library adds into it, so a new (unwritten)
    tensor would give garbage: the caller must pass the one to add into."""
    if grad_value is not None:
        return grad_value
    if flags & MSDA_ACCUMULATE_GRAD_VALUE:
        raise ValueError("MSDA_ACCUMULATE_GRAD_VALUE adds into the caller's grad_value: pass grad_value")
    N, S, M, D = value.shape
    return torch.empty((N, S, M, D), dtype=torch.float32, device=value.device)


def problem(value, Len_q, n_levels, n_points, options=0, n_groups=0):
    N, S, M, D = value.shape
    return msda_problem(N, S, M, D, Len_q, n_levels, n_points, _dtype_code(value), options,
                        0 if n_groups == M else n_groups)


@_on_value_device
def msda_forward(value, spatial_shapes, level_start_index, sampling_locations, attention_weights,
                 output=None, stream=None, options=0):
    """out[N, Len_q, M*D] from value [N,Len_in,M,D] (f32|bf16), sampling_locations
    [N,Len_q,G,L,K,2] f32 and attention_weights [N,Len_q,G,L,K] f32 (G = M, or the
    number of head groups)."""
    lv = _HostLevels(spatial_shapes, level_start_index)
    N, S, M, D = value.shape
    if sampling_locations.dim() != 6 or sampling_locations.shape[-1] != 2:
        raise ValueError("sampling_locations must be [N, Len_q, G, L, K, 2]")
    G = groups_of(value, sampling_locations)
    Lq, L, K = sampling_locations.shape[1], sampling_locations.shape[3], sampling_locations.shape[4]
    if tuple(sampling_locations.shape[:5]) != (N, Lq, G, L, K) or tuple(attention_weights.shape) != (N, Lq, G, L, K):
        raise ValueError("sampling_locations / attention_weights shapes disagree with value")
    if L != lv.L:
        raise ValueError("n_levels of sampling_locations and spatial_shapes disagree")
    if output is None:
        output = torch.empty((N, Lq, M * D), dtype=value.dtype, device=value.device)
    elif tuple(output.shape) != (N, Lq, M * D) or output.dtype != value.dtype:
        raise ValueError("output must be [N, Len_q, M*D] with the dtype of value")
    prob = problem(value, Lq, L, K, options, G)
    _check(_lib.msda_forward(ctypes.byref(prob), _dev(value, "value"), lv.shp, lv.stp,
                             _dev(sampling_locations, "sampling_locations", torch.float32),
                             _dev(attention_weights, "attention_weights", torch.float32),
                             _dev(output, "output"), _stream(stream, value.device)))
    return output


@_on_value_device
def msda_forward_fused(value, spatial_shapes, level_start_index, reference_points, sampling_offsets,
                       attention_logits, output=None, stream=None, options=0):
    """out[N, Len_q, M*D] from reference_points [N,Len_q,L,2], sampling_offsets
    [N,Len_q,G,L,K,2] (pixels of each level) and attention_logits [N,Len_q,G,L*K]
    (G = M, or the number of head groups)."""
    lv = _HostLevels(spatial_shapes, level_start_index)
    N, S, M, D = value.shape
    if sampling_offsets.dim() != 6 or sampling_offsets.shape[-1] != 2:
        raise ValueError("sampling_offsets must be [N, Len_q, G, L, K, 2]")
    G = groups_of(value, sampling_offsets)
    Lq, L, K = sampling_offsets.shape[1], sampling_offsets.shape[3], sampling_offsets.shape[4]
    if tuple(sampling_offsets.shape[:5]) != (N, Lq, G, L, K):
        raise ValueError("sampling_offsets disagrees with value (N)")
    if tuple(reference_points.shape) != (N, Lq, L, 2):
        raise ValueError("reference_points must be [N, Len_q, L, 2]")
    if attention_logits.numel() != N * Lq * G * L * K:
        raise ValueError("attention_logits must hold N*Len_q*G*L*K values")
    if L != lv.L:
        raise ValueError("n_levels of sampling_offsets and spatial_shapes disagree")
    _check_out(output, "output", (N, Lq, M * D), value.dtype)
    if output is None:
        output = torch.empty((N, Lq, M * D), dtype=value.dtype, device=value.device)
    prob = problem(value, Lq, L, K, options, G)
    _check(_lib.msda_forward_fused(ctypes.byref(prob), _dev(value, "value"), lv.shp, lv.stp,
                                   _dev(reference_points, "reference_points", torch.float32),
                                   _dev(sampling_offsets, "sampling_offsets", torch.float32),
                                   _dev(attention_logits, "attention_logits", torch.float32),
                                   _dev(output, "output"), _stream(stream, value.device)))
    return output


def msda_backward_workspace_size(value, Len_q, n_levels, n_points, flags=0):
    prob = problem(value, Len_q, n_levels, n_points)  # the size does not depend on the options
    return int(_lib.msda_backward_workspace_size(ctypes.byref(prob), flags))


@_on_value_device
def msda_backward(value, spatial_shapes, level_start_index, sampling_locations, attention_weights, grad_output,
                  grad_value=None, grad_sampling_locations=None, grad_attention_weights=None, flags=0,
                  workspace=None, stream=None, options=0):
    """Returns (grad_value f32 [N,Len_in,M,D], grad_sampling_locations, grad_attention_weights)."""
    lv = _HostLevels(spatial_shapes, level_start_index)
    N, S, M, D = value.shape
    Lq, L, K = _check_backward_args(value, lv.L, sampling_locations, attention_weights, grad_output, grad_value,
                                    grad_sampling_locations, grad_attention_weights)
    dev = value.device
    grad_value = _grad_value_out(value, grad_value, flags)
    if grad_sampling_locations is None:
        grad_sampling_locations = torch.empty_like(sampling_locations)
    if grad_attention_weights is None:
        grad_attention_weights = torch.empty_like(attention_weights)
    prob = problem(value, Lq, L, K, options, sampling_locations.shape[2])
    need = int(_lib.msda_backward_workspace_size(ctypes.byref(prob), flags))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = _dev(workspace, "workspace") if workspace is not None else ctypes.c_void_p(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.msda_backward(ctypes.byref(prob), _dev(value, "value"), lv.shp, lv.stp,
                              _dev(sampling_locations, "sampling_locations", torch.float32),
                              _dev(attention_weights, "attention_weights", torch.float32),
                              _dev(grad_output, "grad_output"), _dev(grad_value, "grad_value", torch.float32),
                              _dev(grad_sampling_locations, "grad_sampling_locations", torch.float32),
                              _dev(grad_attention_weights, "grad_attention_weights", torch.float32),
                              flags, ws_ptr, ws_bytes, _stream(stream, dev)))
    return grad_value, grad_sampling_locations, grad_attention_weights


@_on_value_device
def msda_backward_fused(value, spatial_shapes, level_start_index, reference_points, sampling_offsets,
                        attention_logits, grad_output, grad_value=None, grad_reference_points=None,
                        grad_sampling_offsets=None, grad_attention_logits=None, flags=0, workspace=None,
                        stream=None, options=0):
    """Gradient of msda_forward_fused.  Returns (grad_value f32 [N,Len_in,M,D],
    grad_reference_points [N,Len_q,L,2], grad_sampling_offsets [N,Len_q,G,L,K,2],
    grad_attention_logits shaped like attention_logits)."""
    lv = _HostLevels(spatial_shapes, level_start_index)
    N, S, M, D = value.shape
    if sampling_offsets.dim() != 6 or sampling_offsets.shape[-1] != 2:
        raise ValueError("sampling_offsets must be [N, Len_q, G, L, K, 2]")
    G = groups_of(value, sampling_offsets)
    Lq, L, K = sampling_offsets.shape[1], sampling_offsets.shape[3], sampling_offsets.shape[4]
    if tuple(sampling_offsets.shape[:5]) != (N, Lq, G, L, K):
        raise ValueError("sampling_offsets disagrees with value (N)")
    if tuple(reference_points.shape) != (N, Lq, L, 2):
        raise ValueError("reference_points must be [N, Len_q, L, 2]")
    if attention_logits.numel() != N * Lq * G * L * K or tuple(grad_output.shape) != (N, Lq, M * D):
        raise ValueError("attention_logits / grad_output shapes disagree with value")
    if grad_output.dtype != value.dtype:
        raise TypeError("grad_output must have the dtype of value")
    if L != lv.L:
        raise ValueError("n_levels of sampling_offsets and spatial_shapes disagree")
    _check_out(grad_value, "grad_value", (N, S, M, D), torch.float32)
    _check_out(grad_reference_points, "grad_reference_points", reference_points.shape, torch.float32)
    _check_out(grad_sampling_offsets, "grad_sampling_offsets", sampling_offsets.shape, torch.float32)
    _check_out(grad_attention_logits, "grad_attention_logits", attention_logits.shape, torch.float32)
    dev = value.device
    grad_value = _grad_value_out(value, grad_value, flags)
    if grad_reference_points is None:
        grad_reference_points = torch.empty_like(reference_points)
    if grad_sampling_offsets is None:
        grad_sampling_offsets = torch.empty_like(sampling_offsets)
    if grad_attention_logits is None:
        grad_attention_logits = torch.empty_like(attention_logits)
    prob = problem(value, Lq, L, K, options, G)
    need = int(_lib.msda_backward_workspace_size(ctypes.byref(prob), flags))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = _dev(workspace, "workspace") if workspace is not None else ctypes.c_void_p(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.msda_backward_fused(ctypes.byref(prob), _dev(value, "value"), lv.shp, lv.stp,
                                    _dev(reference_points, "reference_points", torch.float32),
                                    _dev(sampling_offsets, "sampling_offsets", torch.float32),
                                    _dev(attention_logits, "attention_logits", torch.float32),
                                    _dev(grad_output, "grad_output"), _dev(grad_value, "grad_value", torch.float32),
                                    _dev(grad_reference_points, "grad_reference_points", torch.float32),
                                    _dev(grad_sampling_offsets, "grad_sampling_offsets", torch.float32),
                                    _dev(grad_attention_logits, "grad_attention_logits", torch.float32),
                                    flags, ws_ptr, ws_bytes, _stream(stream, dev)))
    return grad_value, grad_reference_points, grad_sampling_offsets, grad_attention_logits


@_on_value_device
def msda_backward_noalloc(value, spatial_shapes, level_start_index, sampling_locations, attention_weights,
                          grad_output, grad_value, grad_sampling_locations, grad_attention_weights, flags=0,
                          stream=None, options=0):
    """Deterministic backward with the library's built-in scratch (no workspace,
    no allocation anywhere, the outputs included: the caller passes them).
    For callers that may not allocate device memory; see include/msda.h for
    the size limit and for why overlapping calls race."""
    lv = _HostLevels(spatial_shapes, level_start_index)
    for t, name in ((grad_value, "grad_value"), (grad_sampling_locations, "grad_sampling_locations"),
                    (grad_attention_weights, "grad_attention_weights")):
        if t is None:
            raise ValueError(f"{name} must be passed: this call allocates nothing, its outputs included")
    Lq, L, K = _check_backward_args(value, lv.L, sampling_locations, attention_weights, grad_output, grad_value,
                                    grad_sampling_locations, grad_attention_weights)
    prob = problem(value, Lq, L, K, options, sampling_locations.shape[2])
    _check(_lib.msda_backward_noalloc(ctypes.byref(prob), _dev(value, "value"), lv.shp, lv.stp,
                                      _dev(sampling_locations, "sampling_locations", torch.float32),
                                      _dev(attention_weights, "attention_weights", torch.float32),
                                      _dev(grad_output, "grad_output"), _dev(grad_value, "grad_value", torch.float32),
                                      _dev(grad_sampling_locations, "grad_sampling_locations", torch.float32),
                                      _dev(grad_attention_weights, "grad_attention_weights", torch.float32),
                                      flags, _stream(stream, value.device)))
    return grad_value, grad_sampling_locations, grad_attention_weights


class _HostVolumes:
    """spatial_shapes [L,3] = (D,H,W) and level_start_index [L] as host int64 arrays."""

    def __init__(self, spatial_shapes, level_start_index):
        sh = torch.as_tensor(spatial_shapes).detach().to("cpu", torch.int64).contiguous().reshape(-1, 3)
        st = torch.as_tensor(level_start_index).detach().to("cpu", torch.int64).contiguous().reshape(-1)
        self.sh, self.st = sh, st
        self.L = sh.shape[0]
        self.shp = ctypes.cast(sh.data_ptr(), ctypes.POINTER(ctypes.c_int64))
        self.stp = ctypes.cast(st.data_ptr(), ctypes.POINTER(ctypes.c_int64))


@_on_value_device
def msda3d_forward(value, spatial_shapes, level_start_index, sampling_locations, attention_weights, output=None,
                   stream=None, options=0):
    """3-D variant: out[N, Len_q, M*D] from value [N,Len_in,M,D], spatial_shapes [L,3] (D,H,W),
    sampling_locations [N,Len_q,M,L,K,3] (x,y,z) and attention_weights [N,Len_q,M,L,K]."""
    lv = _HostVolumes(spatial_shapes, level_start_index)
    N, S, M, D = value.shape
    if sampling_locations.dim() != 6 or sampling_locations.shape[-1] != 3:
        raise ValueError("sampling_locations must be [N, Len_q, G, L, K, 3]")
    G = groups_of(value, sampling_locations)
    Lq, L, K = sampling_locations.shape[1], sampling_locations.shape[3], sampling_locations.shape[4]
    if tuple(sampling_locations.shape[:5]) != (N, Lq, G, L, K) or tuple(attention_weights.shape) != (N, Lq, G, L, K) \
            or L != lv.L:
        raise ValueError("attention_weights / spatial_shapes disagree with sampling_locations")
    _check_out(output, "output", (N, Lq, M * D), value.dtype)
    if output is None:
        output = torch.empty((N, Lq, M * D), dtype=value.dtype, device=value.device)
    prob = problem(value, Lq, L, K, options, G)
    _check(_lib.msda3d_forward(ctypes.byref(prob), _dev(value, "value"), lv.shp, lv.stp,
                               _dev(sampling_locations, "sampling_locations", torch.float32),
                               _dev(attention_weights, "attention_weights", torch.float32),
                               _dev(output, "output"), _stream(stream, value.device)))
    return output


@_on_value_device
def msda3d_backward(value, spatial_shapes, level_start_index, sampling_locations, attention_weights, grad_output,
                    grad_value=None, grad_sampling_locations=None, grad_attention_weights=None, flags=0,
                    workspace=None, stream=None, options=0):
    """3-D variant of msda_backward.  Returns (grad_value, grad_sampling_locations [..,3], grad_attention_weights)."""
    lv = _HostVolumes(spatial_shapes, level_start_index)
    N, S, M, D = value.shape
    Lq, L, K = _check_backward_args(value, lv.L, sampling_locations, attention_weights, grad_output, grad_value,
                                    grad_sampling_locations, grad_attention_weights, coords=3)
    dev = value.device
    grad_value = _grad_value_out(value, grad_value, flags)
    if grad_sampling_locations is None:
        grad_sampling_locations = torch.empty_like(sampling_locations)
    if grad_attention_weights is None:
        grad_attention_weights = torch.empty_like(attention_weights)
    prob = problem(value, Lq, L, K, options, sampling_locations.shape[2])
    need = int(_lib.msda_backward_workspace_size(ctypes.byref(prob), flags))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = _dev(workspace, "workspace") if workspace is not None else ctypes.c_void_p(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.msda3d_backward(ctypes.byref(prob), _dev(value, "value"), lv.shp, lv.stp,
                                _dev(sampling_locations, "sampling_locations", torch.float32),
                                _dev(attention_weights, "attention_weights", torch.float32),
                                _dev(grad_output, "grad_output"), _dev(grad_value, "grad_value", torch.float32),
                                _dev(grad_sampling_locations, "grad_sampling_locations", torch.float32),
                                _dev(grad_attention_weights, "grad_attention_weights", torch.float32),
                                flags, ws_ptr, ws_bytes, _stream(stream, dev)))
    return grad_value, grad_sampling_locations, grad_attention_weights
