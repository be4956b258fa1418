"""fp64 CPU oracle for the MSDeformAttn core -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and the two share no
code.  The arithmetic lives in ``msda_oracle.c`` (plain single-threaded C,
double precision); this module only marshals numpy arrays to it.

Every function takes and returns float64 numpy arrays in the layouts listed
at the top of ``msda_oracle.c``; spatial_shapes / level_start_index are
int64.  Inputs given in float32 or bfloat16-rounded float32 are upcast
exactly.
"""
import ctypes

import numpy as np

from . import build as _build

_lib = None


def bind(path):
    """Load an oracle shared library at `path` and declare its C signatures."""
    lib = ctypes.CDLL(path)
    i64 = ctypes.c_int64
    dp = ctypes.POINTER(ctypes.c_double)
    lp = ctypes.POINTER(ctypes.c_int64)
    lib.msda_oracle_locations.argtypes = [i64] * 5 + [lp, dp, dp, dp]
    lib.msda_oracle_softmax.argtypes = [i64, i64, dp, dp]
    lib.msda_oracle_forward.argtypes = [i64] * 7 + [dp, lp, lp, dp, dp, dp, i64]
    lib.msda_oracle_forward_fused.argtypes = [i64] * 7 + [dp, lp, lp, dp, dp, dp, dp, i64]
    lib.msda_oracle_backward.argtypes = [i64] * 7 + [dp, lp, lp, dp, dp, dp, dp, dp, dp, i64]
    lib.msda_oracle_backward_fused.argtypes = [i64] * 7 + [dp, lp, lp, dp, dp, dp, dp, dp, dp, dp, dp, i64]
    lib.msda_oracle_forward3d.argtypes = [i64] * 7 + [dp, lp, lp, dp, dp, dp, i64]
    lib.msda_oracle_backward3d.argtypes = [i64] * 7 + [dp, lp, lp, dp, dp, dp, dp, dp, dp, i64]
    lib.msda_oracle_forward_grouped.argtypes = [i64] * 8 + [dp, lp, lp, dp, dp, dp, i64]
    lib.msda_oracle_forward_fused_grouped.argtypes = [i64] * 8 + [dp, lp, lp, dp, dp, dp, dp, i64]
    lib.msda_oracle_backward_grouped.argtypes = [i64] * 8 + [dp, lp, lp, dp, dp, dp, dp, dp, dp, i64]
    lib.msda_oracle_backward_fused_grouped.argtypes = [i64] * 8 + [dp, lp, lp, dp, dp, dp, dp, dp, dp, dp, dp, i64]
    for f in ("msda_oracle_locations", "msda_oracle_softmax", "msda_oracle_forward",
              "msda_oracle_forward_fused", "msda_oracle_backward", "msda_oracle_backward_fused",
              "msda_oracle_forward3d", "msda_oracle_backward3d", "msda_oracle_forward_grouped",
              "msda_oracle_forward_fused_grouped", "msda_oracle_backward_grouped",
              "msda_oracle_backward_fused_grouped"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


def use_library(lib):
    """Route the module-level functions to `lib` (None: the built oracle).
    Tests use this to run the pins against a deliberately broken copy."""
    global _lib
    _lib = lib


def _load():
    global _lib
    if _lib is None:
        _lib = bind(_build.build())
    return _lib


def _d(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _l(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int64))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name}: the oracle rejected its arguments")


def _dims(value, shapes, loc_like):
    """(N, Len_in, M, D, Len_q, L, K, G) from value [N,S,M,D] and a per-sample tensor
    [N,Lq,G,L,K,...]: G = M (one set of locations per head), or the number of
    head groups that share one set each."""
    N, S, M, D = value.shape
    L = shapes.shape[0]
    Lq, G, K = loc_like.shape[1], loc_like.shape[2], loc_like.shape[4]
    return N, S, M, D, Lq, L, K, G


# option bits of the forward and backward functions (msda_oracle.c header)
PER_LEVEL_SOFTMAX = 1   # the fused calls normalise each level's n_points logits separately
ALIGN_CORNERS = 2       # px = loc * (W - 1) instead of loc * W - 0.5


def locations(spatial_shapes, reference_points, sampling_offsets):
    """a1: loc = ref + off / (W_l, H_l); offsets in pixels of their level."""
    lib = _load()
    sh, shp = _l(spatial_shapes)
    ref, refp = _d(reference_points)
    off, offp = _d(sampling_offsets)
    N, Lq, M, L, K, _ = off.shape
    out = np.empty_like(off)
    _check(lib.msda_oracle_locations(N, Lq, M, L, K, shp, refp, offp, _d(out)[1]), "locations")
    return out


def softmax(logits):
    """a2: softmax over the last axis (the n_levels*n_points samples of one query-head)."""
    lib = _load()
    x, xp = _d(logits)
    cols = x.shape[-1]
    rows = x.size // cols if cols else 0
    out = np.empty_like(x)
    _check(lib.msda_oracle_softmax(rows, cols, xp, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double))),
           "softmax")
    return out


def forward(value, spatial_shapes, level_start_index, sampling_locations, attention_weights, options=0):
    """a3-a5.  Returns output [N, Len_q, M*D] in float64.  sampling_locations is
    [N, Len_q, G, L, K, 2] with G = M, or G groups of M / G heads sharing a set
    (attention_weights likewise); so are the per-sample arguments below."""
    lib = _load()
    v, vp = _d(value)
    sh, shp = _l(spatial_shapes)
    st, stp = _l(level_start_index)
    loc, locp = _d(sampling_locations)
    a, ap = _d(attention_weights)
    N, S, M, D, Lq, L, K, G = _dims(v, sh, loc)
    out = np.zeros((N, Lq, M * D))
    _check(lib.msda_oracle_forward_grouped(N, S, M, G, D, Lq, L, K, vp, shp, stp, locp, ap, _d(out)[1], options),
           "forward")
    return out


def forward_fused(value, spatial_shapes, level_start_index, reference_points, sampling_offsets,
                  attention_logits, options=0):
    """a1-a5.  attention_logits is [N, Len_q, M, L*K] (or [N,Lq,M,L,K])."""
    lib = _load()
    v, vp = _d(value)
    sh, shp = _l(spatial_shapes)
    st, stp = _l(level_start_index)
    ref, refp = _d(reference_points)
    off, offp = _d(sampling_offsets)
    lg, lgp = _d(attention_logits)
    N, S, M, D, Lq, L, K, G = _dims(v, sh, off)
    out = np.zeros((N, Lq, M * D))
    _check(lib.msda_oracle_forward_fused_grouped(N, S, M, G, D, Lq, L, K, vp, shp, stp, refp, offp, lgp,
                                                 _d(out)[1], options), "forward_fused")
    return out


def backward(value, spatial_shapes, level_start_index, sampling_locations, attention_weights, grad_output,
             options=0):
    """a6-a8.  Returns (grad_value [N,S,M,D], grad_loc [N,Lq,M,L,K,2], grad_attn [N,Lq,M,L,K])."""
    lib = _load()
    v, vp = _d(value)
    sh, shp = _l(spatial_shapes)
    st, stp = _l(level_start_index)
    loc, locp = _d(sampling_locations)
    a, ap = _d(attention_weights)
    g, gp = _d(grad_output)
    N, S, M, D, Lq, L, K, G = _dims(v, sh, loc)
    gv = np.zeros(v.shape)
    gl = np.zeros(loc.shape)
    ga = np.zeros(a.shape)
    _check(lib.msda_oracle_backward_grouped(N, S, M, G, D, Lq, L, K, vp, shp, stp, locp, ap, gp,
                                            _d(gv)[1], _d(gl)[1], _d(ga)[1], options), "backward")
    return gv, gl, ga


def backward_fused(value, spatial_shapes, level_start_index, reference_points, sampling_offsets,
                   attention_logits, grad_output, options=0):
    """a9.  Returns (grad_value, grad_reference_points, grad_sampling_offsets, grad_attention_logits)."""
    lib = _load()
    v, vp = _d(value)
    sh, shp = _l(spatial_shapes)
    st, stp = _l(level_start_index)
    ref, refp = _d(reference_points)
    off, offp = _d(sampling_offsets)
    lg, lgp = _d(attention_logits)
    g, gp = _d(grad_output)
    N, S, M, D, Lq, L, K, G = _dims(v, sh, off)
    gv = np.zeros(v.shape)
    gr = np.zeros(ref.shape)
    go = np.zeros(off.shape)
    gl = np.zeros(lg.shape)
    _check(lib.msda_oracle_backward_fused_grouped(N, S, M, G, D, Lq, L, K, vp, shp, stp, refp, offp, lgp, gp,
                                                  _d(gv)[1], _d(gr)[1], _d(go)[1], _d(gl)[1], options),
           "backward_fused")
    return gv, gr, go, gl



def forward3d(value, spatial_shapes, level_start_index, sampling_locations, attention_weights, options=0):
    """3-D variant, a3-a5 with trilinear sampling.  spatial_shapes [L,3] = (D,H,W),
    sampling_locations [N,Lq,M,L,K,3] (x,y,z).  Returns output [N, Len_q, M*D]."""
    lib = _load()
    v, vp = _d(value)
    sh, shp = _l(np.asarray(spatial_shapes).reshape(-1, 3))
    st, stp = _l(level_start_index)
    loc, locp = _d(sampling_locations)
    a, ap = _d(attention_weights)
    N, S, M, D = v.shape
    Lq, L, K = loc.shape[1], sh.shape[0], loc.shape[4]
    out = np.zeros((N, Lq, M * D))
    _check(lib.msda_oracle_forward3d(N, S, M, D, Lq, L, K, vp, shp, stp, locp, ap, _d(out)[1], options),
           "forward3d")
    return out


def backward3d(value, spatial_shapes, level_start_index, sampling_locations, attention_weights, grad_output,
               options=0):
    """3-D variant of a6-a8.  Returns (grad_value, grad_loc [..,3], grad_attn)."""
    lib = _load()
    v, vp = _d(value)
    sh, shp = _l(np.asarray(spatial_shapes).reshape(-1, 3))
    st, stp = _l(level_start_index)
    loc, locp = _d(sampling_locations)
    a, ap = _d(attention_weights)
    g, gp = _d(grad_output)
    N, S, M, D = v.shape
    Lq, L, K = loc.shape[1], sh.shape[0], loc.shape[4]
    gv = np.zeros(v.shape)
    gl = np.zeros(loc.shape)
    ga = np.zeros(a.shape)
    _check(lib.msda_oracle_backward3d(N, S, M, D, Lq, L, K, vp, shp, stp, locp, ap, gp,
                                      _d(gv)[1], _d(gl)[1], _d(ga)[1], options), "backward3d")
    return gv, gl, ga
