"""Shared helpers of the parity tests: inputs of each call built from the
seeded raw draws, the oracle's answers, and the tolerance checks.

The oracle turns the raw draws into the inputs of the unfused calls
(locations from reference points and offsets, weights from logits); those
fp32 inputs then go to both sides unchanged.

Cell edges.  The oracle takes x0 = floor(px) on the fp64 pixel coordinate,
the kernels on a two-float representation of it; where px lies within
rounding of an integer the two may take neighbouring cells.  The output,
grad_attention_weights and grad_value are continuous across the edge, but the
location gradient is one-sided there and jumps: either side's derivative is
right.  The *_reference helpers flag every coordinate within EDGE_REL of an
integer, evaluate the oracle with those coordinates moved NUDGE_PX to either
side, keep per coordinate the side whose location gradient the GPU result
is closer to, and return the oracle's answer on that choice (all outputs of
one consistent oracle call).  Every other coordinate keeps its exact value.
"""
import numpy as np
import torch

import oracle
import workloads

# Tolerances (per tensor, normwise: rel = max|gpu - ref| / max|ref|)
FWD_F32_ABS = 1e-5
FWD_F32_REL = 1e-5
BWD_F32_REL = 1e-4
BF16_REL = 2e-2


# a coordinate is "at a cell edge" when |px - round(px)| <= EDGE_REL * (sum of
# the magnitudes of the terms that form px + 1): a few fp32 roundings of the
# error terms the kernels carry, far below one fp32 ulp of px
EDGE_REL = 2.0 ** -26
NUDGE_PX = 1e-6


def _axis_scales(spatial_shapes, options):
    """Per level and coordinate (x, y[, z]): the pixel scale S (size, or
    size - 1 with align_corners), the size, and the half-pixel shift."""
    sizes = np.asarray(spatial_shapes, dtype=np.float64)[:, ::-1]      # (W, H) or (W, H, D)
    align = bool(options & oracle.ALIGN_CORNERS)
    return (sizes - 1.0 if align else sizes), sizes, (0.0 if align else 0.5)


def edges_unfused(loc, spatial_shapes, options=0):
    """(mask, below, above) for sampling_locations [..., L, K, c]: mask marks the
    coordinates at a cell edge; below / above are float64 copies of loc with
    those coordinates moved NUDGE_PX pixels under / over the edge."""
    S, _, shift = _axis_scales(spatial_shapes, options)
    Sb = S[:, None, :]
    x = np.asarray(loc, dtype=np.float64)
    px = x * Sb - shift
    B = np.rint(px)
    mask = (np.abs(px - B) <= EDGE_REL * (np.abs(x * Sb) + 1.0)) & (Sb > 0)
    Sd = np.where(Sb > 0, Sb, 1.0)
    return mask, np.where(mask, (B - NUDGE_PX + shift) / Sd, x), np.where(mask, (B + NUDGE_PX + shift) / Sd, x)


def edges_fused(reference_points, sampling_offsets, spatial_shapes, options=0):
    """The same for the fused calls, on the offsets: px = ref * S + off * S / size
    - shift.  With align_corners the kernels scale the offset by S / size
    rounded to fp32, which widens the window by a relative 2^-23 of |off|."""
    S, sizes, shift = _axis_scales(spatial_shapes, options)
    Sb, Rb = S[:, None, :], (S / sizes)[:, None, :]
    r = np.asarray(reference_points, dtype=np.float64)[:, :, None, :, None, :]
    o = np.asarray(sampling_offsets, dtype=np.float64)
    px = r * Sb + o * Rb - shift
    B = np.rint(px)
    win = EDGE_REL * (np.abs(r * Sb) + np.abs(o * Rb) + 1.0)
    if options & oracle.ALIGN_CORNERS:
        win = win + 2.0 ** -23 * np.abs(o)
    mask = (np.abs(px - B) <= win) & (Sb > 0)
    Rd = np.where(Rb > 0, Rb, 1.0)
    return mask, np.where(mask, o + (B - NUDGE_PX - px) / Rd, o), np.where(mask, o + (B + NUDGE_PX - px) / Rd, o)


class BackwardReference:
    """Oracle reference for the outputs of one backward problem.  `call(x)`
    runs the oracle with the location-like input x (locations, or offsets for
    the fused call); output `which` of it is the location gradient that picks
    the side at each cell edge.  Oracle runs are cached, so several GPU results
    (atomic and deterministic mode, repeated calls) cost one run each side."""

    def __init__(self, call, x, edges, which):
        self.call, self.x, self.which = call, np.asarray(x, dtype=np.float64), which
        self.mask, self.below, self.above = edges
        self.edge_count = int(self.mask.sum())
        self._sides = None
        self._cache = {}

    def for_gpu(self, gpu):
        """The oracle's outputs for the GPU's outputs `gpu` (a sequence ordered
        like the oracle's)."""
        if not self.edge_count:
            key, x = b"", self.x
        else:
            if self._sides is None:
                self._sides = (self.call(self.below), self.call(self.above))
            lo, hi = self._sides
            g = np.asarray(gpu[self.which], dtype=np.float64).reshape(lo[self.which].shape)
            take_lo = self.mask & (np.abs(g - lo[self.which]) <= np.abs(g - hi[self.which]))
            key = take_lo[self.mask].tobytes()
            x = np.where(take_lo, self.below, np.where(self.mask, self.above, self.x))
        if key not in self._cache:
            self._cache[key] = self.call(x)
        return self._cache[key]


def backward_reference(p, options=0):
    """msda_backward: (grad_value, grad_sampling_locations, grad_attention_weights)."""
    sh, st = p["spatial_shapes"], p["level_start_index"]

    def call(loc):
        return oracle.backward(p["value"], sh, st, loc, p["attention_weights"], p["grad_output"], options=options)

    return BackwardReference(call, p["sampling_locations"], edges_unfused(p["sampling_locations"], sh, options), 1)


def backward3d_reference(p, options=0):
    """msda3d_backward (spatial_shapes [L,3], locations (x, y, z))."""
    sh, st = p["spatial_shapes"], p["level_start_index"]

    def call(loc):
        return oracle.backward3d(p["value"], sh, st, loc, p["attention_weights"], p["grad_output"], options=options)

    return BackwardReference(call, p["sampling_locations"], edges_unfused(p["sampling_locations"], sh, options), 1)


def backward_fused_reference(p, options=0):
    """msda_backward_fused: (grad_value, grad_reference_points,
    grad_sampling_offsets, grad_attention_logits); edges are resolved on the
    offsets, so the reference-point gradient sums the chosen sides."""
    sh, st = p["spatial_shapes"], p["level_start_index"]

    def call(off):
        return oracle.backward_fused(p["value"], sh, st, p["reference_points"], off, p["attention_logits"],
                                     p["grad_output"], options=options)

    edges = edges_fused(p["reference_points"], p["sampling_offsets"], sh, options)
    return BackwardReference(call, p["sampling_offsets"], edges, 2)


def bf16_round(a):
    """Round float32 to bfloat16 (RNE) and back, as stored on the device."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).to(torch.float32).numpy()


def unfused_inputs(w, raw):
    """sampling_locations and attention_weights (float32) of workload `w`."""
    L, K = w.L, w.K
    if "sampling_locations" in raw:
        loc = raw["sampling_locations"].astype(np.float32)
    else:
        loc = oracle.locations(raw["spatial_shapes"], raw["reference_points"], raw["sampling_offsets"]).astype(np.float32)
    shape = loc.shape[:-1]
    attn = oracle.softmax(raw["attention_logits"]).astype(np.float32).reshape(shape)
    return loc, attn


def prepared(w, raw=None, round_bf16=True):
    """All host inputs of workload `w` as float32 (value and grad_output already
    rounded to bf16 when the workload stores bf16, unless round_bf16 is False:
    the unrounded draws measure the storage error itself)."""
    raw = workloads.draw(w) if raw is None else raw
    loc, attn = unfused_inputs(w, raw)
    value, g = raw["value"], raw["grad_output"]
    if w.dtype == "bf16" and round_bf16:
        value, g = bf16_round(value), bf16_round(g)
    out = dict(raw)
    out.update(value=value, grad_output=g, sampling_locations=loc, attention_weights=attn)
    return out


def dev(a, dtype=torch.float32, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dtype).contiguous()


def storage_dtype(w):
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


def errors(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    if ref.size == 0:
        return 0.0, 0.0
    d = np.abs(gpu - ref)
    if not np.all(np.isfinite(gpu)):
        return float("inf"), float("inf")
    scale = max(float(np.abs(ref).max()), 1e-30)
    return float(d.max()), float(d.max()) / scale


def assert_fwd(gpu, ref, dtype, what="output"):
    ab, rel = errors(gpu, ref)
    if dtype == "bf16":
        assert rel <= BF16_REL, f"{what}: bf16 rel {rel:.3e} > {BF16_REL}"
    else:
        assert ab <= FWD_F32_ABS and rel <= FWD_F32_REL, f"{what}: abs {ab:.3e} rel {rel:.3e} > 1e-5"
    return ab, rel


def assert_bwd(gpu, ref, dtype, what):
    ab, rel = errors(gpu, ref)
    tol = BF16_REL if dtype == "bf16" else BWD_F32_REL
    assert rel <= tol, f"{what}: rel {rel:.3e} > {tol} (abs {ab:.3e})"
    return ab, rel


RANDOM_PROBLEMS = 64


def random_problem(i):
    """Seeded random problem i of the randomized parity tests: (workload,
    options, head groups G).
    Head width 8-256, 1-8 heads, 1-5 levels of 1-12 x 1-12 pixels, 1-8 points,
    Len_q either every pixel (pixel-centre references) or 1-69 random queries,
    either dtype, any option combination, any head grouping the kernels take."""
    r = np.random.default_rng(5000 + i)
    D = int(r.choice([8, 16, 32, 64, 128, 256]))
    M = int(r.choice([m for m in (1, 2, 3, 4, 8) if m * D <= 1024]))
    L = int(r.integers(1, 6))
    K = int(r.integers(1, 9))
    levels = [(int(r.integers(1, 13)), int(r.integers(1, 13))) for _ in range(L)]
    pixel_queries = bool(r.integers(0, 2))
    w = workloads.custom(N=int(r.integers(1, 4)), M=M, D=D, levels=levels, K=K,
                         Len_q=-1 if pixel_queries else int(r.integers(1, 70)),
                         dtype=str(r.choice(["f32", "bf16"])), refs="pixel_centres" if pixel_queries else "uniform",
                         ref_range=(-0.05, 1.05), offset_sigma=float(r.choice([0.05, 0.2])), seed=6000 + i)
    opt = int(r.integers(0, 4))
    # head groups: G sets shared by M / G heads each, where the group width
    # (M / G) * D is a power of two the kernels take (G = M half the time)
    widths = {8, 16, 32, 64, 128, 256}
    Gs = [g for g in range(1, M + 1) if M % g == 0 and (M // g) * D in widths]
    G = M if r.integers(0, 2) == 0 else int(r.choice(Gs))
    return w, opt, G


PER_SAMPLE = ("sampling_locations", "attention_weights", "sampling_offsets", "attention_logits")


def grouped(p, G):
    """The inputs cut to G sets of locations and weights: the per-sample tensors
    keep their first G heads' sets, shared by groups of M / G heads."""
    return {k: (np.ascontiguousarray(v[:, :, :G]) if k in PER_SAMPLE else v) for k, v in p.items()}


RANDOM_VOLUMES = 24


def random_volume_problem(i):
    """Seeded random 3-D problem i: (raw draws, value, grad_output, attention
    weights, dtype, options).  Head width 8-64, 1-4 heads, 1-4 levels of 1-6
    frames x 1-6 rows x 1-6 columns, 1-6 points, 1-60 queries, locations over
    [-0.15, 1.15]^3, either dtype, align_corners or not."""
    r = np.random.default_rng(7000 + i)
    D = int(r.choice([8, 16, 32, 64]))
    M, L, K = int(r.integers(1, 5)), int(r.integers(1, 5)), int(r.integers(1, 7))
    levels = [tuple(int(x) for x in r.integers(1, 7, size=3)) for _ in range(L)]
    N, Lq = int(r.integers(1, 4)), int(r.integers(1, 61))
    dtype, opt = str(r.choice(["f32", "bf16"])), int(r.choice([0, 2]))
    raw = workloads.draw_volumes(N, M, D, levels, K, Lq, dtype=dtype, loc_range=(-0.15, 1.15), seed=7500 + i)
    attn = oracle.softmax(raw["attention_logits"]).astype(np.float32).reshape(N, Lq, M, L, K)
    value, g = raw["value"], raw["grad_output"]
    if dtype == "bf16":
        value, g = bf16_round(value), bf16_round(g)
    return raw, value, g, attn, dtype, opt


def check_3d_calls(msda, case, what):
    """msda3d_forward and msda3d_backward (both modes) of a 3-D case against the oracle."""
    raw, value, g, attn, dtype, opt = case
    sh, st, loc = raw["spatial_shapes"], raw["level_start_index"], raw["sampling_locations"]
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    v, gd, locd, ad = dev(value, dt), dev(g, dt), dev(loc), dev(attn)
    out = msda.msda3d_forward(v, sh, st, locd, ad, options=opt).float().cpu().numpy()
    assert_fwd(out, oracle.forward3d(value, sh, st, loc, attn, options=opt), dtype, what + " forward")
    ref = backward3d_reference(dict(value=value, spatial_shapes=sh, level_start_index=st, sampling_locations=loc,
                                    attention_weights=attn, grad_output=g), opt)
    for flags in (0, msda.MSDA_DETERMINISTIC):
        got = [t.cpu().numpy() for t in msda.msda3d_backward(v, sh, st, locd, ad, gd, flags=flags, options=opt)]
        for nm, a, b in zip(("grad_value", "grad_loc", "grad_attn"), got, ref.for_gpu(got)):
            assert_bwd(a, b, "f32", f"{what} {nm} flags {flags}")
