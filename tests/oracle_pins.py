"""Pins of the fp64 oracle to facts other than itself.

Each pin returns (error, tolerance).  They are used twice: on the built oracle
(every pin must hold) and on deliberately broken copies of it
(test_oracle_mutants.py: at least one pin must fail for every planted bug).

What pins what:
  worked_example      step a1 against the worked example printed in the
                      Deformable DETR deployment notes, section 2.2, run both
                      through the location step and through the fused forward.
  softmax_closed      step a2: softmax(log[1,2,3,4]) = [.1,.2,.3,.4], overflow-safe
                      at logits 1000/1001, zero logits give 1/(L*K).
  constant_map        steps a3-a5: a constant map c returns
                      c * sum_s A_s * s(px) * s(py), s(p) = max(0, min(1, p+1, size-p)).
  pixel_centres       sampling at pixel centres is a pure gather.
  linear_ramp         a map linear in (x, y) is reproduced exactly inside the map.
  far_outside         samples far outside every level give exactly 0.
  grid_sample         torch.nn.functional.grid_sample (bilinear, zeros,
                      align_corners=False) in float64 on the CPU, one call per
                      level as in the tutorial's module, agrees to 1e-12.
  dense_tent          out = Wmat @ value with Wmat built from the tent form
                      max(0,1-|px-x|) max(0,1-|py-y|) over every pixel.
  backward_autograd   steps a6-a8 against torch autograd through grid_sample.
  backward_fd         central finite differences of the oracle forward.
  adjoint             <grad_value, dV> = <g, forward(dV)> (the forward is linear in value).
  fused_*             a9 and the fused forward: finite differences through
                      a1-a2, sum of logit gradients is 0, composition with a1/a2.
  grouped_*           locations and weights shared by a group of heads (the DAT
                      pages' sampler): the per-head call on the sets broadcast
                      to every head, gradients summed over each group (forward,
                      backward, fused forward and backward); and the plain call
                      on value viewed as G heads of (M / G) * D channels.
  align_*             the align_corners option (px = loc * (W - 1)): torch
                      grid_sample(align_corners=True) forward and autograd in
                      float64, and exact gathers at loc = i / (W - 1).
  per_level_*         the per-level softmax option: logits = log p with each
                      level's p summing to 1 give A = p; a constant added to one
                      level's logits changes nothing (it would change the
                      whole-row softmax); with one level it equals the whole-row
                      softmax; finite differences of the fused backward and
                      zero-sum logit gradients per level.
  trilinear_*         the 3-D variant: torch grid_sample on 5-D volumes (trilinear,
                      zeros, both align_corners settings) forward and autograd in
                      float64; one-slice volumes sampled at their centre plane
                      give the 2-D result; finite differences.
"""
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        return math.inf
    if a.size == 0:
        return 0.0
    d = np.abs(a - b)
    if not np.all(np.isfinite(d)):
        return math.inf
    return float(d.max())


def _rel(a, b):
    scale = max(float(np.abs(np.asarray(b)).max()), 1e-300) if np.asarray(b).size else 1.0
    return _err(a, b) / scale


def _tiny(seed=7, loc_lo=-0.1, loc_hi=1.1, levels=((8, 8), (4, 4)), N=1, M=2, D=8, Lq=20, K=2):
    rng = np.random.Generator(np.random.PCG64(seed))
    shapes = np.asarray(levels, dtype=np.int64)
    starts = workloads.level_start_index(shapes)
    S = int((shapes[:, 0] * shapes[:, 1]).sum())
    L = len(levels)
    value = rng.standard_normal((N, S, M, D))
    loc = rng.uniform(loc_lo, loc_hi, size=(N, Lq, M, L, K, 2))
    attn = oracle.softmax(rng.standard_normal((N, Lq, M, L * K))).reshape(N, Lq, M, L, K)
    g = rng.standard_normal((N, Lq, M * D))
    return dict(value=value, shapes=shapes, starts=starts, loc=loc, attn=attn, g=g,
                N=N, S=S, M=M, D=D, Lq=Lq, L=L, K=K)


def _px(loc, size):
    return loc * size - 0.5


# --------------------------------------------------------------------------- a1
def read_worked_example():
    rows = []
    with open(os.path.join(GOLDEN, "worked_example_locations.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([float(t) for t in line.split()])
    return np.asarray(rows)


def pin_worked_example():
    rows = read_worked_example()
    worst = 0.0
    for (H, W) in [(100, 167), (13, 21), (1, 1), (64, 64)]:
        shapes = np.asarray([[H, W]], dtype=np.int64)
        ref = np.zeros((1, 1, 1, 2))
        ref[0, 0, 0] = rows[0, 0:2]
        off = np.zeros((1, 1, 1, 1, 4, 2))
        off[0, 0, 0, 0, :, 0] = rows[:, 2] * W
        off[0, 0, 0, 0, :, 1] = rows[:, 3] * H
        loc = oracle.locations(shapes, ref, off)
        worst = max(worst, _err(loc[0, 0, 0, 0], rows[:, 4:6]))
    # the same points seen through the fused forward: a ramp map whose two
    # channels are the pixel column and row, one sample at a time (A = 1)
    H, W = 100, 167
    shapes = np.asarray([[H, W]], dtype=np.int64)
    ys, xs = np.meshgrid(np.arange(H), np.arange(W), indexing="ij")
    value = np.stack([xs.ravel(), ys.ravel()], axis=-1).astype(np.float64)[None, :, None, :]
    for r in rows:
        ref = np.asarray(r[0:2]).reshape(1, 1, 1, 2)
        off = np.asarray([r[2] * W, r[3] * H]).reshape(1, 1, 1, 1, 1, 2)
        out = oracle.forward_fused(value, shapes, np.zeros(1, np.int64), ref, off, np.zeros((1, 1, 1, 1)))
        got = np.asarray([(out[0, 0, 0] + 0.5) / W, (out[0, 0, 1] + 0.5) / H])
        worst = max(worst, _err(got, r[4:6]))
    return worst, 1e-12


# --------------------------------------------------------------------------- a2
def pin_softmax_closed():
    worst = _err(oracle.softmax(np.log([[1.0, 2.0, 3.0, 4.0]])), [[0.1, 0.2, 0.3, 0.4]])
    e = math.e
    worst = max(worst, _err(oracle.softmax(np.asarray([[1000.0, 1001.0]])), [[1 / (1 + e), e / (1 + e)]]))
    worst = max(worst, _err(oracle.softmax(np.zeros((3, 16))), np.full((3, 16), 1 / 16)))
    x = np.random.Generator(np.random.PCG64(3)).standard_normal((5, 12))
    worst = max(worst, _err(oracle.softmax(x + 37.25), oracle.softmax(x)))
    return worst, 1e-14


# --------------------------------------------------------------------------- a3-a5
def _coverage(p, size):
    return np.maximum(0.0, np.minimum(np.minimum(1.0, p + 1.0), size - p))


def pin_constant_map():
    t = _tiny(seed=11, loc_lo=-0.6, loc_hi=1.6, levels=((8, 8), (4, 4), (1, 5), (3, 1)), Lq=40, K=3)
    c = 1.7
    value = np.full_like(t["value"], c)
    out = oracle.forward(value, t["shapes"], t["starts"], t["loc"], t["attn"])
    expect = np.zeros((t["N"], t["Lq"], t["M"]))
    for l, (H, W) in enumerate(t["shapes"]):
        sx = _coverage(_px(t["loc"][..., l, :, 0], W), W)
        sy = _coverage(_px(t["loc"][..., l, :, 1], H), H)
        expect += c * (t["attn"][..., l, :] * sx * sy).sum(-1)
    expect = np.repeat(expect[..., None], t["D"], axis=-1).reshape(t["N"], t["Lq"], -1)
    return _err(out, expect), 1e-12


def pin_pixel_centres():
    t = _tiny(seed=12, levels=((8, 8), (4, 4), (2, 7)), Lq=30, K=3)
    rng = np.random.Generator(np.random.PCG64(5))
    loc = np.zeros_like(t["loc"])
    expect = np.zeros((t["N"], t["Lq"], t["M"], t["D"]))
    for l, (H, W) in enumerate(t["shapes"]):
        i = rng.integers(0, W, size=loc.shape[:3] + (t["K"],))
        j = rng.integers(0, H, size=loc.shape[:3] + (t["K"],))
        loc[..., l, :, 0] = (i + 0.5) / W
        loc[..., l, :, 1] = (j + 0.5) / H
        for n in range(t["N"]):
            for q in range(t["Lq"]):
                for m in range(t["M"]):
                    for k in range(t["K"]):
                        row = t["starts"][l] + j[n, q, m, k] * W + i[n, q, m, k]
                        expect[n, q, m] += t["attn"][n, q, m, l, k] * t["value"][n, row, m]
    out = oracle.forward(t["value"], t["shapes"], t["starts"], loc, t["attn"])
    return _err(out, expect.reshape(out.shape)), 1e-12


def pin_linear_ramp():
    t = _tiny(seed=13, levels=((8, 8), (4, 6), (5, 2)), Lq=30, K=3, M=3, D=4)
    rng = np.random.Generator(np.random.PCG64(6))
    L, M, D = t["L"], t["M"], t["D"]
    alpha, beta, gamma = (rng.standard_normal((L, M, D)) for _ in range(3))
    value = np.zeros_like(t["value"])
    loc = np.zeros_like(t["loc"])
    expect = np.zeros((t["N"], t["Lq"], M, D))
    for l, (H, W) in enumerate(t["shapes"]):
        ys, xs = np.meshgrid(np.arange(H), np.arange(W), indexing="ij")
        lvl = (alpha[l][None] * xs.ravel()[:, None, None] + beta[l][None] * ys.ravel()[:, None, None]
               + gamma[l][None])
        value[:, t["starts"][l]:t["starts"][l] + H * W] = lvl[None]
        # keep all four corners inside: px in [0, W-1], py in [0, H-1]
        loc[..., l, :, 0] = (rng.uniform(0, W - 1, size=loc.shape[:3] + (t["K"],)) + 0.5) / W
        loc[..., l, :, 1] = (rng.uniform(0, H - 1, size=loc.shape[:3] + (t["K"],)) + 0.5) / H
        px = _px(loc[..., l, :, 0], W)
        py = _px(loc[..., l, :, 1], H)
        A = t["attn"][..., l, :]
        expect += np.einsum("nqmk,md->nqmd", A * px, alpha[l]) + np.einsum("nqmk,md->nqmd", A * py, beta[l]) \
            + np.einsum("nqmk,md->nqmd", A, gamma[l])
    out = oracle.forward(value, t["shapes"], t["starts"], loc, t["attn"])
    return _err(out, expect.reshape(out.shape)), 1e-11


def pin_far_outside():
    t = _tiny(seed=14)
    loc = t["loc"].copy()
    far = np.asarray([[-5.0, 0.5], [2.0, 0.5], [0.5, -3.0], [0.5, 7.0], [-1.0, -1.0], [9.0, 9.0]])
    idx = np.arange(loc[..., 0].size) % len(far)
    loc.reshape(-1, 2)[:] = far[idx]
    out = oracle.forward(t["value"], t["shapes"], t["starts"], loc, t["attn"])
    return float(np.abs(out).max()), 0.0


def _grid_sample_forward(value, shapes, starts, loc, attn, align_corners=False):
    """The tutorial module's per-level grid_sample path, in float64 torch."""
    N, S, M, D = value.shape
    _, Lq, _, L, K, _ = loc.shape
    out = 0
    for l in range(L):
        H, W = int(shapes[l, 0]), int(shapes[l, 1])
        s0 = int(starts[l])
        v_l = value[:, s0:s0 + H * W].reshape(N, H, W, M, D).permute(0, 3, 4, 1, 2).reshape(N * M, D, H, W)
        grid = (2.0 * loc[:, :, :, l] - 1.0).permute(0, 2, 1, 3, 4).reshape(N * M, Lq, K, 2)
        smp = F.grid_sample(v_l, grid, mode="bilinear", padding_mode="zeros", align_corners=align_corners)
        a = attn[:, :, :, l].permute(0, 2, 1, 3).reshape(N * M, 1, Lq, K)
        out = out + (smp * a).sum(-1)                       # (N*M, D, Lq)
    return out.reshape(N, M, D, Lq).permute(0, 3, 1, 2).reshape(N, Lq, M * D)


def pin_grid_sample():
    worst = 0.0
    for seed, lv in [(15, ((8, 8), (4, 4))), (16, ((5, 9), (3, 2), (1, 1)))]:
        t = _tiny(seed=seed, levels=lv, loc_lo=-0.3, loc_hi=1.3, Lq=25, K=3, M=3, D=5)
        out = oracle.forward(t["value"], t["shapes"], t["starts"], t["loc"], t["attn"])
        ref = _grid_sample_forward(torch.from_numpy(t["value"]), t["shapes"], t["starts"],
                                   torch.from_numpy(t["loc"]), torch.from_numpy(t["attn"])).numpy()
        worst = max(worst, _err(out, ref))
    return worst, 1e-12


def pin_dense_tent():
    t = _tiny(seed=17, levels=((6, 7), (3, 4)), loc_lo=-0.2, loc_hi=1.2, Lq=15, K=3, M=2, D=3)
    out = oracle.forward(t["value"], t["shapes"], t["starts"], t["loc"], t["attn"])
    N, Lq, M = t["N"], t["Lq"], t["M"]
    expect = np.zeros((N, Lq, M, t["D"]))
    for n in range(N):
        for m in range(M):
            Wmat = np.zeros((Lq, t["S"]))
            for l, (H, W) in enumerate(t["shapes"]):
                ys, xs = np.meshgrid(np.arange(H), np.arange(W), indexing="ij")
                cols = t["starts"][l] + ys.ravel() * W + xs.ravel()
                for q in range(Lq):
                    for k in range(t["K"]):
                        px = _px(t["loc"][n, q, m, l, k, 0], W)
                        py = _px(t["loc"][n, q, m, l, k, 1], H)
                        tent = np.maximum(0, 1 - np.abs(px - xs.ravel())) * np.maximum(0, 1 - np.abs(py - ys.ravel()))
                        Wmat[q, cols] += t["attn"][n, q, m, l, k] * tent
            expect[n, :, m] = Wmat @ t["value"][n, :, m]
    return _err(out, expect.reshape(out.shape)), 1e-12


# --------------------------------------------------------------------------- a6-a8
def pin_backward_autograd():
    t = _tiny(seed=18, levels=((8, 8), (4, 4), (3, 5)), loc_lo=-0.2, loc_hi=1.2, Lq=20, K=2, M=2, D=4)
    v = torch.from_numpy(t["value"]).requires_grad_(True)
    loc = torch.from_numpy(t["loc"]).requires_grad_(True)
    a = torch.from_numpy(t["attn"]).requires_grad_(True)
    out = _grid_sample_forward(v, t["shapes"], t["starts"], loc, a)
    out.backward(torch.from_numpy(t["g"]))
    gv, gl, ga = oracle.backward(t["value"], t["shapes"], t["starts"], t["loc"], t["attn"], t["g"])
    # grid_sample's grid lives in [-1,1]: d grid / d loc = 2 is inside autograd already
    worst = max(_rel(gv, v.grad.numpy()), _rel(gl, loc.grad.numpy()), _rel(ga, a.grad.numpy()))
    return worst, 1e-12


def _near_kink(loc, shapes, margin):
    """Mask of samples whose pixel coordinate is within `margin` of an integer."""
    bad = np.zeros(loc.shape[:-1], dtype=bool)
    for l, (H, W) in enumerate(shapes):
        for c, size in ((0, W), (1, H)):
            p = _px(loc[..., l, :, c], size)
            bad[..., l, :] |= np.abs(p - np.round(p)) < margin
    return bad


def pin_backward_fd():
    t = _tiny(seed=19, levels=((8, 8), (4, 4)), loc_lo=-0.15, loc_hi=1.15, Lq=6, K=2, M=2, D=3)
    gv, gl, ga = oracle.backward(t["value"], t["shapes"], t["starts"], t["loc"], t["attn"], t["g"])

    def J(value=None, loc=None, attn=None):
        out = oracle.forward(t["value"] if value is None else value, t["shapes"], t["starts"],
                             t["loc"] if loc is None else loc, t["attn"] if attn is None else attn)
        return float((out * t["g"]).sum())

    h = 1e-6
    worst = 0.0
    kink = _near_kink(t["loc"], t["shapes"], 1e-3)
    for idx in np.ndindex(t["loc"].shape):
        if kink[idx[:-1]]:
            continue
        p, m = t["loc"].copy(), t["loc"].copy()
        p[idx] += h
        m[idx] -= h
        fd = (J(loc=p) - J(loc=m)) / (2 * h)
        worst = max(worst, abs(fd - gl[idx]) / (1 + abs(gl[idx])))
    for idx in list(np.ndindex(t["attn"].shape))[:24]:
        p, m = t["attn"].copy(), t["attn"].copy()
        p[idx] += h
        m[idx] -= h
        worst = max(worst, abs((J(attn=p) - J(attn=m)) / (2 * h) - ga[idx]) / (1 + abs(ga[idx])))
    rng = np.random.Generator(np.random.PCG64(20))
    for _ in range(40):
        idx = tuple(int(rng.integers(0, s)) for s in t["value"].shape)
        p, m = t["value"].copy(), t["value"].copy()
        p[idx] += h
        m[idx] -= h
        worst = max(worst, abs((J(value=p) - J(value=m)) / (2 * h) - gv[idx]) / (1 + abs(gv[idx])))
    return worst, 1e-6


def pin_adjoint():
    t = _tiny(seed=21, levels=((8, 8), (4, 4), (2, 3)), Lq=30, K=3, M=2, D=4)
    gv, _, _ = oracle.backward(t["value"], t["shapes"], t["starts"], t["loc"], t["attn"], t["g"])
    dV = np.random.Generator(np.random.PCG64(22)).standard_normal(t["value"].shape)
    lhs = float((gv * dV).sum())
    rhs = float((t["g"] * oracle.forward(dV, t["shapes"], t["starts"], t["loc"], t["attn"])).sum())
    return abs(lhs - rhs) / max(1.0, abs(rhs)), 1e-12


# --------------------------------------------------------------------------- fused
def _fused_inputs(seed, levels=((8, 8), (4, 4), (3, 5)), N=1, Lq=8, M=2, K=2, D=3):
    rng = np.random.Generator(np.random.PCG64(seed))
    shapes = np.asarray(levels, dtype=np.int64)
    starts = workloads.level_start_index(shapes)
    S = int((shapes[:, 0] * shapes[:, 1]).sum())
    L = len(levels)
    ref = rng.uniform(0.1, 0.9, size=(N, Lq, L, 2))
    scale = np.asarray([[w, h] for (h, w) in levels], dtype=np.float64)
    off = rng.standard_normal((N, Lq, M, L, K, 2)) * 0.2 * scale[None, None, None, :, None, :]
    logits = rng.standard_normal((N, Lq, M, L * K))
    value = rng.standard_normal((N, S, M, D))
    g = rng.standard_normal((N, Lq, M * D))
    return dict(shapes=shapes, starts=starts, ref=ref, off=off, logits=logits, value=value, g=g)


def pin_fused_composition():
    f = _fused_inputs(23, Lq=12, M=3, K=3, D=4)
    out = oracle.forward_fused(f["value"], f["shapes"], f["starts"], f["ref"], f["off"], f["logits"])
    loc = oracle.locations(f["shapes"], f["ref"], f["off"])
    attn = oracle.softmax(f["logits"]).reshape(f["off"].shape[:-1])
    ref_out = _grid_sample_forward(torch.from_numpy(f["value"]), f["shapes"], f["starts"],
                                   torch.from_numpy(loc), torch.from_numpy(attn)).numpy()
    worst = _err(out, ref_out)
    # zero logits: uniform weights 1/(L*K) (zero-initialised weight branch)
    out0 = oracle.forward_fused(f["value"], f["shapes"], f["starts"], f["ref"], f["off"],
                                np.zeros_like(f["logits"]))
    uni = np.full(attn.shape, 1.0 / f["logits"].shape[-1])
    worst = max(worst, _err(out0, oracle.forward(f["value"], f["shapes"], f["starts"], loc, uni)))
    return worst, 1e-12


def pin_fused_backward():
    f = _fused_inputs(24)
    gv, gr, go, gl = oracle.backward_fused(f["value"], f["shapes"], f["starts"], f["ref"], f["off"],
                                           f["logits"], f["g"])

    def J(ref=None, off=None, logits=None):
        out = oracle.forward_fused(f["value"], f["shapes"], f["starts"], f["ref"] if ref is None else ref,
                                   f["off"] if off is None else off, f["logits"] if logits is None else logits)
        return float((out * f["g"]).sum())

    h = 1e-6
    worst = 0.0
    loc = oracle.locations(f["shapes"], f["ref"], f["off"])
    kink = _near_kink(loc, f["shapes"], 1e-3)
    for idx in np.ndindex(f["off"].shape):
        if kink[idx[:-1]]:
            continue
        p, m = f["off"].copy(), f["off"].copy()
        p[idx] += h
        m[idx] -= h
        worst = max(worst, abs((J(off=p) - J(off=m)) / (2 * h) - go[idx]) / (1 + abs(go[idx])))
    for idx in np.ndindex(f["ref"].shape):
        if kink[idx[0], idx[1], :, idx[2]].any():
            continue
        p, m = f["ref"].copy(), f["ref"].copy()
        p[idx] += h
        m[idx] -= h
        worst = max(worst, abs((J(ref=p) - J(ref=m)) / (2 * h) - gr[idx]) / (1 + abs(gr[idx])))
    for idx in np.ndindex(f["logits"].shape):
        p, m = f["logits"].copy(), f["logits"].copy()
        p[idx] += h
        m[idx] -= h
        worst = max(worst, abs((J(logits=p) - J(logits=m)) / (2 * h) - gl[idx]) / (1 + abs(gl[idx])))
    # softmax invariant: the logit gradients of one (query, head) sum to zero
    worst = max(worst, float(np.abs(gl.sum(-1)).max()))
    # grad_value does not depend on how the location was formed
    attn = oracle.softmax(f["logits"]).reshape(f["off"].shape[:-1])
    gv2, _, _ = oracle.backward(f["value"], f["shapes"], f["starts"], loc, attn, f["g"])
    worst = max(worst, _err(gv, gv2))
    return worst, 1e-6


# --------------------------------------------------------------------------- grouped locations
def _grouped_inputs(seed, G, M=4, levels=((6, 7), (3, 4)), N=2, Lq=7, K=3, D=3):
    """Per-sample tensors with G groups of M / G heads (one set of locations,
    weights, offsets and logits per group)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    shapes = np.asarray(levels, dtype=np.int64)
    starts = workloads.level_start_index(shapes)
    S = int((shapes[:, 0] * shapes[:, 1]).sum())
    L = len(levels)
    scale = np.asarray([[w, h] for (h, w) in levels], dtype=np.float64)
    return dict(shapes=shapes, starts=starts, value=rng.standard_normal((N, S, M, D)),
                g=rng.standard_normal((N, Lq, M * D)), loc=rng.uniform(-0.1, 1.1, (N, Lq, G, L, K, 2)),
                attn=rng.uniform(-0.5, 1.0, (N, Lq, G, L, K)), ref=rng.uniform(0.1, 0.9, (N, Lq, L, 2)),
                off=rng.standard_normal((N, Lq, G, L, K, 2)) * 0.3 * scale[None, None, None, :, None, :],
                logits=rng.standard_normal((N, Lq, G, L * K)), M=M, G=G)


def _to_heads(x, M):
    """Broadcast a per-group tensor [N, Lq, G, ...] to every head of its group."""
    return np.repeat(x, M // x.shape[2], axis=2)


def _sum_groups(x, G):
    """Sum a per-head tensor [N, Lq, M, ...] over the heads of each group."""
    return x.reshape(x.shape[:2] + (G, x.shape[2] // G) + x.shape[3:]).sum(axis=3)


def pin_grouped_broadcast():
    """A group's heads sample with the group's set: the grouped call equals the
    per-head call on the set broadcast to every head of its group, and its
    location, weight, offset and logit gradients are the per-head ones summed
    over the group (the chain rule through the broadcast); grad_value and the
    reference-point gradient are the same.  G = 1, 2 of M = 4 heads."""
    worst = 0.0
    for G in (1, 2):
        f = _grouped_inputs(61 + G, G)
        M, sh, st = f["M"], f["shapes"], f["starts"]
        loc_h, attn_h = _to_heads(f["loc"], M), _to_heads(f["attn"], M)
        worst = max(worst, _err(oracle.forward(f["value"], sh, st, f["loc"], f["attn"]),
                                oracle.forward(f["value"], sh, st, loc_h, attn_h)))
        gv, gl, ga = oracle.backward(f["value"], sh, st, f["loc"], f["attn"], f["g"])
        hv, hl, ha = oracle.backward(f["value"], sh, st, loc_h, attn_h, f["g"])
        worst = max(worst, _err(gv, hv), _err(gl, _sum_groups(hl, G)), _err(ga, _sum_groups(ha, G)))
        off_h, lg_h = _to_heads(f["off"], M), _to_heads(f["logits"], M)
        worst = max(worst, _err(oracle.forward_fused(f["value"], sh, st, f["ref"], f["off"], f["logits"]),
                                oracle.forward_fused(f["value"], sh, st, f["ref"], off_h, lg_h)))
        fg = oracle.backward_fused(f["value"], sh, st, f["ref"], f["off"], f["logits"], f["g"])
        fh = oracle.backward_fused(f["value"], sh, st, f["ref"], off_h, lg_h, f["g"])
        worst = max(worst, _err(fg[0], fh[0]), _err(fg[1], fh[1]), _err(fg[2], _sum_groups(fh[2], G)),
                    _err(fg[3], _sum_groups(fh[3], G)))
    return worst, 1e-12


def pin_grouped_as_wide_heads():
    """A group's heads are contiguous in value and in the output, so G groups of
    M / G heads of D channels are the plain call with G heads of (M / G) * D
    channels (the value tensor viewed as [N, Len_in, G, (M / G) * D])."""
    f = _grouped_inputs(71, 2)
    N, S, M, D = f["value"].shape
    G, sh, st = f["G"], f["shapes"], f["starts"]
    wide = f["value"].reshape(N, S, G, M // G * D)
    worst = _err(oracle.forward(f["value"], sh, st, f["loc"], f["attn"]),
                 oracle.forward(wide, sh, st, f["loc"], f["attn"]))
    gv, gl, ga = oracle.backward(f["value"], sh, st, f["loc"], f["attn"], f["g"])
    wv, wl, wa = oracle.backward(wide, sh, st, f["loc"], f["attn"], f["g"])
    return max(worst, _err(gv, wv.reshape(gv.shape)), _err(gl, wl), _err(ga, wa)), 1e-12


# --------------------------------------------------------------------------- options
AL = oracle.ALIGN_CORNERS
PL = oracle.PER_LEVEL_SOFTMAX


def pin_align_grid_sample():
    worst = 0.0
    for seed, lv in [(31, ((8, 8), (4, 4))), (32, ((5, 9), (3, 2), (2, 2)))]:
        t = _tiny(seed=seed, levels=lv, loc_lo=-0.3, loc_hi=1.3, Lq=25, K=3, M=3, D=5)
        out = oracle.forward(t["value"], t["shapes"], t["starts"], t["loc"], t["attn"], options=AL)
        ref = _grid_sample_forward(torch.from_numpy(t["value"]), t["shapes"], t["starts"],
                                   torch.from_numpy(t["loc"]), torch.from_numpy(t["attn"]),
                                   align_corners=True).numpy()
        worst = max(worst, _err(out, ref))
    return worst, 1e-12


def pin_align_pixel_centres():
    """With align_corners the pixel centres sit at i / (W - 1), the borders included."""
    t = _tiny(seed=33, levels=((5, 7), (3, 4)), Lq=30, K=2, M=2, D=3)
    rng = np.random.Generator(np.random.PCG64(34))
    loc = np.empty_like(t["loc"])
    expect = np.zeros((t["N"], t["Lq"], t["M"], t["D"]))
    for l, (H, W) in enumerate(t["shapes"]):
        ix = rng.integers(0, W, size=loc[..., l, :, 0].shape)
        iy = rng.integers(0, H, size=loc[..., l, :, 1].shape)
        ix[..., 0, 0] = W - 1          # the far border is a pixel centre too
        iy[..., 0, 0] = 0
        loc[..., l, :, 0] = ix / (W - 1)
        loc[..., l, :, 1] = iy / (H - 1)
        rows = t["starts"][l] + iy * W + ix
        for n in range(t["N"]):
            for q in range(t["Lq"]):
                for m in range(t["M"]):
                    for k in range(t["K"]):
                        expect[n, q, m] += t["attn"][n, q, m, l, k] * t["value"][n, rows[n, q, m, k], m]
    out = oracle.forward(t["value"], t["shapes"], t["starts"], loc, t["attn"], options=AL)
    return _err(out, expect.reshape(out.shape)), 1e-12


def pin_align_backward_autograd():
    t = _tiny(seed=35, levels=((8, 8), (4, 4), (3, 5)), loc_lo=-0.2, loc_hi=1.2, Lq=20, K=2, M=2, D=4)
    v = torch.from_numpy(t["value"]).requires_grad_(True)
    loc = torch.from_numpy(t["loc"]).requires_grad_(True)
    a = torch.from_numpy(t["attn"]).requires_grad_(True)
    out = _grid_sample_forward(v, t["shapes"], t["starts"], loc, a, align_corners=True)
    out.backward(torch.from_numpy(t["g"]))
    gv, gl, ga = oracle.backward(t["value"], t["shapes"], t["starts"], t["loc"], t["attn"], t["g"], options=AL)
    worst = max(_rel(gv, v.grad.numpy()), _rel(gl, loc.grad.numpy()), _rel(ga, a.grad.numpy()))
    return worst, 1e-12


def pin_per_level_closed():
    f = _fused_inputs(36, Lq=10, M=2, K=3, D=4)
    L, K = f["shapes"].shape[0], 3
    rng = np.random.Generator(np.random.PCG64(37))
    p = rng.uniform(0.1, 1.0, size=f["logits"].shape).reshape(-1, L, K)
    p /= p.sum(-1, keepdims=True)                      # each level's K weights sum to 1
    logits = np.log(p).reshape(f["logits"].shape)
    loc = oracle.locations(f["shapes"], f["ref"], f["off"])
    out = oracle.forward_fused(f["value"], f["shapes"], f["starts"], f["ref"], f["off"], logits, options=PL)
    worst = _err(out, oracle.forward(f["value"], f["shapes"], f["starts"], loc, p.reshape(loc.shape[:-1])))
    # a constant added to one level's logits does not move that level's weights
    shifted = logits.reshape(-1, L, K).copy()
    shifted[:, 1, :] += 3.0
    out2 = oracle.forward_fused(f["value"], f["shapes"], f["starts"], f["ref"], f["off"],
                                shifted.reshape(logits.shape), options=PL)
    worst = max(worst, _err(out2, out))
    # one level: the per-level softmax is the whole-row softmax
    f1 = _fused_inputs(38, levels=((6, 7),), Lq=9, M=2, K=4, D=3)
    a = oracle.forward_fused(f1["value"], f1["shapes"], f1["starts"], f1["ref"], f1["off"], f1["logits"], options=PL)
    b = oracle.forward_fused(f1["value"], f1["shapes"], f1["starts"], f1["ref"], f1["off"], f1["logits"])
    return max(worst, _err(a, b)), 1e-12


def pin_options_fused_backward():
    """Finite differences through the fused forward with each option, and the
    per-level zero sum of the logit gradients."""
    worst = 0.0
    for opt, seed in ((PL, 39), (AL, 40), (PL | AL, 41)):
        f = _fused_inputs(seed, Lq=4, K=2, D=3)
        gv, gr, go, gl = oracle.backward_fused(f["value"], f["shapes"], f["starts"], f["ref"], f["off"],
                                               f["logits"], f["g"], options=opt)

        def J(ref=None, off=None, logits=None):
            out = oracle.forward_fused(f["value"], f["shapes"], f["starts"], f["ref"] if ref is None else ref,
                                       f["off"] if off is None else off,
                                       f["logits"] if logits is None else logits, options=opt)
            return float((out * f["g"]).sum())

        h = 1e-6
        loc = oracle.locations(f["shapes"], f["ref"], f["off"])
        kink = np.zeros(loc.shape[:-1], dtype=bool)
        for l, (H, W) in enumerate(f["shapes"]):
            for c, size in ((0, W), (1, H)):
                px = loc[..., l, :, c] * (size - 1) if opt & AL else _px(loc[..., l, :, c], size)
                kink[..., l, :] |= np.abs(px - np.round(px)) < 1e-3
        for idx in np.ndindex(f["off"].shape):
            if kink[idx[:-1]]:
                continue
            p, m = f["off"].copy(), f["off"].copy()
            p[idx] += h
            m[idx] -= h
            worst = max(worst, abs((J(off=p) - J(off=m)) / (2 * h) - go[idx]) / (1 + abs(go[idx])))
        for idx in np.ndindex(f["ref"].shape):
            if kink[idx[0], idx[1], :, idx[2]].any():
                continue
            p, m = f["ref"].copy(), f["ref"].copy()
            p[idx] += h
            m[idx] -= h
            worst = max(worst, abs((J(ref=p) - J(ref=m)) / (2 * h) - gr[idx]) / (1 + abs(gr[idx])))
        for idx in np.ndindex(f["logits"].shape):
            p, m = f["logits"].copy(), f["logits"].copy()
            p[idx] += h
            m[idx] -= h
            worst = max(worst, abs((J(logits=p) - J(logits=m)) / (2 * h) - gl[idx]) / (1 + abs(gl[idx])))
        if opt & PL:
            L = f["shapes"].shape[0]
            worst = max(worst, float(np.abs(gl.reshape(gl.shape[:-1] + (L, -1)).sum(-1)).max()))
    return worst, 1e-6


# --------------------------------------------------------------------------- 3-D variant
def _vol_inputs(seed, levels, N=1, Lq=9, M=2, K=3, D=4, lo=-0.2, hi=1.2):
    rng = np.random.Generator(np.random.PCG64(seed))
    shapes = np.asarray(levels, dtype=np.int64).reshape(-1, 3)
    sizes = shapes.prod(-1)
    starts = np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64)
    S = int(sizes.sum())
    L = len(levels)
    value = rng.standard_normal((N, S, M, D))
    loc = rng.uniform(lo, hi, size=(N, Lq, M, L, K, 3))
    attn = rng.standard_normal((N, Lq, M, L, K))
    g = rng.standard_normal((N, Lq, M * D))
    return dict(shapes=shapes, starts=starts, value=value, loc=loc, attn=attn, g=g)


def _grid_sample_3d(value, shapes, starts, loc, attn, align_corners):
    """Per-level 5-D grid_sample (trilinear) in float64 torch."""
    N, S, M, D = value.shape
    _, Lq, _, L, K, _ = loc.shape
    out = 0
    for l in range(L):
        Dd, H, W = (int(x) for x in shapes[l])
        s0 = int(starts[l])
        v_l = value[:, s0:s0 + Dd * H * W].reshape(N, Dd, H, W, M, D).permute(0, 4, 5, 1, 2, 3).reshape(N * M, D, Dd, H, W)
        grid = (2.0 * loc[:, :, :, l] - 1.0).permute(0, 2, 1, 3, 4).reshape(N * M, Lq, K, 1, 3)
        smp = F.grid_sample(v_l, grid, mode="bilinear", padding_mode="zeros", align_corners=align_corners)
        a = attn[:, :, :, l].permute(0, 2, 1, 3).reshape(N * M, 1, Lq, K, 1)
        out = out + (smp * a).sum((-1, -2))
    return out.reshape(N, M, D, Lq).permute(0, 3, 1, 2).reshape(N, Lq, M * D)


def pin_trilinear_grid_sample():
    worst = 0.0
    for seed, lv, opt in [(51, ((3, 4, 5), (2, 2, 3)), 0), (52, ((4, 3, 6), (1, 2, 2), (2, 5, 1)), 0),
                          (53, ((3, 4, 5), (2, 3, 2)), AL)]:
        t = _vol_inputs(seed, lv)
        out = oracle.forward3d(t["value"], t["shapes"], t["starts"], t["loc"], t["attn"], options=opt)
        ref = _grid_sample_3d(torch.from_numpy(t["value"]), t["shapes"], t["starts"], torch.from_numpy(t["loc"]),
                              torch.from_numpy(t["attn"]), align_corners=bool(opt & AL)).numpy()
        worst = max(worst, _err(out, ref))
    return worst, 1e-12


def pin_trilinear_one_slice():
    """A one-slice volume sampled at its centre plane (pz = 0) is the 2-D map."""
    lv2 = ((5, 6), (3, 4))
    t = _tiny(seed=54, levels=lv2, Lq=12, K=3, M=2, D=4)
    shapes3 = np.asarray([[1, h, w] for (h, w) in lv2], dtype=np.int64)
    loc3 = np.concatenate([t["loc"], np.full(t["loc"].shape[:-1] + (1,), 0.5)], axis=-1)
    out3 = oracle.forward3d(t["value"], shapes3, t["starts"], loc3, t["attn"])
    out2 = oracle.forward(t["value"], t["shapes"], t["starts"], t["loc"], t["attn"])
    return _err(out3, out2), 1e-12


def pin_trilinear_backward():
    worst = 0.0
    for seed, opt in ((55, 0), (56, AL)):
        t = _vol_inputs(seed, ((3, 4, 5), (2, 3, 2)), Lq=7)
        v = torch.from_numpy(t["value"]).requires_grad_(True)
        loc = torch.from_numpy(t["loc"]).requires_grad_(True)
        a = torch.from_numpy(t["attn"]).requires_grad_(True)
        out = _grid_sample_3d(v, t["shapes"], t["starts"], loc, a, align_corners=bool(opt & AL))
        out.backward(torch.from_numpy(t["g"]))
        gv, gl, ga = oracle.backward3d(t["value"], t["shapes"], t["starts"], t["loc"], t["attn"], t["g"], options=opt)
        worst = max(worst, _rel(gv, v.grad.numpy()), _rel(gl, loc.grad.numpy()), _rel(ga, a.grad.numpy()))
    return worst, 1e-12


def pin_trilinear_fd():
    """Central finite differences of the 3-D forward in the locations, away from the kinks."""
    t = _vol_inputs(57, ((3, 4, 5), (2, 2, 3)), Lq=4, K=2, D=3, lo=-0.1, hi=1.1)
    gv, gl, ga = oracle.backward3d(t["value"], t["shapes"], t["starts"], t["loc"], t["attn"], t["g"])

    def J(loc):
        return float((oracle.forward3d(t["value"], t["shapes"], t["starts"], loc, t["attn"]) * t["g"]).sum())

    h = 1e-6
    worst = 0.0
    for idx in np.ndindex(t["loc"].shape):
        size = t["shapes"][idx[3]][2 - idx[5]]          # (D, H, W) against (x, y, z)
        p = t["loc"][idx] * size - 0.5
        if abs(p - round(p)) < 1e-3:
            continue
        pl, mi = t["loc"].copy(), t["loc"].copy()
        pl[idx] += h
        mi[idx] -= h
        worst = max(worst, abs((J(pl) - J(mi)) / (2 * h) - gl[idx]) / (1 + abs(gl[idx])))
    return worst, 1e-6


ALL_PINS = {
    "worked_example": pin_worked_example,
    "softmax_closed": pin_softmax_closed,
    "constant_map": pin_constant_map,
    "pixel_centres": pin_pixel_centres,
    "linear_ramp": pin_linear_ramp,
    "far_outside": pin_far_outside,
    "grid_sample": pin_grid_sample,
    "dense_tent": pin_dense_tent,
    "backward_autograd": pin_backward_autograd,
    "backward_fd": pin_backward_fd,
    "adjoint": pin_adjoint,
    "fused_composition": pin_fused_composition,
    "fused_backward": pin_fused_backward,
    "grouped_broadcast": pin_grouped_broadcast,
    "grouped_as_wide_heads": pin_grouped_as_wide_heads,
    "align_grid_sample": pin_align_grid_sample,
    "align_pixel_centres": pin_align_pixel_centres,
    "align_backward_autograd": pin_align_backward_autograd,
    "per_level_closed": pin_per_level_closed,
    "options_fused_backward": pin_options_fused_backward,
    "trilinear_grid_sample": pin_trilinear_grid_sample,
    "trilinear_one_slice": pin_trilinear_one_slice,
    "trilinear_backward": pin_trilinear_backward,
    "trilinear_fd": pin_trilinear_fd,
}


def run_all():
    """{name: (passed, error, tol)}; an exception counts as a failed pin."""
    res = {}
    for name, fn in ALL_PINS.items():
        try:
            err, tol = fn()
            res[name] = (bool(err <= tol), err, tol)
        except Exception as exc:  # a broken oracle may reject its own arguments
            res[name] = (False, repr(exc), None)
    return res
