"""Seeded synthetic inputs for the MSDeformAttn core.

This module is shared by the tests, the benchmark and the smoke check.  It
holds random draws with the shapes and structure of the workloads and nothing
of the method's arithmetic: no location step, no softmax, no sampling.  The
consumers turn the raw draws into the inputs of each call.

Workloads (Deformable DETR on COCO-sized 800x1333 inputs is the setting the
pages describe; no dataset is used, these draws stand in for it):

  tiny      N=1, M=2, D=8, levels 8x8, 4x4 (Len_in=80), Len_q=80, K=2.
            Locations drawn directly ~U(-0.1, 1.1) per coordinate.
  encoder   N=2, M=8, D=32, levels 100x167, 50x84, 25x42, 13x21 (Len_in=22223),
            Len_q=Len_in, K=4.  Query i sits at the centre of its own pixel
            (normalised), the same reference point for every level; offsets
            ~N(0, 0.02 * size of the level) in pixels of that level.
  decoder   N=8, Len_q=300, the encoder's levels, M=8, D=32, K=4, bf16 value.
            Reference points ~U(0.05, 0.95)^2 (shared by the levels); offsets
            ~N(0, 0.05 * size of the level) in pixels.
  large     N=8, M=8, D=32, levels 128^2, 64^2, 32^2, 16^2 (Len_in=21760),
            Len_q=Len_in, K=4, bf16 value; pixel-centre references, offsets
            ~N(0, 0.05 * size of the level) in pixels.

Every draw: value ~N(0,1), attention logits ~N(0,1), grad_output ~N(0,1),
numpy PCG64 seeded with the workload's seed.
"""
from dataclasses import dataclass, field
from typing import List, Tuple

import numpy as np

ENCODER_LEVELS = [(100, 167), (50, 84), (25, 42), (13, 21)]
LARGE_LEVELS = [(128, 128), (64, 64), (32, 32), (16, 16)]


@dataclass
class Workload:
    name: str
    N: int
    M: int
    D: int
    levels: List[Tuple[int, int]]     # (H, W) per level
    K: int
    Len_q: int = -1                    # -1: one query per value pixel
    dtype: str = "f32"                 # storage of value / output / grad_output
    refs: str = "pixel_centres"        # "pixel_centres" | "uniform" | "none"
    ref_range: Tuple[float, float] = (0.05, 0.95)
    offset_sigma: float = 0.02         # normalised; drawn in pixels as sigma * size
    loc_range: Tuple[float, float] = (-0.1, 1.1)   # refs == "none": direct location draw
    seed: int = 1234

    @property
    def L(self):
        return len(self.levels)

    @property
    def Len_in(self):
        return sum(h * w for h, w in self.levels)

    @property
    def Lq(self):
        return self.Len_in if self.Len_q < 0 else self.Len_q

    @property
    def samples(self):
        return self.N * self.Lq * self.M * self.L * self.K

    def spatial_shapes(self):
        return np.asarray(self.levels, dtype=np.int64).reshape(-1, 2)

    def level_start_index(self):
        return level_start_index(self.spatial_shapes())


def level_start_index(spatial_shapes):
    """Start of each level in the flattened value sequence (layout, not method)."""
    sh = np.asarray(spatial_shapes, dtype=np.int64).reshape(-1, 2)
    sizes = sh[:, 0] * sh[:, 1]
    return np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64)


WORKLOADS = {
    "tiny": Workload("tiny", N=1, M=2, D=8, levels=[(8, 8), (4, 4)], K=2, refs="none", seed=1234),
    "encoder": Workload("encoder", N=2, M=8, D=32, levels=ENCODER_LEVELS, K=4, offset_sigma=0.02,
                        seed=1235),
    "decoder": Workload("decoder", N=8, M=8, D=32, levels=ENCODER_LEVELS, K=4, Len_q=300, dtype="bf16",
                        refs="uniform", offset_sigma=0.05, seed=1236),
    "encoder_train": Workload("encoder_train", N=2, M=8, D=32, levels=ENCODER_LEVELS, K=4,
                              offset_sigma=0.02, seed=1237),
    "large": Workload("large", N=8, M=8, D=32, levels=LARGE_LEVELS, K=4, dtype="bf16",
                      offset_sigma=0.05, seed=1238),
}


def _pixel_centre_refs(levels, N):
    """One query per pixel of every level, in flattened order; its reference is
    the centre of that pixel in normalised coordinates, the same for all levels."""
    parts = []
    for (h, w) in levels:
        ys, xs = np.meshgrid(np.arange(h), np.arange(w), indexing="ij")
        parts.append(np.stack([(xs.ravel() + 0.5) / w, (ys.ravel() + 0.5) / h], axis=-1))
    per_query = np.concatenate(parts, axis=0)                       # [Len_in, 2]
    L = len(levels)
    refs = np.broadcast_to(per_query[None, :, None, :], (N, per_query.shape[0], L, 2))
    return np.ascontiguousarray(refs, dtype=np.float32)


def draw(w: Workload, seed=None):
    """Raw draws for workload `w` (float32 numpy arrays):

    value [N,Len_in,M,D], attention_logits [N,Lq,M,L*K], grad_output [N,Lq,M*D],
    and either reference_points [N,Lq,L,2] + sampling_offsets [N,Lq,M,L,K,2]
    (pixels of the level), or, for refs == "none", sampling_locations
    [N,Lq,M,L,K,2] drawn directly.
    """
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    N, M, D, L, K, Lq, S = w.N, w.M, w.D, w.L, w.K, w.Lq, w.Len_in
    out = {"spatial_shapes": w.spatial_shapes(), "level_start_index": w.level_start_index()}
    out["value"] = rng.standard_normal((N, S, M, D), dtype=np.float32)
    if w.refs == "none":
        lo, hi = w.loc_range
        out["sampling_locations"] = rng.uniform(lo, hi, size=(N, Lq, M, L, K, 2)).astype(np.float32)
    else:
        if w.refs == "pixel_centres":
            if Lq != S:
                raise ValueError("pixel-centre references need one query per value pixel")
            out["reference_points"] = _pixel_centre_refs(w.levels, N)
        else:
            lo, hi = w.ref_range
            one = rng.uniform(lo, hi, size=(N, Lq, 1, 2)).astype(np.float32)
            out["reference_points"] = np.ascontiguousarray(np.broadcast_to(one, (N, Lq, L, 2)))
        # per-level pixel scale: sigma * (W_l, H_l)
        scale = np.asarray([[wl, hl] for (hl, wl) in w.levels], dtype=np.float32) * w.offset_sigma
        z = rng.standard_normal((N, Lq, M, L, K, 2), dtype=np.float32)
        out["sampling_offsets"] = (z * scale[None, None, None, :, None, :]).astype(np.float32)
    out["attention_logits"] = rng.standard_normal((N, Lq, M, L * K), dtype=np.float32)
    out["grad_output"] = rng.standard_normal((N, Lq, M * D), dtype=np.float32)
    return out


def custom(name="custom", **kw):
    """A workload with explicit fields (tests of ragged and edge shapes)."""
    return Workload(name=name, **kw)


# ----------------------------------------------------------------------------- volumes (3-D variant)
VIDEO_LEVELS = [(8, 50, 84), (4, 25, 42), (2, 13, 21)]   # (D, H, W): frames x rows x columns


def draw_volumes(N, M, D, levels, K, Len_q, dtype="f32", loc_range=(-0.05, 1.05), seed=1239):
    """Raw draws for the 3-D variant: value [N,Len_in,M,D] ~N(0,1) with
    Len_in = sum D_l*H_l*W_l, sampling_locations [N,Len_q,M,L,K,3] ~U(loc_range)
    per coordinate, attention_logits [N,Len_q,M,L*K] and grad_output ~N(0,1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    sh = np.asarray(levels, dtype=np.int64).reshape(-1, 3)
    sizes = sh.prod(-1)
    S = int(sizes.sum())
    L = sh.shape[0]
    lo, hi = loc_range
    return {"spatial_shapes": sh, "level_start_index": np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64),
            "value": rng.standard_normal((N, S, M, D), dtype=np.float32),
            "sampling_locations": rng.uniform(lo, hi, size=(N, Len_q, M, L, K, 3)).astype(np.float32),
            "attention_logits": rng.standard_normal((N, Len_q, M, L * K), dtype=np.float32),
            "grad_output": rng.standard_normal((N, Len_q, M * D), dtype=np.float32), "dtype": dtype}
