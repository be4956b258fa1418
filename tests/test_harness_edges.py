"""The parity harness's handling of cell edges, on the CPU.

Where a pixel coordinate sits on an integer, the location gradient is
one-sided and either side is a correct answer; everywhere else the oracle's
own value is the only one.  These tests feed the harness "GPU" results made by
the oracle itself at each side of an edge (and a planted wrong one) and check
that it accepts both sides, and only them.
"""
import numpy as np
import pytest

import harness as H
import oracle
import workloads


# level 0 is 8 pixels wide: (i + 0.5) / 8 is exact in fp32, so px = i exactly
LEVELS = [(6, 8), (3, 4)]


def _problem(refs="none", seed=5):
    w = workloads.custom(N=1, M=2, D=8, levels=LEVELS, K=3, Len_q=12, refs=refs, seed=seed)
    return w, H.prepared(w)


def _put_on_edges(p, w):
    """Moves the x coordinate of every other sample of level 0 onto an exact
    pixel edge: px = i, an integer in fp32 and in fp64."""
    loc = p["sampling_locations"].copy()
    Hl, Wl = w.levels[0]
    rng = np.random.Generator(np.random.PCG64(3))
    ix = rng.integers(0, Wl, size=loc[..., 0, ::2, 0].shape)
    loc[..., 0, ::2, 0] = ((ix + 0.5) / Wl).astype(np.float32)
    p = dict(p)
    p["sampling_locations"] = loc
    return p


def test_random_locations_have_no_edges():
    w, p = _problem()
    mask, _, _ = H.edges_unfused(p["sampling_locations"], p["spatial_shapes"])
    assert not mask.any()
    ref = H.backward_reference(p)
    base = oracle.backward(p["value"], p["spatial_shapes"], p["level_start_index"], p["sampling_locations"],
                           p["attention_weights"], p["grad_output"])
    got = ref.for_gpu(base)
    for a, b in zip(got, base):
        assert np.array_equal(a, b)


def test_either_side_of_an_edge_is_accepted_and_nothing_else():
    w, p = _problem()
    p = _put_on_edges(p, w)
    mask, below, above = H.edges_unfused(p["sampling_locations"], p["spatial_shapes"])
    assert mask[..., 0, ::2, 0].all() and mask.sum() == mask[..., 0, ::2, 0].size
    sh, st = p["spatial_shapes"], p["level_start_index"]

    def orc(loc):
        return oracle.backward(p["value"], sh, st, loc, p["attention_weights"], p["grad_output"])

    lo, hi = orc(below), orc(above)
    # the two sides differ at the edges: the x gradient jumps
    assert np.abs(lo[1][mask] - hi[1][mask]).max() > 1e-2
    ref = H.backward_reference(p)
    for side in (lo, hi):
        for a, b in zip(side, ref.for_gpu(side)):
            H.assert_bwd(a, b, "f32", "one-sided gradient")
    # a mixture, side by side per coordinate, is accepted too
    pick = np.zeros_like(mask)
    pick[..., 0, ::4, 0] = True
    mixed = orc(np.where(pick, below, above))
    for a, b in zip(mixed, ref.for_gpu(mixed)):
        H.assert_bwd(a, b, "f32", "mixed one-sided gradients")
    # a location gradient that is neither side fails
    wrong = [t.copy() for t in lo]
    wrong[1][mask] = 0.5 * (lo[1][mask] + hi[1][mask])
    with pytest.raises(AssertionError):
        r = ref.for_gpu(wrong)
        H.assert_bwd(wrong[1], r[1], "f32", "halfway")
    # and a wrong gradient away from the edges still fails
    wrong = [t.copy() for t in lo]
    wrong[1][~mask] *= 1.01
    with pytest.raises(AssertionError):
        H.assert_bwd(wrong[1], ref.for_gpu(wrong)[1], "f32", "off by 1%")


def test_fused_edges_resolve_on_the_offsets():
    """Fused call: offsets that put px on an integer; the reference-point
    gradient then follows the chosen sides."""
    w = workloads.custom(N=1, M=2, D=8, levels=LEVELS, K=3, Len_q=12, refs="uniform", seed=11)
    p = dict(H.prepared(w))
    sh, st = p["spatial_shapes"], p["level_start_index"]
    off = p["sampling_offsets"].copy()
    ref_pt = p["reference_points"]
    Wl = w.levels[0][1]
    # px = ref * W + off - 0.5: move off so that px is the nearest integer (up to the fp32 rounding of the
    # new offset, well inside the edge window)
    px = ref_pt[:, :, None, 0, None, 0].astype(np.float64) * Wl + off[..., 0, :, 0] - 0.5
    off[..., 0, :, 0] = (off[..., 0, :, 0] + (np.rint(px) - px)).astype(np.float32)
    p["sampling_offsets"] = off
    mask, below, above = H.edges_fused(ref_pt, off, sh)
    assert mask[..., 0, :, 0].mean() > 0.5

    def orc(o):
        return oracle.backward_fused(p["value"], sh, st, ref_pt, o, p["attention_logits"], p["grad_output"])

    ref = H.backward_fused_reference(p)
    for side in (orc(below), orc(above)):
        for a, b in zip(side, ref.for_gpu(side)):
            H.assert_bwd(a, b, "f32", "fused one-sided gradient")
