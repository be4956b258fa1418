"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Every case runs the same seeded inputs through libmsda on the GPU and through
the oracle on the CPU and compares element by element:
  forward fp32   max-abs <= 1e-5 and normwise rel <= 1e-5
  backward fp32  normwise rel <= 1e-4 per tensor (atomic order is free)
  bf16 storage   normwise rel <= 2e-2 for bf16 outputs; fp32 gradients of a
                 bf16 problem are held to the fp32 bar (same rounded inputs).
"""
import numpy as np
import pytest
import torch

import harness as H
import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msda():
    import scale_deformable_attention_06_b300 as m
    assert torch.cuda.is_available(), "these tests need a CUDA device"
    return m


def _run_forward(msda, w, p):
    dt = H.storage_dtype(w)
    out = msda.msda_forward(H.dev(p["value"], dt), p["spatial_shapes"], p["level_start_index"],
                            H.dev(p["sampling_locations"]), H.dev(p["attention_weights"]))
    return out.float().cpu().numpy()


def _run_fused(msda, w, p):
    dt = H.storage_dtype(w)
    out = msda.msda_forward_fused(H.dev(p["value"], dt), p["spatial_shapes"], p["level_start_index"],
                                  H.dev(p["reference_points"]), H.dev(p["sampling_offsets"]),
                                  H.dev(p["attention_logits"]))
    return out.float().cpu().numpy()


def _run_backward(msda, w, p, flags=0):
    dt = H.storage_dtype(w)
    gv, gl, ga = msda.msda_backward(H.dev(p["value"], dt), p["spatial_shapes"], p["level_start_index"],
                                    H.dev(p["sampling_locations"]), H.dev(p["attention_weights"]),
                                    H.dev(p["grad_output"], dt), flags=flags)
    return gv.cpu().numpy(), gl.cpu().numpy(), ga.cpu().numpy()


def _run_backward_fused(msda, w, p, flags=0):
    dt = H.storage_dtype(w)
    outs = msda.msda_backward_fused(H.dev(p["value"], dt), p["spatial_shapes"], p["level_start_index"],
                                    H.dev(p["reference_points"]), H.dev(p["sampling_offsets"]),
                                    H.dev(p["attention_logits"]), H.dev(p["grad_output"], dt), flags=flags)
    return tuple(o.cpu().numpy() for o in outs)


def _oracle_backward_fused(p, options=0):
    """Edge-aware oracle reference of the fused backward (see harness)."""
    return H.backward_fused_reference(p, options)


def _check_backward_fused(w, got, ref):
    names = ("grad_value", "grad_reference_points", "grad_sampling_offsets", "grad_attention_logits")
    for name, g, r in zip(names, got, ref.for_gpu(got)):
        H.assert_bwd(g.reshape(r.shape), r, "f32", f"{w.name} fused {name}")


def _oracle_forward(p):
    return oracle.forward(p["value"], p["spatial_shapes"], p["level_start_index"], p["sampling_locations"],
                          p["attention_weights"])


def _oracle_backward(p, options=0):
    """Edge-aware oracle reference of the backward (see harness)."""
    return H.backward_reference(p, options)


def _check_backward(w, got, ref):
    dtype = "f32"   # gradients are fp32 outputs of identical (rounded) inputs
    for name, g, r in zip(("grad_value", "grad_sampling_locations", "grad_attention_weights"), got,
                          ref.for_gpu(got)):
        H.assert_bwd(g, r, dtype, f"{w.name} {name}")


# ----------------------------------------------------------------- workloads
def test_tiny_forward_backward(msda):
    w = workloads.WORKLOADS["tiny"]
    p = H.prepared(w)
    H.assert_fwd(_run_forward(msda, w, p), _oracle_forward(p), w.dtype)
    ref = _oracle_backward(p)
    _check_backward(w, _run_backward(msda, w, p), ref)
    _check_backward(w, _run_backward(msda, w, p, msda.MSDA_DETERMINISTIC), ref)


def test_encoder_forward_fp32(msda):
    w = workloads.WORKLOADS["encoder"]
    p = H.prepared(w)
    H.assert_fwd(_run_forward(msda, w, p), _oracle_forward(p), w.dtype, "encoder output")


def test_encoder_forward_fused_fp32(msda):
    w = workloads.WORKLOADS["encoder"]
    p = H.prepared(w)
    ref = oracle.forward_fused(p["value"], p["spatial_shapes"], p["level_start_index"], p["reference_points"],
                               p["sampling_offsets"], p["attention_logits"])
    H.assert_fwd(_run_fused(msda, w, p), ref, w.dtype, "encoder fused output")


def test_decoder_fused_bf16(msda):
    w = workloads.WORKLOADS["decoder"]
    p = H.prepared(w)
    ref = oracle.forward_fused(p["value"], p["spatial_shapes"], p["level_start_index"], p["reference_points"],
                               p["sampling_offsets"], p["attention_logits"])
    fused = _run_fused(msda, w, p)
    H.assert_fwd(fused, ref, w.dtype, "decoder fused output")
    # the unfused call on the locations the oracle forms agrees as well
    H.assert_fwd(_run_forward(msda, w, p), _oracle_forward(p), w.dtype, "decoder output")
    # the storage error itself: against the oracle on the unrounded fp32 draws
    u = H.prepared(w, round_bf16=False)
    ref_u = oracle.forward_fused(u["value"], u["spatial_shapes"], u["level_start_index"], u["reference_points"],
                                 u["sampling_offsets"], u["attention_logits"])
    _, rel = H.errors(fused, ref_u)
    assert rel <= H.BF16_REL, f"decoder fused output against unrounded fp32 inputs: rel {rel:.3e}"
    fb = _run_backward_fused(msda, w, p)
    for name, g, r in zip(("grad_value", "grad_reference_points", "grad_sampling_offsets", "grad_attention_logits"),
                          fb, _oracle_backward_fused(u).for_gpu(fb)):
        _, rel = H.errors(g.reshape(r.shape), r)
        assert rel <= H.BF16_REL, f"decoder fused {name} against unrounded fp32 inputs: rel {rel:.3e}"


def test_encoder_train_backward(msda):
    w = workloads.WORKLOADS["encoder_train"]
    p = H.prepared(w)
    ref = _oracle_backward(p)
    H.assert_fwd(_run_forward(msda, w, p), _oracle_forward(p), w.dtype)
    _check_backward(w, _run_backward(msda, w, p), ref)
    det = [_run_backward(msda, w, p, msda.MSDA_DETERMINISTIC) for _ in range(3)]
    _check_backward(w, det[0], ref)
    for other in det[1:]:
        for a, b in zip(det[0], other):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), "deterministic mode is not bitwise stable"


def test_large_bf16_forward_backward(msda):
    w = workloads.WORKLOADS["large"]
    p = H.prepared(w)
    out = _run_forward(msda, w, p)
    H.assert_fwd(out, _oracle_forward(p), w.dtype, "large output")
    got = _run_backward(msda, w, p)
    _check_backward(w, got, _oracle_backward(p))
    # the storage error itself: against the oracle on the unrounded fp32 value and grad_output
    u = H.prepared(w, round_bf16=False)
    _, rel = H.errors(out, _oracle_forward(u))
    assert rel <= H.BF16_REL, f"large output against unrounded fp32 inputs: rel {rel:.3e}"
    for name, g, r in zip(("grad_value", "grad_sampling_locations", "grad_attention_weights"), got,
                          _oracle_backward(u).for_gpu(got)):
        _, rel = H.errors(g, r)
        assert rel <= H.BF16_REL, f"large {name} against unrounded fp32 inputs: rel {rel:.3e}"


# ----------------------------------------------------------------- shapes and edges
RAGGED_LEVELS = [(7, 5), (3, 9), (1, 1), (2, 1)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("D", [8, 16, 32, 64])
def test_ragged_all_head_dims(msda, dtype, D):
    """Len_q not a multiple of the rows a warp owns, odd level sizes
    including 1x1, 2x1, samples partly outside the maps."""
    w = workloads.custom(N=2, M=3, D=D, levels=RAGGED_LEVELS, K=3, Len_q=37, dtype=dtype, refs="uniform",
                         ref_range=(-0.05, 1.05), offset_sigma=0.2, seed=99 + D)
    p = H.prepared(w)
    H.assert_fwd(_run_forward(msda, w, p), _oracle_forward(p), dtype, f"D={D} {dtype} output")
    ref = oracle.forward_fused(p["value"], p["spatial_shapes"], p["level_start_index"], p["reference_points"],
                               p["sampling_offsets"], p["attention_logits"])
    H.assert_fwd(_run_fused(msda, w, p), ref, dtype, f"D={D} {dtype} fused output")
    ref_b = _oracle_backward(p)
    _check_backward(w, _run_backward(msda, w, p), ref_b)
    _check_backward(w, _run_backward(msda, w, p, msda.MSDA_DETERMINISTIC), ref_b)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_dense_levels_merge_path(msda, dtype):
    """Many queries on small maps: every level carries at least 32 samples per
    pixel, so the backward sums coinciding corners of neighbouring queries
    before reducing into grad_value.  Ragged Len_q (not a multiple of the four
    queries a warp owns), samples partly outside the maps, both modes."""
    w = workloads.custom(N=2, M=3, D=32, levels=[(5, 7), (2, 3), (1, 2)], K=4, Len_q=301, dtype=dtype,
                         refs="uniform", ref_range=(-0.05, 1.05), offset_sigma=0.2, seed=1301)
    p = H.prepared(w)
    H.assert_fwd(_run_forward(msda, w, p), _oracle_forward(p), dtype, f"dense {dtype} output")
    ref_b = _oracle_backward(p)
    _check_backward(w, _run_backward(msda, w, p), ref_b)
    det = [_run_backward(msda, w, p, msda.MSDA_DETERMINISTIC) for _ in range(2)]
    _check_backward(w, det[0], ref_b)
    for a, b in zip(det[0], det[1]):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), "deterministic mode is not bitwise stable"


@pytest.mark.parametrize("L,K", [(1, 1), (1, 4), (16, 16), (5, 7)])
def test_levels_and_points(msda, L, K):
    """Single-scale (L=1), the largest L*K (256), and a ragged L*K."""
    levels = [(3 + (l % 4), 2 + (l * 3) % 7) for l in range(L)]
    w = workloads.custom(N=1, M=2, D=32, levels=levels, K=K, Len_q=21, refs="uniform", ref_range=(0.0, 1.0),
                         offset_sigma=0.3, seed=7 + L * 31 + K)
    p = H.prepared(w)
    H.assert_fwd(_run_forward(msda, w, p), _oracle_forward(p), "f32")
    _check_backward(w, _run_backward(msda, w, p), _oracle_backward(p))
    ref = oracle.forward_fused(p["value"], p["spatial_shapes"], p["level_start_index"], p["reference_points"],
                               p["sampling_offsets"], p["attention_logits"])
    H.assert_fwd(_run_fused(msda, w, p), ref, "f32")


def test_all_outside_and_integer_coordinates(msda):
    w = workloads.custom(N=1, M=2, D=16, levels=[(6, 5), (3, 4)], K=4, Len_q=30, refs="none", seed=5)
    p = H.prepared(w)
    loc = p["sampling_locations"].copy()
    rng = np.random.Generator(np.random.PCG64(8))
    # first third: far outside; second third: exact pixel corners (integer px);
    # last third: exactly on the outer border lines px = -1 and px = W
    n = loc.shape[1] // 3
    loc[:, :n] = rng.choice([-3.0, 4.0], size=loc[:, :n].shape)
    for l, (Hl, Wl) in enumerate(w.levels):
        ix = rng.integers(-1, Wl + 1, size=loc[:, n:2 * n, :, l, :, 0].shape)
        iy = rng.integers(-1, Hl + 1, size=loc[:, n:2 * n, :, l, :, 1].shape)
        loc[:, n:2 * n, :, l, :, 0] = (ix + 0.5) / Wl
        loc[:, n:2 * n, :, l, :, 1] = (iy + 0.5) / Hl
        loc[:, 2 * n:, :, l, :, 0] = rng.choice([-0.5 / Wl, (Wl + 0.5) / Wl], size=loc[:, 2 * n:, :, l, :, 0].shape)
    p["sampling_locations"] = loc.astype(np.float32)
    got = _run_forward(msda, w, p)
    H.assert_fwd(got, _oracle_forward(p), "f32")
    assert np.all(got[:, :n] == 0.0)
    _check_backward(w, _run_backward(msda, w, p), _oracle_backward(p))


def test_empty_problems(msda):
    w = workloads.custom(N=2, M=2, D=8, levels=[(4, 4)], K=2, Len_q=5, refs="none", seed=3)
    p = H.prepared(w)
    dev = "cuda"
    value = H.dev(p["value"])
    # Len_q = 0: nothing to sample; backward still zeroes grad_value
    loc0 = torch.zeros((2, 0, 2, 1, 2, 2), device=dev)
    a0 = torch.zeros((2, 0, 2, 1, 2), device=dev)
    out = msda.msda_forward(value, p["spatial_shapes"], p["level_start_index"], loc0, a0)
    assert out.shape == (2, 0, 16)
    gv = torch.full_like(value, 7.0)
    msda.msda_backward(value, p["spatial_shapes"], p["level_start_index"], loc0, a0, torch.zeros((2, 0, 16), device=dev),
                       grad_value=gv)
    torch.cuda.synchronize()
    assert torch.count_nonzero(gv).item() == 0
    # N = 0
    v0 = torch.zeros((0, 16, 2, 8), device=dev)
    out = msda.msda_forward(v0, p["spatial_shapes"], p["level_start_index"], torch.zeros((0, 5, 2, 1, 2, 2), device=dev),
                            torch.zeros((0, 5, 2, 1, 2), device=dev))
    assert out.shape == (0, 5, 16)


def test_accumulate_grad_value(msda):
    w = workloads.WORKLOADS["tiny"]
    p = H.prepared(w)
    gv0 = np.random.Generator(np.random.PCG64(4)).standard_normal(p["value"].shape).astype(np.float32)
    # grad_value is continuous in the locations: the plain oracle call is its reference
    ref_gv = oracle.backward(p["value"], p["spatial_shapes"], p["level_start_index"], p["sampling_locations"],
                             p["attention_weights"], p["grad_output"])[0]
    for flags in (msda.MSDA_ACCUMULATE_GRAD_VALUE, msda.MSDA_ACCUMULATE_GRAD_VALUE | msda.MSDA_DETERMINISTIC):
        gv = H.dev(gv0)
        msda.msda_backward(H.dev(p["value"]), p["spatial_shapes"], p["level_start_index"], H.dev(p["sampling_locations"]),
                           H.dev(p["attention_weights"]), H.dev(p["grad_output"]), grad_value=gv, flags=flags)
        H.assert_bwd(gv.cpu().numpy(), gv0 + ref_gv, "f32", "accumulated grad_value")


def test_invalid_arguments_return_errors(msda):
    w = workloads.WORKLOADS["tiny"]
    p = H.prepared(w)
    value = H.dev(p["value"])
    loc, attn = H.dev(p["sampling_locations"]), H.dev(p["attention_weights"])
    bad_starts = p["level_start_index"].copy()
    bad_starts[1] += 1
    with pytest.raises(msda.MSDAError) as e:
        msda.msda_forward(value, p["spatial_shapes"], bad_starts, loc, attn)
    assert e.value.name == "MSDA_ERR_INVALID_ARG"
    with pytest.raises(msda.MSDAError) as e:
        msda.msda_forward(value[..., :4].contiguous(), p["spatial_shapes"], p["level_start_index"],
                          loc, attn, output=torch.empty((1, 80, 8), device="cuda"))
    assert e.value.name == "MSDA_ERR_UNSUPPORTED"
    with pytest.raises(ValueError):
        msda.msda_forward(value.cpu(), p["spatial_shapes"], p["level_start_index"], loc, attn)


# ----------------------------------------------------------------- fused backward (a9)
@pytest.mark.parametrize("name", ["encoder_train", "decoder"])
def test_fused_backward_workloads(msda, name):
    """Gradients with respect to reference points, offsets and logits on the
    encoder training workload (fp32) and the decoder workload (bf16 value)."""
    w = workloads.WORKLOADS[name]
    p = H.prepared(w)
    ref = _oracle_backward_fused(p)
    _check_backward_fused(w, _run_backward_fused(msda, w, p), ref)
    det = [_run_backward_fused(msda, w, p, msda.MSDA_DETERMINISTIC) for _ in range(2)]
    _check_backward_fused(w, det[0], ref)
    for a, b in zip(det[0], det[1]):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), "deterministic fused backward is not bitwise stable"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("D,L,K", [(8, 4, 3), (16, 1, 4), (32, 5, 7), (64, 2, 2), (32, 16, 16)])
def test_fused_backward_shapes(msda, dtype, D, L, K):
    """Ragged Len_q, every head_dim, L*K up to 256 (several record chunks per
    query), samples partly outside the maps."""
    levels = [(3 + (l % 4), 2 + (l * 3) % 7) for l in range(L)]
    w = workloads.custom(N=2, M=3, D=D, levels=levels, K=K, Len_q=23, dtype=dtype, refs="uniform",
                         ref_range=(-0.05, 1.05), offset_sigma=0.2, seed=500 + D + 7 * L + K)
    p = H.prepared(w)
    _check_backward_fused(w, _run_backward_fused(msda, w, p), _oracle_backward_fused(p))


def test_fused_backward_dense_merge_and_accumulate(msda):
    """Dense small maps (merge table on every level) and MSDA_ACCUMULATE_GRAD_VALUE."""
    w = workloads.custom(N=1, M=2, D=32, levels=[(4, 6), (2, 3)], K=4, Len_q=203, refs="uniform",
                         ref_range=(0.0, 1.0), offset_sigma=0.15, seed=808)
    p = H.prepared(w)
    ref = _oracle_backward_fused(p)
    got = _run_backward_fused(msda, w, p)
    _check_backward_fused(w, got, ref)
    ref_gv = ref.for_gpu(got)[0]
    gv0 = np.random.Generator(np.random.PCG64(9)).standard_normal(p["value"].shape).astype(np.float32)
    for flags in (msda.MSDA_ACCUMULATE_GRAD_VALUE, msda.MSDA_ACCUMULATE_GRAD_VALUE | msda.MSDA_DETERMINISTIC):
        gv = H.dev(gv0)
        msda.msda_backward_fused(H.dev(p["value"]), p["spatial_shapes"], p["level_start_index"],
                                 H.dev(p["reference_points"]), H.dev(p["sampling_offsets"]),
                                 H.dev(p["attention_logits"]), H.dev(p["grad_output"]), grad_value=gv, flags=flags)
        H.assert_bwd(gv.cpu().numpy(), gv0 + ref_gv, "f32", "fused accumulated grad_value")


@pytest.mark.parametrize("dtype,D", [("bf16", 8), ("f32", 16), ("bf16", 32), ("f32", 64)])
@pytest.mark.parametrize("trend", ["rising", "falling", "spike"])
def test_fused_forward_rows_of_many_chunks(msda, dtype, D, trend):
    """Rows of L*K = 48 logits spread over up to 24 record chunks (the forward
    sums the softmax online, rescaling at every new maximum): logits rising
    along the row (a new maximum in every chunk), falling (none after the
    first), and one spike 30 above the rest in the last chunk."""
    levels = [(5, 6), (3, 4), (2, 2), (1, 3)]
    w = workloads.custom(N=2, M=3, D=D, levels=levels, K=12, Len_q=19, dtype=dtype, refs="uniform",
                         ref_range=(0.0, 1.0), offset_sigma=0.3, seed=1600 + D)
    p = dict(H.prepared(w))
    P = 4 * 12
    base = p["attention_logits"].reshape(-1, P).astype(np.float32)
    ramp = np.linspace(-6.0, 6.0, P, dtype=np.float32)
    if trend == "rising":
        lg = base * 0.1 + ramp
    elif trend == "falling":
        lg = base * 0.1 - ramp
    else:
        lg = base.copy()
        lg[:, -1] += 30.0
    p["attention_logits"] = lg.reshape(p["attention_logits"].shape)
    ref = oracle.forward_fused(p["value"], p["spatial_shapes"], p["level_start_index"], p["reference_points"],
                               p["sampling_offsets"], p["attention_logits"])
    H.assert_fwd(_run_fused(msda, w, p), ref, dtype, f"fused forward, {trend} logits")


# ----------------------------------------------------------------- options (per-level softmax, align_corners)
OPT_CASES = [("per_level", 1), ("align", 2), ("both", 3)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("D", [8, 32])
@pytest.mark.parametrize("oname,opt", OPT_CASES, ids=[c[0] for c in OPT_CASES])
def test_options_all_calls(msda, dtype, D, oname, opt):
    """Every call under each option, against the oracle with the same option.
    L*K = 35 with K = 7: levels straddle the record chunks of the backward."""
    levels = [(5, 7), (3, 4), (1, 1), (6, 2), (2, 3)]
    w = workloads.custom(N=2, M=3, D=D, levels=levels, K=7, Len_q=27, dtype=dtype, refs="uniform",
                         ref_range=(-0.05, 1.05), offset_sigma=0.2, seed=900 + D + opt)
    p = H.prepared(w)
    dt = H.storage_dtype(w)
    v, g = H.dev(p["value"], dt), H.dev(p["grad_output"], dt)
    sh, st = p["spatial_shapes"], p["level_start_index"]
    ref, off, lg = H.dev(p["reference_points"]), H.dev(p["sampling_offsets"]), H.dev(p["attention_logits"])
    loc, attn = H.dev(p["sampling_locations"]), H.dev(p["attention_weights"])
    # unfused calls (the per-level bit has no effect there)
    out = msda.msda_forward(v, sh, st, loc, attn, options=opt).float().cpu().numpy()
    H.assert_fwd(out, oracle.forward(p["value"], sh, st, p["sampling_locations"], p["attention_weights"],
                                     options=opt), dtype, f"{oname} forward")
    ref_b = _oracle_backward(p, opt)
    for flags in (0, msda.MSDA_DETERMINISTIC):
        got = msda.msda_backward(v, sh, st, loc, attn, g, flags=flags, options=opt)
        _check_backward(w, [t.cpu().numpy() for t in got], ref_b)
    # fused calls
    fo = msda.msda_forward_fused(v, sh, st, ref, off, lg, options=opt).float().cpu().numpy()
    H.assert_fwd(fo, oracle.forward_fused(p["value"], sh, st, p["reference_points"], p["sampling_offsets"],
                                          p["attention_logits"], options=opt), dtype, f"{oname} fused forward")
    ref_fb = _oracle_backward_fused(p, opt)
    for flags in (0, msda.MSDA_DETERMINISTIC):
        got = msda.msda_backward_fused(v, sh, st, ref, off, lg, g, flags=flags, options=opt)
        _check_backward_fused(w, [t.cpu().numpy() for t in got], ref_fb)


def test_options_dense_merge_path(msda):
    """Both options on dense small maps (merge table on every level)."""
    w = workloads.custom(N=1, M=2, D=32, levels=[(4, 6), (2, 3)], K=4, Len_q=203, refs="uniform",
                         ref_range=(0.0, 1.0), offset_sigma=0.15, seed=811)
    p = H.prepared(w)
    sh, st = p["spatial_shapes"], p["level_start_index"]
    got = msda.msda_backward_fused(H.dev(p["value"]), sh, st, H.dev(p["reference_points"]),
                                   H.dev(p["sampling_offsets"]), H.dev(p["attention_logits"]),
                                   H.dev(p["grad_output"]), options=3)
    _check_backward_fused(w, [t.cpu().numpy() for t in got], _oracle_backward_fused(p, 3))


# ----------------------------------------------------------------- 3-D variant (trilinear)
def _vol_case(dtype, D, seed, levels=((3, 4, 5), (2, 3, 2), (1, 1, 1), (4, 2, 3)), K=3, Lq=29, N=2, M=3):
    raw = workloads.draw_volumes(N, M, D, levels, K, Lq, dtype=dtype, loc_range=(-0.15, 1.15), seed=seed)
    L = len(levels)
    attn = oracle.softmax(raw["attention_logits"]).astype(np.float32).reshape(N, Lq, M, L, K)
    value, g = raw["value"], raw["grad_output"]
    if dtype == "bf16":
        value, g = H.bf16_round(value), H.bf16_round(g)
    return raw, value, g, attn


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("D", [8, 32, 64])
@pytest.mark.parametrize("opt", [0, 2], ids=["half_pixel", "align_corners"])
def test_3d_forward_backward(msda, dtype, D, opt):
    raw, value, g, attn = _vol_case(dtype, D, seed=1400 + D + opt)
    sh, st, loc = raw["spatial_shapes"], raw["level_start_index"], raw["sampling_locations"]
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    v, gd, locd, ad = H.dev(value, dt), H.dev(g, dt), H.dev(loc), H.dev(attn)
    out = msda.msda3d_forward(v, sh, st, locd, ad, options=opt).float().cpu().numpy()
    H.assert_fwd(out, oracle.forward3d(value, sh, st, loc, attn, options=opt), dtype, f"3-D {dtype} D={D} output")
    ref = H.backward3d_reference(dict(value=value, spatial_shapes=sh, level_start_index=st, sampling_locations=loc,
                                      attention_weights=attn, grad_output=g), opt)
    w = workloads.custom(name="volumes", N=2, M=3, D=D, levels=[(1, 1)], K=3, dtype=dtype)
    _check_backward(w, [t.cpu().numpy() for t in msda.msda3d_backward(v, sh, st, locd, ad, gd, options=opt)], ref)
    det = [[t.cpu().numpy() for t in msda.msda3d_backward(v, sh, st, locd, ad, gd, flags=msda.MSDA_DETERMINISTIC,
                                                           options=opt)] for _ in range(2)]
    _check_backward(w, det[0], ref)
    for a, b in zip(det[0], det[1]):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), "deterministic 3-D backward is not bitwise stable"


@pytest.mark.parametrize("i", range(H.RANDOM_VOLUMES))
def test_3d_random_problems(msda, i):
    """Seeded random 3-D problems (head width 8-64, 1-4 heads, 1-4 levels of
    up to 6 x 6 x 6 voxels, 1-6 points, 1-60 queries, either dtype, with and
    without align_corners): both 3-D calls, both modes, against the oracle."""
    H.check_3d_calls(msda, H.random_volume_problem(i), f"3-D case {i}")


def test_3d_one_slice_is_2d(msda):
    """One-slice volumes sampled on their centre plane give the 2-D call's result."""
    w = workloads.custom(N=1, M=2, D=32, levels=[(6, 7), (3, 4)], K=3, Len_q=19, refs="none", seed=1450)
    p = H.prepared(w)
    sh2 = p["spatial_shapes"]
    sh3 = np.concatenate([np.ones((sh2.shape[0], 1), np.int64), sh2], axis=1)
    loc3 = np.concatenate([p["sampling_locations"], np.full(p["sampling_locations"].shape[:-1] + (1,), 0.5,
                                                            np.float32)], axis=-1)
    out2 = msda.msda_forward(H.dev(p["value"]), sh2, p["level_start_index"], H.dev(p["sampling_locations"]),
                             H.dev(p["attention_weights"])).cpu().numpy()
    out3 = msda.msda3d_forward(H.dev(p["value"]), sh3, p["level_start_index"], H.dev(loc3),
                               H.dev(p["attention_weights"])).cpu().numpy()
    assert np.abs(out3 - out2).max() <= 1e-5


# ----------------------------------------------------------------- the top of the index range
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_element_offsets_near_2_31(msda, dtype):
    """Element offsets (pixel * n_heads * head_dim) within 0.4% of 2^31, the
    largest the host checks accept: a 2048 x 2040 level, then a 4 x 4 level
    whose rows start at element 2.139e9 (8.6 GB of fp32 value).  The first
    level's samples lie far outside it (all four corners padded) and, in the
    fused calls, its logits are -1e4, whose weights are exactly 0 in fp32 and
    fp64.  Every result on the small level then equals the oracle's on the
    1-level problem made of that level's data alone, and everything on the
    large level is exactly zero."""
    M, D, Lq, K = 8, 64, 64, 2
    big, small = (2048, 2040), (4, 4)
    start1 = big[0] * big[1]
    Len_in = start1 + small[0] * small[1]
    assert (Len_in + 2 * big[1] + 4) * M * D < 2 ** 31 <= (Len_in + 2 * big[1] + 4) * M * D * 1.01
    rng = np.random.Generator(np.random.PCG64(2031))
    value_s = rng.standard_normal((1, 16, M, D)).astype(np.float32)
    g = rng.standard_normal((1, Lq, M * D)).astype(np.float32)
    if dtype == "bf16":
        value_s, g = H.bf16_round(value_s), H.bf16_round(g)
    loc_s = rng.uniform(-0.15, 1.15, (1, Lq, M, 1, K, 2)).astype(np.float32)     # some corners padded
    attn_s = rng.uniform(0.1, 1.0, (1, Lq, M, 1, K)).astype(np.float32)
    ref_s = rng.uniform(0.1, 0.9, (1, Lq, 1, 2)).astype(np.float32)
    off_s = rng.normal(0.0, 1.0, (1, Lq, M, 1, K, 2)).astype(np.float32)         # pixels of the 4 x 4 level
    logit_s = rng.standard_normal((1, Lq, M, K)).astype(np.float32)
    sh_s, st_s = np.array([small], np.int64), np.array([0], np.int64)
    sh = np.array([big, small], np.int64)
    st = np.array([0, start1], np.int64)

    # the two-level problem on the device: zeros on the large level
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    value = torch.zeros((1, Len_in, M, D), dtype=dt, device="cuda")
    value[0, start1:] = torch.from_numpy(value_s[0]).to(device="cuda", dtype=dt)
    loc = np.concatenate([np.full((1, Lq, M, 1, K, 2), -3.0, np.float32), loc_s], axis=3)
    attn = np.concatenate([np.full((1, Lq, M, 1, K), 0.3, np.float32), attn_s], axis=3)
    ref = np.concatenate([np.full((1, Lq, 1, 2), -3.0, np.float32), ref_s], axis=2)
    off = np.concatenate([np.zeros((1, Lq, M, 1, K, 2), np.float32), off_s], axis=3)
    logit = np.concatenate([np.full((1, Lq, M, K), -1e4, np.float32), logit_s], axis=3)
    gd = H.dev(g, dt)

    def small_level(x):            # [N, Len_in, M, D] -> the small level's rows, and the rest's largest |x|
        lo, hi = torch.aminmax(x[0, :start1])
        rest = max(-float(lo), float(hi))
        return x[:, start1:].cpu().numpy(), rest

    # unfused
    out = msda.msda_forward(value, sh, st, H.dev(loc), H.dev(attn)).float().cpu().numpy()
    H.assert_fwd(out, oracle.forward(value_s, sh_s, st_s, loc_s, attn_s), dtype, "forward near 2^31")
    bref = H.backward_reference(dict(value=value_s, spatial_shapes=sh_s, level_start_index=st_s,
                                     sampling_locations=loc_s, attention_weights=attn_s, grad_output=g))
    for flags in (0, msda.MSDA_DETERMINISTIC):
        gv, gl, ga = msda.msda_backward(value, sh, st, H.dev(loc), H.dev(attn), gd, flags=flags)
        gv_small, gv_rest = small_level(gv)
        assert gv_rest == 0.0, f"grad_value on the outside level: {gv_rest}"
        gl, ga = gl.cpu().numpy(), ga.cpu().numpy()
        assert not gl[:, :, :, 0].any() and not ga[:, :, :, 0].any()
        gv_r, gl_r, ga_r = bref.for_gpu((gv_small, gl[:, :, :, 1:], ga[:, :, :, 1:]))
        H.assert_bwd(gv_small, gv_r, "f32", f"grad_value near 2^31 (flags {flags})")
        H.assert_bwd(gl[:, :, :, 1:], gl_r, "f32", f"grad_loc near 2^31 (flags {flags})")
        H.assert_bwd(ga[:, :, :, 1:], ga_r, "f32", f"grad_attn near 2^31 (flags {flags})")
        del gv
    # fused
    fo = msda.msda_forward_fused(value, sh, st, H.dev(ref), H.dev(off), H.dev(logit.reshape(1, Lq, M, 2 * K)))
    H.assert_fwd(fo.float().cpu().numpy(), oracle.forward_fused(value_s, sh_s, st_s, ref_s, off_s, logit_s), dtype,
                 "fused forward near 2^31")
    fref = H.backward_fused_reference(dict(value=value_s, spatial_shapes=sh_s, level_start_index=st_s,
                                           reference_points=ref_s, sampling_offsets=off_s, attention_logits=logit_s,
                                           grad_output=g))
    for flags in (0, msda.MSDA_DETERMINISTIC):
        gv, gref, goff, glog = msda.msda_backward_fused(value, sh, st, H.dev(ref), H.dev(off),
                                                        H.dev(logit.reshape(1, Lq, M, 2 * K)), gd, flags=flags)
        gv_small, gv_rest = small_level(gv)
        assert gv_rest == 0.0, f"fused grad_value on the outside level: {gv_rest}"
        gref, goff = gref.cpu().numpy(), goff.cpu().numpy()
        glog = glog.cpu().numpy().reshape(1, Lq, M, 2, K)
        assert not gref[:, :, 0].any() and not goff[:, :, :, 0].any() and not glog[:, :, :, 0].any()
        fr = fref.for_gpu((gv_small, gref[:, :, 1:], goff[:, :, :, 1:], glog[:, :, :, 1]))
        H.assert_bwd(gv_small, fr[0], "f32", f"fused grad_value near 2^31 (flags {flags})")
        H.assert_bwd(gref[:, :, 1:], fr[1], "f32", f"fused grad_ref near 2^31 (flags {flags})")
        H.assert_bwd(goff[:, :, :, 1:], fr[2], "f32", f"fused grad_off near 2^31 (flags {flags})")
        H.assert_bwd(glog[:, :, :, 1], fr[3].reshape(1, Lq, M, K), "f32", f"fused grad_logit near 2^31 (flags {flags})")
        del gv


# ----------------------------------------------------------------- the data-parallel split
def _slice(p, keys, sl):
    return {k: (np.ascontiguousarray(v[sl]) if k in keys else v) for k, v in p.items()}


BATCHED = ("value", "sampling_locations", "attention_weights", "grad_output", "reference_points",
           "sampling_offsets", "attention_logits")


def _bitwise(a, b, what):
    a, b = np.ascontiguousarray(a, np.float32), np.ascontiguousarray(b, np.float32)
    assert a.shape == b.shape and np.array_equal(a.view(np.uint32), b.view(np.uint32)), f"{what} differs"


def test_batch_split_matches_one_call(msda):
    """Ranks that take whole batch elements (the split bench.py makes under
    torchrun) compute exactly what one call on the whole batch computes: the
    encoder training problem as one N=2 call and as two N=1 calls gives
    bitwise the same forward, fused forward and per-sample gradients, and, in
    deterministic mode, the same grad_value (each batch element's fixed-point
    scale comes from its own rows alone)."""
    w = workloads.WORKLOADS["encoder_train"]
    p = H.prepared(w)
    halves = [_slice(p, BATCHED, slice(n, n + 1)) for n in range(w.N)]
    whole = {"fwd": _run_forward(msda, w, p), "fused": _run_fused(msda, w, p),
             "bwd": _run_backward(msda, w, p, msda.MSDA_DETERMINISTIC),
             "bwd_atomic": _run_backward(msda, w, p),
             "fbwd": _run_backward_fused(msda, w, p, msda.MSDA_DETERMINISTIC)}
    parts = [{"fwd": _run_forward(msda, w, h), "fused": _run_fused(msda, w, h),
              "bwd": _run_backward(msda, w, h, msda.MSDA_DETERMINISTIC),
              "bwd_atomic": _run_backward(msda, w, h),
              "fbwd": _run_backward_fused(msda, w, h, msda.MSDA_DETERMINISTIC)} for h in halves]
    for n, part in enumerate(parts):
        _bitwise(part["fwd"], whole["fwd"][n:n + 1], f"forward of batch element {n}")
        _bitwise(part["fused"], whole["fused"][n:n + 1], f"fused forward of batch element {n}")
        for name, a, b in zip(("grad_value", "grad_sampling_locations", "grad_attention_weights"), part["bwd"],
                              whole["bwd"]):
            _bitwise(a, b[n:n + 1], f"deterministic {name} of batch element {n}")
        # atomic mode: the per-sample gradients use no atomics
        for name, a, b in zip(("grad_sampling_locations", "grad_attention_weights"), part["bwd_atomic"][1:],
                              whole["bwd_atomic"][1:]):
            _bitwise(a, b[n:n + 1], f"{name} of batch element {n}")
        for name, a, b in zip(("grad_value", "grad_reference_points", "grad_sampling_offsets",
                               "grad_attention_logits"), part["fbwd"], whole["fbwd"]):
            _bitwise(a, b[n:n + 1], f"deterministic fused {name} of batch element {n}")


def test_query_split_of_one_batch_element(msda):
    """The queries of one image split over two calls (ranks that would share
    its value map): the outputs and per-sample gradients of the two halves
    are bitwise those of one call, and the two grad_value halves, summed on the
    host (the all-reduce such a split needs), match the oracle.  The split
    point is not a multiple of the queries a warp owns."""
    w = workloads.WORKLOADS["encoder_train"]
    p = _slice(H.prepared(w), BATCHED, slice(0, 1))
    cut = 11111
    q_keys = ("sampling_locations", "attention_weights", "grad_output", "reference_points", "sampling_offsets",
              "attention_logits")
    halves = [_slice(p, q_keys, (slice(None), slice(0, cut))), _slice(p, q_keys, (slice(None), slice(cut, None)))]
    whole_fwd = _run_forward(msda, w, p)
    whole_bwd = _run_backward(msda, w, p, msda.MSDA_DETERMINISTIC)
    gv_sum = np.zeros(p["value"].shape, np.float64)
    for i, (h, sl) in enumerate(zip(halves, (slice(0, cut), slice(cut, None)))):
        _bitwise(_run_forward(msda, w, h), whole_fwd[:, sl], f"forward of query half {i}")
        gv, gl, ga = _run_backward(msda, w, h, msda.MSDA_DETERMINISTIC)
        _bitwise(gl, whole_bwd[1][:, sl], f"grad_sampling_locations of query half {i}")
        _bitwise(ga, whole_bwd[2][:, sl], f"grad_attention_weights of query half {i}")
        gv_sum += gv
    ref = _oracle_backward(p).for_gpu((gv_sum, whole_bwd[1], whole_bwd[2]))
    H.assert_bwd(gv_sum, ref[0], "f32", "grad_value summed over the query halves")


# ----------------------------------------------------------------- head groups sharing one set of locations
PER_SAMPLE = ("sampling_locations", "attention_weights", "sampling_offsets", "attention_logits")


def _grouped(p, G):
    """The inputs cut to G sets of locations and weights: the per-sample tensors
    keep their first G heads' sets, shared by groups of M / G heads."""
    return {k: (np.ascontiguousarray(v[:, :, :G]) if k in PER_SAMPLE else v) for k, v in p.items()}


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("G,K", [(1, 4), (2, 4), (4, 4), (1, 20)])
def test_grouped_locations_all_calls(msda, dtype, G, K):
    """8 heads of 32 channels in G groups that each share one set of locations
    and weights (the DAT pages' sampler): the kernels sample 256 / G channels a
    set (G = 1: two 16-byte vectors a lane in fp32).  Every call against the
    oracle's grouped form; K = 20 gives rows of 80 samples over two record
    chunks.  Ragged Len_q, samples partly outside the maps."""
    levels = [(23, 31), (12, 16), (6, 8), (3, 4)]
    w = workloads.custom(N=2, M=8, D=32, levels=levels, K=K, Len_q=53, dtype=dtype, refs="uniform",
                         ref_range=(-0.05, 1.05), offset_sigma=0.1, seed=2000 + 10 * G + K)
    p = _grouped(H.prepared(w), G)
    dt = H.storage_dtype(w)
    v, g = H.dev(p["value"], dt), H.dev(p["grad_output"], dt)
    sh, st = p["spatial_shapes"], p["level_start_index"]
    loc, attn = H.dev(p["sampling_locations"]), H.dev(p["attention_weights"])
    ref, off, lg = H.dev(p["reference_points"]), H.dev(p["sampling_offsets"]), H.dev(p["attention_logits"])
    out = msda.msda_forward(v, sh, st, loc, attn).float().cpu().numpy()
    H.assert_fwd(out, oracle.forward(p["value"], sh, st, p["sampling_locations"], p["attention_weights"]), dtype,
                 f"G={G} forward")
    fo = msda.msda_forward_fused(v, sh, st, ref, off, lg).float().cpu().numpy()
    H.assert_fwd(fo, oracle.forward_fused(p["value"], sh, st, p["reference_points"], p["sampling_offsets"],
                                          p["attention_logits"]), dtype, f"G={G} fused forward")
    ref_b, ref_fb = _oracle_backward(p), _oracle_backward_fused(p)
    for flags in (0, msda.MSDA_DETERMINISTIC):
        got = [t.cpu().numpy() for t in msda.msda_backward(v, sh, st, loc, attn, g, flags=flags)]
        _check_backward(w, got, ref_b)
        got = [t.cpu().numpy() for t in msda.msda_backward_fused(v, sh, st, ref, off, lg, g, flags=flags)]
        _check_backward_fused(w, got, ref_fb)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,D", [(1, 128), (1, 256), (3, 128)])
def test_wide_heads(msda, dtype, M, D):
    """head_dim 128 and 256 without groups: one query a warp, 64 record slots a
    row; ragged Len_q and level sizes, both backward modes."""
    w = workloads.custom(N=2, M=M, D=D, levels=RAGGED_LEVELS, K=3, Len_q=19, dtype=dtype, refs="uniform",
                         ref_range=(-0.05, 1.05), offset_sigma=0.2, seed=2100 + D + M)
    p = H.prepared(w)
    H.assert_fwd(_run_forward(msda, w, p), _oracle_forward(p), dtype, f"D={D} output")
    fr = oracle.forward_fused(p["value"], p["spatial_shapes"], p["level_start_index"], p["reference_points"],
                              p["sampling_offsets"], p["attention_logits"])
    H.assert_fwd(_run_fused(msda, w, p), fr, dtype, f"D={D} fused output")
    ref_b, ref_fb = _oracle_backward(p), _oracle_backward_fused(p)
    for flags in (0, msda.MSDA_DETERMINISTIC):
        _check_backward(w, _run_backward(msda, w, p, flags), ref_b)
        _check_backward_fused(w, _run_backward_fused(msda, w, p, flags), ref_fb)


@pytest.mark.parametrize("M,D,K", [(3, 32, 5), (2, 64, 3), (1, 128, 4), (1, 256, 2)])
@pytest.mark.parametrize("opt", [0, 1, 2], ids=["row_softmax", "per_level", "align"])
def test_pixel_queries_band_order(msda, M, D, K, opt):
    """One query per value pixel (Len_q == Len_in, the encoder's shape): the
    fp32 forward takes each head's queries in bands of four rows, walked
    column by column.  Level heights that are no multiple of four (a short
    last band), odd widths and one-row levels; every head width the forward
    takes head-major, unfused and fused: K = 5 at D = 32 is two record chunks
    a row (the online softmax), the other widths one (the one-chunk kernels);
    the per-level softmax, and align_corners (option code in the one-chunk
    kernels)."""
    w = workloads.custom(N=2, M=M, D=D, levels=[(7, 9), (5, 3), (1, 5), (2, 1)], K=K, offset_sigma=0.1,
                         seed=2300 + D + opt)
    p = H.prepared(w)
    assert w.Lq == w.Len_in == 85
    sh, st = p["spatial_shapes"], p["level_start_index"]
    if opt == 0:
        H.assert_fwd(_run_forward(msda, w, p), _oracle_forward(p), "f32", f"D={D} pixel queries")
    fo = msda.msda_forward_fused(H.dev(p["value"]), sh, st, H.dev(p["reference_points"]),
                                 H.dev(p["sampling_offsets"]), H.dev(p["attention_logits"]), options=opt)
    ref = oracle.forward_fused(p["value"], sh, st, p["reference_points"], p["sampling_offsets"],
                               p["attention_logits"], options=opt)
    H.assert_fwd(fo.float().cpu().numpy(), ref, "f32", f"D={D} pixel queries, fused, options {opt}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_band_order_with_any_queries(msda, dtype):
    """Len_q == Len_in with queries that are not the value pixels (reference
    points drawn at random): the fp32 forward still takes them in band order,
    which only permutes the rows; unfused and fused against the oracle."""
    w = workloads.custom(N=2, M=2, D=32, levels=[(6, 5), (3, 7), (2, 2)], K=4, dtype=dtype, refs="uniform",
                         ref_range=(-0.05, 1.05), offset_sigma=0.2, seed=2400)
    p = H.prepared(w)
    assert w.Lq == w.Len_in
    H.assert_fwd(_run_forward(msda, w, p), _oracle_forward(p), dtype, "random queries, band order")
    ref = oracle.forward_fused(p["value"], p["spatial_shapes"], p["level_start_index"], p["reference_points"],
                               p["sampling_offsets"], p["attention_logits"])
    H.assert_fwd(_run_fused(msda, w, p), ref, dtype, "random queries, band order, fused")


@pytest.mark.parametrize("i", range(H.RANDOM_PROBLEMS))
def test_random_problems_all_calls(msda, i):
    """Seeded random problems: head width 8-256, 1-8 heads in any supported
    grouping, 1-5 levels of 1-12 x 1-12 pixels, 1-8 points, Len_q either every
    pixel (band order in the fp32 forward) or 1-69 random queries, either dtype,
    every option combination; every call against the oracle, both backward
    modes."""
    w, opt, G = H.random_problem(i)
    p = H.grouped(H.prepared(w), G)
    dt = H.storage_dtype(w)
    v, g = H.dev(p["value"], dt), H.dev(p["grad_output"], dt)
    sh, st = p["spatial_shapes"], p["level_start_index"]
    loc, attn = H.dev(p["sampling_locations"]), H.dev(p["attention_weights"])
    ref, off, lg = H.dev(p["reference_points"]), H.dev(p["sampling_offsets"]), H.dev(p["attention_logits"])
    what = f"case {i}: N={w.N} M={w.M} G={G} D={w.D} levels={w.levels} K={w.K} Lq={w.Lq} {w.dtype} options={opt}"
    out = msda.msda_forward(v, sh, st, loc, attn, options=opt).float().cpu().numpy()
    H.assert_fwd(out, oracle.forward(p["value"], sh, st, p["sampling_locations"], p["attention_weights"],
                                     options=opt), w.dtype, what + " forward")
    fo = msda.msda_forward_fused(v, sh, st, ref, off, lg, options=opt).float().cpu().numpy()
    H.assert_fwd(fo, oracle.forward_fused(p["value"], sh, st, p["reference_points"], p["sampling_offsets"],
                                          p["attention_logits"], options=opt), w.dtype, what + " fused forward")
    ref_b, ref_fb = _oracle_backward(p, opt), _oracle_backward_fused(p, opt)
    for flags in (0, msda.MSDA_DETERMINISTIC):
        got = msda.msda_backward(v, sh, st, loc, attn, g, flags=flags, options=opt)
        _check_backward(w, [t.cpu().numpy() for t in got], ref_b)
        got = msda.msda_backward_fused(v, sh, st, ref, off, lg, g, flags=flags, options=opt)
        _check_backward_fused(w, [t.cpu().numpy() for t in got], ref_fb)


def test_group_count_must_divide_the_heads(msda):
    w = workloads.custom(N=1, M=6, D=8, levels=[(4, 4)], K=2, Len_q=5, refs="none", seed=3)
    p = H.prepared(w)
    with pytest.raises(ValueError):
        msda.msda_forward(H.dev(p["value"]), p["spatial_shapes"], p["level_start_index"],
                          H.dev(p["sampling_locations"][:, :, :4]), H.dev(p["attention_weights"][:, :, :4]))
    # 6 heads of 8 channels in 3 groups: 16 channels a set, supported
    out = msda.msda_forward(H.dev(p["value"]), p["spatial_shapes"], p["level_start_index"],
                            H.dev(p["sampling_locations"][:, :, :3]), H.dev(p["attention_weights"][:, :, :3]))
    ref = oracle.forward(p["value"], p["spatial_shapes"], p["level_start_index"], p["sampling_locations"][:, :, :3],
                         p["attention_weights"][:, :, :3])
    H.assert_fwd(out.cpu().numpy(), ref, "f32", "6 heads in 3 groups")
