"""The debug build (libmsda_debug.so, -DMSDA_DEBUG): every value gather,
grad_output load and grad_value reduction of every kernel is checked against
its tensor's extent and alignment; a bad access is counted and skipped, never
trapped.  These cases run the shapes most likely to expose an index mistake
(ragged query counts and level sizes, 1 x 1 and 2 x 1 levels, samples outside
the maps, every head width, the merge table, both options, head groups, the
3-D calls, the built-in-scratch backward, and the randomized parity tests'
problems) through it, and check that nothing was skipped and that the results
still match the oracle."""
import numpy as np
import pytest
import torch

import harness as H
import oracle
import workloads

pytestmark = pytest.mark.gpu

RAGGED = [(7, 5), (3, 9), (1, 1), (2, 1)]


def _cases():
    yield "tiny", workloads.WORKLOADS["tiny"], 0, None
    for dtype in ("f32", "bf16"):
        for D in (8, 32, 64, 256):
            yield f"ragged-{dtype}-D{D}", workloads.custom(N=2, M=3 if D < 256 else 1, D=D, levels=RAGGED, K=3,
                                                           Len_q=37, dtype=dtype, refs="uniform",
                                                           ref_range=(-0.05, 1.05), offset_sigma=0.2,
                                                           seed=3100 + D), 0, None
    yield "dense-merge", workloads.custom(N=2, M=3, D=32, levels=[(5, 7), (2, 3), (1, 2)], K=4, Len_q=301,
                                          refs="uniform", ref_range=(-0.05, 1.05), offset_sigma=0.2, seed=3200), 0, None
    yield "options", workloads.custom(N=2, M=3, D=32, levels=[(5, 7), (3, 4), (1, 1)], K=7, Len_q=27, refs="uniform",
                                      ref_range=(-0.05, 1.05), offset_sigma=0.2, seed=3300), 3, None
    yield "groups", workloads.custom(N=2, M=8, D=32, levels=[(23, 31), (6, 8), (3, 4)], K=4, Len_q=53,
                                     refs="uniform", offset_sigma=0.1, seed=3400), 0, 1
    for i in range(H.RANDOM_PROBLEMS):        # the randomized parity tests' problems
        w, opt, G = H.random_problem(i)
        yield f"random-{i}", w, opt, G if G < w.M else None


@pytest.fixture(scope="module")
def debug_msda():
    import __graft_entry__
    __graft_entry__.build()
    import scale_deformable_attention_06_b300 as m
    from scale_deformable_attention_06_b300 import _capi
    with _capi.using_library(_capi.DEBUG_LIBRARY) as lib:
        lib.msda_debug_violations(1)
        yield m, lib


@pytest.mark.parametrize("name,w,opt,groups", list(_cases()), ids=[c[0] for c in _cases()])
def test_debug_build_skips_nothing(debug_msda, name, w, opt, groups):
    msda, lib = debug_msda
    p = H.prepared(w)
    if groups:
        p = {k: (np.ascontiguousarray(v[:, :, :groups]) if k in ("sampling_locations", "attention_weights",
                                                                  "sampling_offsets", "attention_logits") else v)
             for k, v in p.items()}
    dt = H.storage_dtype(w)
    v, g = H.dev(p["value"], dt), H.dev(p["grad_output"], dt)
    sh, st = p["spatial_shapes"], p["level_start_index"]
    loc, attn = H.dev(p["sampling_locations"]), H.dev(p["attention_weights"])
    out = msda.msda_forward(v, sh, st, loc, attn, options=opt).float().cpu().numpy()
    H.assert_fwd(out, oracle.forward(p["value"], sh, st, p["sampling_locations"], p["attention_weights"],
                                     options=opt), w.dtype, f"{name} forward")
    ref = H.backward_reference(p, opt)
    for flags in (0, msda.MSDA_DETERMINISTIC):
        got = [t.cpu().numpy() for t in msda.msda_backward(v, sh, st, loc, attn, g, flags=flags, options=opt)]
        for nm, a, b in zip(("grad_value", "grad_loc", "grad_attn"), got, ref.for_gpu(got)):
            H.assert_bwd(a, b, "f32", f"{name} {nm} flags {flags}")
    if "reference_points" in p:
        r, o, lg = H.dev(p["reference_points"]), H.dev(p["sampling_offsets"]), H.dev(p["attention_logits"])
        fo = msda.msda_forward_fused(v, sh, st, r, o, lg, options=opt).float().cpu().numpy()
        H.assert_fwd(fo, oracle.forward_fused(p["value"], sh, st, p["reference_points"], p["sampling_offsets"],
                                              p["attention_logits"], options=opt), w.dtype, f"{name} fused forward")
        fref = H.backward_fused_reference(p, opt)
        for flags in (0, msda.MSDA_DETERMINISTIC):
            got = [t.cpu().numpy() for t in msda.msda_backward_fused(v, sh, st, r, o, lg, g, flags=flags, options=opt)]
            for nm, a, b in zip(("grad_value", "grad_ref", "grad_off", "grad_logit"), got, fref.for_gpu(got)):
                H.assert_bwd(a.reshape(b.shape), b, "f32", f"{name} fused {nm} flags {flags}")
    torch.cuda.synchronize()
    assert lib.msda_debug_violations(1) == 0, f"{name}: the debug build skipped accesses"


def test_debug_build_3d_and_noalloc(debug_msda):
    msda, lib = debug_msda
    raw = workloads.draw_volumes(2, 3, 32, [(3, 4, 5), (1, 1, 1), (2, 3, 2)], 3, 29, loc_range=(-0.15, 1.15),
                                 seed=3500)
    sh, st, loc = raw["spatial_shapes"], raw["level_start_index"], raw["sampling_locations"]
    attn = oracle.softmax(raw["attention_logits"]).astype(np.float32).reshape(loc.shape[:-1])
    v, g = H.dev(raw["value"]), H.dev(raw["grad_output"])
    out = msda.msda3d_forward(v, sh, st, H.dev(loc), H.dev(attn)).cpu().numpy()
    H.assert_fwd(out, oracle.forward3d(raw["value"], sh, st, loc, attn), "f32", "3-D forward")
    p3 = dict(value=raw["value"], spatial_shapes=sh, level_start_index=st, sampling_locations=loc,
              attention_weights=attn, grad_output=raw["grad_output"])
    ref = H.backward3d_reference(p3)
    for flags in (0, msda.MSDA_DETERMINISTIC):
        got = [t.cpu().numpy() for t in msda.msda3d_backward(v, sh, st, H.dev(loc), H.dev(attn), g, flags=flags)]
        for nm, a, b in zip(("grad_value", "grad_loc", "grad_attn"), got, ref.for_gpu(got)):
            H.assert_bwd(a, b, "f32", f"3-D {nm} flags {flags}")
    w = workloads.WORKLOADS["tiny"]
    p = H.prepared(w)
    vv, gg = H.dev(p["value"]), H.dev(p["grad_output"])
    ll, aa = H.dev(p["sampling_locations"]), H.dev(p["attention_weights"])
    gv, gl, ga = torch.empty_like(vv), torch.empty_like(ll), torch.empty_like(aa)
    msda.msda_backward_noalloc(vv, p["spatial_shapes"], p["level_start_index"], ll, aa, gg, gv, gl, ga)
    got = [t.cpu().numpy() for t in (gv, gl, ga)]
    for nm, a, b in zip(("grad_value", "grad_loc", "grad_attn"), got, H.backward_reference(p).for_gpu(got)):
        H.assert_bwd(a, b, "f32", f"built-in scratch {nm}")
    torch.cuda.synchronize()
    assert lib.msda_debug_violations(1) == 0, "the debug build skipped accesses"


def test_debug_build_3d_random_problems(debug_msda):
    """The randomized 3-D parity tests' problems through the debug build."""
    msda, lib = debug_msda
    lib.msda_debug_violations(1)
    for i in range(H.RANDOM_VOLUMES):
        H.check_3d_calls(msda, H.random_volume_problem(i), f"3-D case {i}")
    torch.cuda.synchronize()
    assert lib.msda_debug_violations(1) == 0, "the debug build skipped accesses"
