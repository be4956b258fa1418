"""msda_backward_noalloc: the deterministic backward for callers that may not
allocate device memory (a plugin handed only its input and output buffers, a
loop that must not call cudaMalloc after start-up).  Its scratch is a device
array inside the library, so it takes no workspace.

This file is collected last on purpose: if its GPU test fails, a run that
stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import harness as H
import workloads


def _load():
    import __graft_entry__
    __graft_entry__.build()
    import scale_deformable_attention_06_b300 as m
    return m


def _case(case):
    if case in ("tiny", "tiny_accumulate"):
        return workloads.WORKLOADS["tiny"]
    dtype = "bf16" if case == "ragged_bf16" else "f32"
    return workloads.custom(N=2, M=8, D=32, levels=[(23, 31), (12, 16), (6, 8), (3, 4)], K=4, Len_q=301,
                            dtype=dtype, refs="uniform", offset_sigma=0.1, seed=77)


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["tiny", "ragged", "ragged_bf16", "tiny_accumulate"])
def test_noalloc_matches_backward_on_two_calls_in_a_row(case):
    """Two calls in a row through the C ABI, each checked against msda_backward
    (deterministic mode, own workspace) and against the oracle.  bf16: value
    and grad_output stored in bf16 (the oracle takes the same rounded inputs).
    accumulate: grad_value starts from a given field and the call adds into
    it (MSDA_ACCUMULATE_GRAD_VALUE)."""
    msda = _load()
    assert torch.cuda.is_available()
    w = _case(case)
    accumulate = case.endswith("accumulate")
    p = H.prepared(w)
    dt = H.storage_dtype(w)
    value, g = H.dev(p["value"], dt), H.dev(p["grad_output"], dt)
    loc, attn = H.dev(p["sampling_locations"]), H.dev(p["attention_weights"])
    sh, st = p["spatial_shapes"], p["level_start_index"]
    flags = msda.MSDA_ACCUMULATE_GRAD_VALUE if accumulate else 0
    gv0 = np.random.Generator(np.random.PCG64(31)).standard_normal(p["value"].shape).astype(np.float32)

    # the existing entry point, deterministic mode, with its own workspace
    gv_ref = H.dev(gv0) if accumulate else None
    ref = msda.msda_backward(value, sh, st, loc, attn, g, grad_value=gv_ref, flags=msda.MSDA_DETERMINISTIC | flags)
    torch.cuda.synchronize()
    ref = [t.cpu().numpy() for t in ref]
    orc = H.backward_reference(p)          # the oracle, cell edges resolved as the harness says

    names = ("grad_value", "grad_sampling_locations", "grad_attention_weights")
    for call in range(2):
        # outputs come from the caller; junk in them shows they are overwritten
        gv = H.dev(gv0) if accumulate else torch.full(value.shape, float(7 + call), dtype=torch.float32,
                                                        device="cuda")
        gl = torch.full(loc.shape, -3.0, dtype=torch.float32, device="cuda")
        ga = torch.full(attn.shape, 5.0, dtype=torch.float32, device="cuda")
        msda.msda_backward_noalloc(value, sh, st, loc, attn, g, gv, gl, ga, flags=flags)
        torch.cuda.synchronize()
        got = [t.cpu().numpy() for t in (gv, gl, ga)]
        want = list(orc.for_gpu([got[0] - gv0 if accumulate else got[0], got[1], got[2]]))
        if accumulate:
            want[0] = want[0] + gv0
        for name, g_, w_, exact in zip(names, got, want, ref):
            H.assert_bwd(g_, w_, "f32", f"{case} call {call + 1}: {name} against the oracle")
            H.assert_bwd(g_, exact, "f32", f"{case} call {call + 1}: {name} against msda_backward")


@pytest.mark.gpu
def test_noalloc_binding_refuses_short_outputs():
    """A caller-passed output of the wrong size or dtype is refused in Python,
    before the library is called."""
    msda = _load()
    w = workloads.WORKLOADS["tiny"]
    p = H.prepared(w)
    value, g = H.dev(p["value"]), H.dev(p["grad_output"])
    loc, attn = H.dev(p["sampling_locations"]), H.dev(p["attention_weights"])
    sh, st = p["spatial_shapes"], p["level_start_index"]
    gl, ga = torch.empty_like(loc), torch.empty_like(attn)
    short = torch.empty((1, w.Len_in - 1, w.M, w.D), device="cuda")
    with pytest.raises(ValueError):
        msda.msda_backward_noalloc(value, sh, st, loc, attn, g, short, gl, ga)
    with pytest.raises(TypeError):
        msda.msda_backward_noalloc(value, sh, st, loc, attn, g.to(torch.bfloat16), torch.empty_like(value), gl, ga)


def test_noalloc_rejects_problems_above_its_scratch():
    """Checked on the host before anything touches the GPU."""
    msda = _load()
    lib = msda.lib()
    # 2 x 22223 x 8 x 64 = 22.8M accumulators: more than the built-in scratch holds
    p = msda.msda_problem(N=2, Len_in=22223, n_heads=8, head_dim=64, Len_q=100, n_levels=4, n_points=4, dtype=0)
    sh = (ctypes.c_int64 * 8)(100, 167, 50, 84, 25, 42, 13, 21)
    st = (ctypes.c_int64 * 4)(0, 16700, 20900, 21950)
    fake = ctypes.c_void_p(0x10000)
    rc = lib.msda_backward_noalloc(ctypes.byref(p), fake, sh, st, fake, fake, fake, fake, fake, fake, 0, None)
    assert rc == 2
    assert b"scratch" in lib.msda_last_error()
    # an unknown flag is refused too (the deterministic mode is implied)
    p.head_dim = 8
    rc = lib.msda_backward_noalloc(ctypes.byref(p), fake, sh, st, fake, fake, fake, fake, fake, fake, 1, None)
    assert rc == 1
