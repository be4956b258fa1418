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


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["tiny", "ragged"])
def test_noalloc_matches_backward_on_two_calls_in_a_row(case):
    msda = _load()
    assert torch.cuda.is_available()
    if case == "tiny":
        w = workloads.WORKLOADS["tiny"]
    else:
        w = workloads.custom(N=2, M=8, D=32, levels=[(23, 31), (12, 16), (6, 8), (3, 4)], K=4, Len_q=301,
                             refs="uniform", offset_sigma=0.1, seed=77)
    p = H.prepared(w)
    value, loc, attn, g = (H.dev(p[k]) for k in ("value", "sampling_locations", "attention_weights", "grad_output"))
    sh, st = p["spatial_shapes"], p["level_start_index"]

    # the existing entry point, deterministic mode, with its own workspace
    ref = msda.msda_backward(value, sh, st, loc, attn, g, flags=msda.MSDA_DETERMINISTIC)
    torch.cuda.synchronize()
    ref = [t.cpu().numpy() for t in ref]

    for call in range(2):
        # outputs come from the caller; fill them with junk to see them overwritten
        gv = torch.full(value.shape, float(7 + call), dtype=torch.float32, device="cuda")
        gl = torch.full(loc.shape, -3.0, dtype=torch.float32, device="cuda")
        ga = torch.full(attn.shape, 5.0, dtype=torch.float32, device="cuda")
        msda.msda_backward_noalloc(value, sh, st, loc, attn, g, gv, gl, ga)
        torch.cuda.synchronize()
        for name, got, want in zip(("grad_value", "grad_sampling_locations", "grad_attention_weights"),
                                   (gv, gl, ga), ref):
            H.assert_bwd(got.cpu().numpy(), want, "f32", f"{case} call {call + 1}: {name}")


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
