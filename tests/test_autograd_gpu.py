"""The autograd Functions of the binding: backward through each of them gives
exactly the gradients of the direct backward call it wraps (deterministic
mode, so the comparison is bitwise), in the dtypes autograd expects.  The
direct calls are held to the oracle by the parity tests."""
import pytest
import torch

import harness as H
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msda():
    import scale_deformable_attention_06_b300 as m
    assert torch.cuda.is_available(), "these tests need a CUDA device"
    return m


def _workload(dtype):
    # two batch elements, ragged levels, queries with uniform reference points
    return workloads.custom(N=2, M=4, D=32, levels=[(6, 9), (3, 5), (2, 2)], K=3, Len_q=37, dtype=dtype,
                            refs="uniform", offset_sigma=0.05, seed=4242)


def _leaf(a, dtype=torch.float32):
    return H.dev(a, dtype).requires_grad_()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_function_equals_the_direct_calls(msda, dtype):
    w = _workload(dtype)
    p = H.prepared(w)
    dt = H.storage_dtype(w)
    sh, st = p["spatial_shapes"], p["level_start_index"]
    value, loc, attn = _leaf(p["value"], dt), _leaf(p["sampling_locations"]), _leaf(p["attention_weights"])
    g = H.dev(p["grad_output"], dt)
    out = msda.MSDeformAttnFunction.apply(value, sh, st, loc, attn, msda.MSDA_DETERMINISTIC)
    assert out.dtype == dt and out.requires_grad
    assert torch.equal(out, msda.msda_forward(value.detach(), sh, st, loc.detach(), attn.detach()))
    out.backward(g)
    gv, gl, ga = msda.msda_backward(value.detach(), sh, st, loc.detach(), attn.detach(), g,
                                    flags=msda.MSDA_DETERMINISTIC)
    assert value.grad.dtype == dt
    assert torch.equal(value.grad, gv.to(dt))
    assert torch.equal(loc.grad, gl) and torch.equal(attn.grad, ga)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_function_equals_the_direct_calls(msda, dtype):
    w = _workload(dtype)
    p = H.prepared(w)
    dt = H.storage_dtype(w)
    sh, st = p["spatial_shapes"], p["level_start_index"]
    value = _leaf(p["value"], dt)
    ref, off, lg = _leaf(p["reference_points"]), _leaf(p["sampling_offsets"]), _leaf(p["attention_logits"])
    g = H.dev(p["grad_output"], dt)
    out = msda.MSDeformAttnFusedFunction.apply(value, sh, st, ref, off, lg, msda.MSDA_DETERMINISTIC)
    direct = msda.msda_forward_fused(value.detach(), sh, st, ref.detach(), off.detach(), lg.detach())
    assert torch.equal(out, direct)
    # a loss of the output: autograd hands the Function d loss / d out = g
    (out.float() * g.float()).sum().backward()
    gv, gref, goff, glg = msda.msda_backward_fused(value.detach(), sh, st, ref.detach(), off.detach(), lg.detach(),
                                                    g, flags=msda.MSDA_DETERMINISTIC)
    assert torch.equal(value.grad, gv.to(dt))
    assert torch.equal(ref.grad, gref) and torch.equal(off.grad, goff) and torch.equal(lg.grad, glg)


def test_function_under_a_torch_graph(msda):
    """Locations formed by torch ops upstream of the Function receive their
    gradients through it by the chain rule (loc = ref + off / (W, H))."""
    w = _workload("f32")
    p = H.prepared(w)
    sh, st = p["spatial_shapes"], p["level_start_index"]
    value = H.dev(p["value"])
    ref, off = _leaf(p["reference_points"]), _leaf(p["sampling_offsets"])
    wh = torch.tensor([[wl, hl] for (hl, wl) in w.levels], dtype=torch.float32, device="cuda")
    loc = ref[:, :, None, :, None, :] + off / wh[None, None, None, :, None, :]
    attn = H.dev(p["attention_weights"])
    out = msda.MSDeformAttnFunction.apply(value, sh, st, loc, attn, msda.MSDA_DETERMINISTIC)
    g = H.dev(p["grad_output"])
    out.backward(g)
    _, gl, _ = msda.msda_backward(value, sh, st, loc.detach(), attn, g, flags=msda.MSDA_DETERMINISTIC)
    assert value.grad is None
    torch.testing.assert_close(off.grad, gl / wh[None, None, None, :, None, :], rtol=0, atol=0)
    torch.testing.assert_close(ref.grad, gl.sum(dim=(2, 4)), rtol=1e-5, atol=1e-5)   # torch's own summation order


def test_3d_function_equals_the_direct_calls(msda):
    raw, value_h, g_h, attn_h, dtype, opt = H.random_volume_problem(3)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    sh, st = raw["spatial_shapes"], raw["level_start_index"]
    value, loc, attn = _leaf(value_h, dt), _leaf(raw["sampling_locations"]), _leaf(attn_h)
    g = H.dev(g_h, dt)
    out = msda.MSDeformAttn3DFunction.apply(value, sh, st, loc, attn, msda.MSDA_DETERMINISTIC, opt)
    assert torch.equal(out, msda.msda3d_forward(value.detach(), sh, st, loc.detach(), attn.detach(), options=opt))
    out.backward(g)
    gv, gl, ga = msda.msda3d_backward(value.detach(), sh, st, loc.detach(), attn.detach(), g,
                                      flags=msda.MSDA_DETERMINISTIC, options=opt)
    assert torch.equal(value.grad, gv.to(dt)) and torch.equal(loc.grad, gl) and torch.equal(attn.grad, ga)


def test_accumulate_flag(msda):
    """The bindings refuse MSDA_ACCUMULATE_GRAD_VALUE without a grad_value to
    add into; the Functions drop it (autograd sums into .grad itself)."""
    w = _workload("f32")
    p = H.prepared(w)
    sh, st = p["spatial_shapes"], p["level_start_index"]
    value, loc, attn, g = (H.dev(p[k]) for k in ("value", "sampling_locations", "attention_weights", "grad_output"))
    with pytest.raises(ValueError, match="pass grad_value"):
        msda.msda_backward(value, sh, st, loc, attn, g, flags=msda.MSDA_ACCUMULATE_GRAD_VALUE)
    leaf = value.clone().requires_grad_()
    flags = msda.MSDA_DETERMINISTIC | msda.MSDA_ACCUMULATE_GRAD_VALUE
    msda.MSDeformAttnFunction.apply(leaf, sh, st, loc, attn, flags).backward(g)
    gv, _, _ = msda.msda_backward(value, sh, st, loc, attn, g, flags=msda.MSDA_DETERMINISTIC)
    assert torch.equal(leaf.grad, gv)
