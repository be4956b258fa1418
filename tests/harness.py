"""Shared helpers of the parity tests: inputs of each call built from the
seeded raw draws, the oracle's answers, and the tolerance checks.

The oracle turns the raw draws into the inputs of the unfused calls
(locations from reference points and offsets, weights from logits); those
fp32 inputs then go to both sides unchanged.
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


def prepared(w, raw=None):
    """All host inputs of workload `w` as float32 (value and grad_output already
    rounded to bf16 when the workload stores bf16)."""
    raw = workloads.draw(w) if raw is None else raw
    loc, attn = unfused_inputs(w, raw)
    value, g = raw["value"], raw["grad_output"]
    if w.dtype == "bf16":
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
