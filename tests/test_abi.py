"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports
every symbol include/msda.h declares, and rejects bad arguments on the host
before any launch (no compute call is made here)."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msda.h")


@pytest.fixture(scope="module")
def msda():
    import __graft_entry__
    __graft_entry__.build()
    import scale_deformable_attention_06_b300 as m
    return m


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MSDA_API\s+[\w\s\*]+?\b(msda_\w+)\s*\(", text)))


def test_header_declares_the_three_calls():
    syms = declared_symbols()
    for name in ("msda_forward", "msda_forward_fused", "msda_backward", "msda_backward_workspace_size"):
        assert name in syms


def test_autograd_functions_refuse_host_tensors(msda):
    """Each autograd Function is a torch.autograd.Function over the library's
    calls: with host tensors its forward fails in the binding, before any C
    call, like the calls it wraps."""
    import torch
    for fn in (msda.MSDeformAttnFunction, msda.MSDeformAttnFusedFunction, msda.MSDeformAttn3DFunction):
        assert issubclass(fn, torch.autograd.Function)
    v = torch.zeros(1, 4, 1, 8)
    with pytest.raises((ValueError, TypeError)):
        msda.MSDeformAttnFunction.apply(v, [[2, 2]], [0], torch.zeros(1, 1, 1, 1, 1, 2), torch.zeros(1, 1, 1, 1, 1))


def test_accumulate_needs_a_grad_value(msda):
    """MSDA_ACCUMULATE_GRAD_VALUE adds into grad_value: without the caller's
    tensor the backward bindings refuse before allocating or calling (a fresh
    tensor would be unwritten memory).  Shapes only, so CPU tensors stand in."""
    import torch
    from scale_deformable_attention_06_b300 import _capi
    v = torch.zeros((2, 5, 3, 8), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="pass grad_value"):
        _capi._grad_value_out(v, None, msda.MSDA_ACCUMULATE_GRAD_VALUE | msda.MSDA_DETERMINISTIC)
    fresh = _capi._grad_value_out(v, None, msda.MSDA_DETERMINISTIC)
    assert fresh.shape == v.shape and fresh.dtype == torch.float32
    mine = torch.ones((2, 5, 3, 8))
    assert _capi._grad_value_out(v, mine, msda.MSDA_ACCUMULATE_GRAD_VALUE) is mine
    src = open(_capi.__file__).read()
    assert src.count("= _grad_value_out(value, grad_value, flags)") == 3     # msda_backward, _fused, msda3d_


def test_library_exports_every_declared_symbol(msda):
    out = subprocess.run(["nm", "-D", "--defined-only", msda.LIBRARY], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(msda_\w+)", out))
    missing = [s for s in declared_symbols() if s not in exported]
    assert not missing, f"declared but not exported: {missing}"
    # and nothing else leaks out under the msda_ prefix
    assert exported == set(declared_symbols())
    for s in declared_symbols():
        assert hasattr(msda.lib(), s)


def test_library_targets_sm_103a(msda):
    out = subprocess.run(["cuobjdump", "--list-elf", msda.LIBRARY], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    assert "sm_103a" in out.stdout


def _problem(msda, **kw):
    base = dict(N=1, Len_in=80, n_heads=2, head_dim=8, Len_q=80, n_levels=2, n_points=2, dtype=0)
    base.update(kw)
    return msda.msda_problem(**base)


def _levels(shapes, starts):
    sh = (ctypes.c_int64 * len(shapes))(*shapes)
    st = (ctypes.c_int64 * len(starts))(*starts)
    return sh, st


FAKE = ctypes.c_void_p(0x10000)   # never dereferenced: every call below fails its checks first


@pytest.mark.parametrize("kw,shapes,starts,expect", [
    (dict(head_dim=12), [8, 8, 4, 4], [0, 64], 2),
    (dict(head_dim=4), [8, 8, 4, 4], [0, 64], 2),
    (dict(dtype=7), [8, 8, 4, 4], [0, 64], 2),
    (dict(n_levels=17), [1, 1] * 17, list(range(17)), 2),
    (dict(n_points=200), [8, 8, 4, 4], [0, 64], 2),
    (dict(), [8, 8, 4, 4], [0, 63], 1),
    (dict(), [8, 8, 4, 4], [1, 64], 1),
    (dict(Len_in=81), [8, 8, 4, 4], [0, 64], 1),
    (dict(), [8, 0, 4, 4], [0, 0], 1),
    (dict(N=-1), [8, 8, 4, 4], [0, 64], 1),
    (dict(n_heads=0), [8, 8, 4, 4], [0, 64], 1),
    (dict(options=4), [8, 8, 4, 4], [0, 64], 1),
    (dict(n_groups=3), [8, 8, 4, 4], [0, 64], 1),                   # does not divide the 2 heads
    (dict(n_groups=-1), [8, 8, 4, 4], [0, 64], 1),
    (dict(n_heads=3, n_groups=1), [8, 8, 4, 4], [0, 64], 2),       # 24 channels a set: not a power of two
    (dict(n_heads=2, head_dim=256, n_groups=1), [8, 8, 4, 4], [0, 64], 2),   # 512 channels a set
])
def test_host_checks_reject_before_launch(msda, kw, shapes, starts, expect):
    p = _problem(msda, **kw)
    sh, st = _levels(shapes, starts)
    rc = msda.lib().msda_forward(ctypes.byref(p), FAKE, sh, st, FAKE, FAKE, FAKE, None)
    assert rc == expect, msda.lib().msda_last_error()
    assert msda.lib().msda_last_error().decode()
    rc = msda.lib().msda_forward_fused(ctypes.byref(p), FAKE, sh, st, FAKE, FAKE, FAKE, FAKE, None)
    assert rc == expect
    rc = msda.lib().msda_backward(ctypes.byref(p), FAKE, sh, st, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, None, 0, None)
    assert rc == expect
    rc = msda.lib().msda_backward_fused(ctypes.byref(p), FAKE, sh, st, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                        0, None, 0, None)
    assert rc == expect


def test_null_and_misaligned_pointers(msda):
    p = _problem(msda)
    sh, st = _levels([8, 8, 4, 4], [0, 64])
    lib = msda.lib()
    assert lib.msda_forward(ctypes.byref(p), None, sh, st, FAKE, FAKE, FAKE, None) == 1
    assert lib.msda_forward(ctypes.byref(p), ctypes.c_void_p(0x10004), sh, st, FAKE, FAKE, FAKE, None) == 1
    assert lib.msda_forward(None, FAKE, sh, st, FAKE, FAKE, FAKE, None) == 1
    assert lib.msda_forward(ctypes.byref(p), FAKE, None, st, FAKE, FAKE, FAKE, None) == 1
    # unknown backward flag
    assert lib.msda_backward(ctypes.byref(p), FAKE, sh, st, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, None, 0, None) == 1
    # deterministic mode without a workspace
    assert lib.msda_backward(ctypes.byref(p), FAKE, sh, st, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, None, 0, None) == 4
    # fused backward: a missing gradient output, a misaligned offset tensor, a bad flag, no workspace
    fb = lib.msda_backward_fused
    assert fb(ctypes.byref(p), FAKE, sh, st, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 0, None, 0, None) == 1
    assert fb(ctypes.byref(p), FAKE, sh, st, FAKE, ctypes.c_void_p(0x10004), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
              0, None, 0, None) == 1
    assert fb(ctypes.byref(p), FAKE, sh, st, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, None, 0, None) == 1
    assert fb(ctypes.byref(p), FAKE, sh, st, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, None, 0, None) == 4


def test_workspace_size(msda):
    p = _problem(msda)
    lib = msda.lib()
    assert lib.msda_backward_workspace_size(ctypes.byref(p), 0) == 0
    assert lib.msda_backward_workspace_size(ctypes.byref(p), 1) == 256 + 1 * 80 * 2 * 8 * 8
    assert lib.msda_version() > 0
    assert lib.msda_status_string(3) == b"MSDA_ERR_CUDA"


def test_binding_fails_loudly_without_the_library(tmp_path):
    """No silent fallback: without libmsda.so the package does not import."""
    code = ("import sys, os; sys.path.insert(0, %r); import scale_deformable_attention_06_b300._capi as c" % ROOT)
    env = dict(os.environ)
    pkg = os.path.join(ROOT, "scale_deformable_attention_06_b300")
    # run against a copy of the package without the .so
    dst = tmp_path / "scale_deformable_attention_06_b300"
    dst.mkdir()
    for f in ("__init__.py", "_capi.py"):
        (dst / f).write_text(open(os.path.join(pkg, f)).read())
    code = "import sys; sys.path.insert(0, %r); import scale_deformable_attention_06_b300" % str(tmp_path)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    assert r.returncode != 0 and "ImportError" in r.stderr


def test_product_path_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "scale_deformable_attention_06_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f"{f} mentions the oracle"
                assert "_work/" not in text and "/_work" not in text, f"{f} refers to working files"


@pytest.mark.parametrize("shapes,starts,Len_in,expect", [
    ([2, 3, 4, 1, 2, 2], [0, 24], 28, 0),       # valid: reaches the pointer checks (NULL value)
    ([2, 3, 4, 1, 2, 2], [0, 24], 29, 1),       # Len_in disagrees with sum D*H*W
    ([2, 0, 4, 1, 2, 2], [0, 0], 4, 1),         # empty volume
    ([2, 3, 4, 1, 2, 2], [0, 23], 28, 1),       # level start off by one
])
def test_3d_host_checks(msda, shapes, starts, Len_in, expect):
    p = _problem(msda, Len_in=Len_in, n_levels=2)
    sh, st = _levels(shapes, starts)
    lib = msda.lib()
    rc = lib.msda3d_forward(ctypes.byref(p), None if expect == 0 else FAKE, sh, st, FAKE, FAKE, FAKE, None)
    assert rc == (1 if expect == 0 else expect), lib.msda_last_error()
    rc = lib.msda3d_backward(ctypes.byref(p), FAKE, sh, st, FAKE, FAKE, FAKE, FAKE, FAKE, None if expect == 0 else FAKE,
                             0, None, 0, None)
    assert rc == (1 if expect == 0 else expect)


def test_index_limits_rejected_before_launch(msda):
    """Sizes whose element offsets would not fit the kernels' 32-bit index
    arithmetic are refused on the host (MSDA_ERR_UNSUPPORTED)."""
    lib = msda.lib()
    # a single level of 2^14 x 2^14 pixels: Len_in = 2^28 (corner records hold pixel indices below 2^28)
    p = _problem(msda, Len_in=1 << 28, n_levels=1, head_dim=8, n_heads=1)
    sh, st = _levels([1 << 14, 1 << 14], [0])
    assert lib.msda_forward(ctypes.byref(p), FAKE, sh, st, FAKE, FAKE, FAKE, None) == 2
    assert b"2^28" in lib.msda_last_error()
    # (Len_in + 2 W + 4) * n_heads * head_dim >= 2^31
    p = _problem(msda, Len_in=4096 * 4096, n_levels=1, head_dim=64, n_heads=2)
    sh, st = _levels([4096, 4096], [0])
    assert lib.msda_forward(ctypes.byref(p), FAKE, sh, st, FAKE, FAKE, FAKE, None) == 2
    assert b"2^31" in lib.msda_last_error()
    # N * Len_q * n_heads >= 2^31
    p = _problem(msda, N=1 << 16, Len_q=1 << 12, n_heads=8)
    sh, st = _levels([8, 8, 4, 4], [0, 64])
    assert lib.msda_forward(ctypes.byref(p), FAKE, sh, st, FAKE, FAKE, FAKE, None) == 2
    # the same limits for the 3-D calls
    p = _problem(msda, Len_in=1 << 28, n_levels=1, head_dim=8, n_heads=1)
    sh3, st3 = _levels([1 << 4, 1 << 12, 1 << 12], [0])
    assert lib.msda3d_forward(ctypes.byref(p), FAKE, sh3, st3, FAKE, FAKE, FAKE, None) == 2


@pytest.mark.parametrize("call", ["msda_forward", "msda_backward", "msda3d_forward"])
def test_binding_refuses_host_tensors(msda, call):
    """The binding refuses tensors that are not on a CUDA device before any
    C call: there is no CPU path."""
    import torch
    v = torch.zeros((1, 4, 1, 8))
    with pytest.raises(ValueError, match="CUDA device"):
        getattr(msda, call)(v, [[2, 2]], [0], torch.zeros((1, 2, 1, 1, 1, 2)), torch.ones((1, 2, 1, 1, 1)),
                            *([torch.zeros((1, 2, 8))] if call == "msda_backward" else []))


def test_backward_argument_checks_in_the_binding(msda):
    """The binding refuses mismatched backward tensors (and caller-passed
    outputs of the wrong size or dtype) before it calls the library: a wrong
    size there would be read or written out of bounds on the device.  Only
    shapes and dtypes are looked at, so CPU tensors stand in here."""
    import torch
    from scale_deformable_attention_06_b300 import _capi
    N, S, M, D, Lq, L, K = 2, 80, 2, 8, 5, 2, 2
    bf16 = torch.bfloat16
    ok = dict(value=torch.zeros(N, S, M, D), sampling_locations=torch.zeros(N, Lq, M, L, K, 2),
              attention_weights=torch.zeros(N, Lq, M, L, K), grad_output=torch.zeros(N, Lq, M * D),
              grad_value=torch.zeros(N, S, M, D), grad_sampling_locations=torch.zeros(N, Lq, M, L, K, 2),
              grad_attention_weights=torch.zeros(N, Lq, M, L, K))

    def call(**over):
        a = dict(ok)
        a.update(over)
        return _capi._check_backward_args(a["value"], L, a["sampling_locations"], a["attention_weights"],
                                          a["grad_output"], a["grad_value"], a["grad_sampling_locations"],
                                          a["grad_attention_weights"])

    assert call() == (Lq, L, K)
    bad = [
        (ValueError, dict(attention_weights=torch.zeros(N, Lq, M, L, K + 1))),
        (ValueError, dict(attention_weights=torch.zeros(N, Lq + 1, M, L, K))),
        (ValueError, dict(grad_output=torch.zeros(N, Lq, M * D - 1))),
        (TypeError, dict(grad_output=torch.zeros(N, Lq, M * D, dtype=bf16))),
        (ValueError, dict(sampling_locations=torch.zeros(N, Lq, M + 1, L, K, 2))),
        (ValueError, dict(sampling_locations=torch.zeros(N, Lq, M, L, K, 3))),
        (TypeError, dict(sampling_locations=torch.zeros(N, Lq, M, L, K, 2, dtype=torch.float64))),
        (ValueError, dict(sampling_locations=torch.zeros(N, Lq, M, L + 1, K, 2),
                          attention_weights=torch.zeros(N, Lq, M, L + 1, K),
                          grad_sampling_locations=torch.zeros(N, Lq, M, L + 1, K, 2),
                          grad_attention_weights=torch.zeros(N, Lq, M, L + 1, K))),      # L vs spatial_shapes
        (ValueError, dict(grad_value=torch.zeros(N, S - 1, M, D))),
        (TypeError, dict(grad_value=torch.zeros(N, S, M, D, dtype=bf16))),
        (ValueError, dict(grad_sampling_locations=torch.zeros(N, Lq, M, L, K, 1))),
        (TypeError, dict(grad_sampling_locations=torch.zeros(N, Lq, M, L, K, 2, dtype=bf16))),
        (ValueError, dict(grad_attention_weights=torch.zeros(N, Lq, M, L, K - 1))),
    ]
    for exc, over in bad:
        with pytest.raises(exc):
            call(**over)
    # a bf16 problem: grad_output must be bf16 too, the gradients stay float32
    assert call(value=torch.zeros(N, S, M, D, dtype=bf16), grad_output=torch.zeros(N, Lq, M * D, dtype=bf16)) \
        == (Lq, L, K)
    with pytest.raises(TypeError):
        call(value=torch.zeros(N, S, M, D, dtype=bf16))


def test_probe_library_exports_its_header(msda):
    """libmsda_probes.so (the line-rate measurements bench.py makes) exports
    exactly what include/msda_probes.h declares, and nothing of the method."""
    lib = os.path.join(os.path.dirname(msda.LIBRARY), "libmsda_probes.so")
    text = open(os.path.join(ROOT, "include", "msda_probes.h")).read()
    declared = set(re.findall(r"\b(msda_probe_\w+)\s*\(", text))
    out = subprocess.run(["nm", "-D", "--defined-only", lib], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(msda_\w+)", out))
    assert declared and exported == declared
    probes = ctypes.CDLL(lib)
    probes.msda_probe_accesses.argtypes = [ctypes.c_int64]
    probes.msda_probe_accesses.restype = ctypes.c_int64
    n = probes.msda_probe_accesses(22756352)
    assert 22756352 <= n < 22756352 * 1.02
    assert probes.msda_probe_accesses(0) == 0


def test_debug_library_exports(msda):
    """libmsda_debug.so exports what include/msda.h declares plus the one entry
    point of include/msda_debug.h."""
    from scale_deformable_attention_06_b300 import _capi
    out = subprocess.run(["nm", "-D", "--defined-only", _capi.DEBUG_LIBRARY], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT\s+(msda_\w+)", out))
    assert exported == set(declared_symbols()) | {"msda_debug_violations"}
