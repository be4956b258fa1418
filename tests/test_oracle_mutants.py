"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them (CPU only; the planted bugs never leave a temp dir)."""
import json
import os
import subprocess
import sys
import tempfile

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "msda_oracle.c")

# (name, text to find, replacement): each is a mistake someone could make
MUTANTS = [
    ("half_pixel_sign", "lx * (double)(W - 1) : lx * (double)W - 0.5;", "lx * (double)(W - 1) : lx * (double)W + 0.5;"),
    ("align_corners_true", "lx * (double)(W - 1) : lx * (double)W - 0.5;", "lx * (double)(W - 1) : lx * (double)(W - 1);"),
    ("align_corners_ignored", "int align = (options & OPT_ALIGN_CORNERS) != 0;", "int align = 0;"),
    ("align_corners_uses_W", "lx * (double)(W - 1) : lx", "lx * (double)W : lx"),
    ("align_grad_uses_W", "(double)(align ? W - 1 : W)", "(double)W"),
    ("per_level_softmax_over_row", "return msda_oracle_softmax(rows * n_levels, n_points, logits, weights);",
     "return msda_oracle_softmax(rows, n_levels * n_points, logits, weights);"),
    ("per_level_softmax_grad_over_row", "? n_points : cols;", "? cols : cols;"),
    ("swapped_x_weights", "(i ? fx : 1.0 - fx)", "(i ? 1.0 - fx : fx)"),
    ("x_uses_fy", "(i ? fx : 1.0 - fx) * (j ? fy : 1.0 - fy)", "(i ? fy : 1.0 - fy) * (j ? fy : 1.0 - fy)"),
    ("bounds_off_by_one", "xc < W && yc >= 0", "xc <= W && yc >= 0"),
    ("transposed_rows", "start + yc * W + xc", "start + xc * H + yc"),
    ("level_start_ignored", "start + yc * W + xc", "yc * W + xc"),
    ("dropped_corner", "for (int ci = 0; ci < 4; ++ci) {\n        if (c->row[ci] < 0) continue;",
     "for (int ci = 0; ci < 3; ++ci) {\n        if (c->row[ci] < 0) continue;"),
    ("softmax_not_normalised", "for (int64_t j = 0; j < cols; ++j) y[j] /= sum;", ""),
    ("softmax_not_shifted", "y[j] = exp(x[j] - mx);", "y[j] = exp(x[j]);"),
    ("offset_x_scaled_by_H", "sampling_offsets[i + 0] / W;", "sampling_offsets[i + 0] / H;"),
    ("fused_offset_x_scaled_by_H", "double lx = rx + ox / (double)W;", "double lx = rx + ox / (double)H;"),
    ("grad_loc_missing_scale", "attn[s] * gx * (double)(align ? W - 1 : W)", "attn[s] * gx"),
    ("grad_loc_wrong_sign", "(1.0 - c.fy) * (v[D + d] - v[d])", "(1.0 - c.fy) * (v[d] - v[D + d])"),
    ("grad_loc_y_uses_fy", "(1.0 - c.fx) * (v[2 * D + d] - v[d]) + c.fx",
     "(1.0 - c.fy) * (v[2 * D + d] - v[d]) + c.fy"),
    ("grad_value_missing_attn", "gv[d] += attn[s] * c.w[ci] * g[d];", "gv[d] += c.w[ci] * g[d];"),
    ("grad_attn_of_first_corner", "ga += g[d] * smp;", "ga += g[d] * v[d];"),
    ("fused_grad_offset_scaled_wrong", "gloc[2 * s + 0] / W;", "gloc[2 * s + 0] * W;"),
    ("softmax_grad_missing_dot", "(gattn[r * cols + j] - dot)", "(gattn[r * cols + j])"),
    ("grad_ref_not_summed", "gref[0] += gloc[2 * s + 0];", "gref[0] = gloc[2 * s + 0];"),
    ("trilinear_drops_z_weight", "* (k ? c->f[2] : 1.0 - c->f[2]);", ";"),
    ("trilinear_z_stride", "start + (zc * H + yc) * W + xc", "start + (zc * W + yc) * W + xc"),
    ("trilinear_z_bound", "zc >= 0 && zc < Dd)", "zc >= 0 && zc <= Dd)"),
    ("trilinear_grad_z_scale", "(double)(align ? sh[0] - 1 : sh[0])};", "(double)(align ? sh[1] - 1 : sh[1])};"),
    ("trilinear_grad_sign", "double dw = bit[a] ? 1.0 : -1.0;", "double dw = bit[a] ? -1.0 : 1.0;"),
    ("group_index_interleaved", "int64_t gm = m / hpg;", "int64_t gm = m % n_groups;"),
    ("grouped_grad_attn_not_summed", "gr->grad_attn[s] += ga;", "gr->grad_attn[s] = ga;"),
    ("grouped_grad_loc_not_summed", "gr->grad_loc[2 * s + 0] += attn[s] * gx", "gr->grad_loc[2 * s + 0] = attn[s] * gx"),
]


def _build_mutant(tmp, find, repl):
    src = open(SRC).read()
    assert src.count(find) >= 1, f"mutation anchor not found: {find!r}"
    mutated = src.replace(find, repl, 1)
    c_path = os.path.join(tmp, "mutant.c")
    so_path = os.path.join(tmp, "mutant.so")
    with open(c_path, "w") as f:
        f.write(mutated)
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-w",
                    "-o", so_path, c_path, "-lm"], check=True)
    return so_path


_RUNNER = """
import json, sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
oracle.use_library(oracle.bind({so!r}))
print(json.dumps({{k: bool(v[0]) for k, v in oracle_pins.run_all().items()}}))
"""


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, find, repl):
    """A mutant runs in its own process: one that corrupts memory and crashes
    has been caught as surely as one that fails a pin."""
    here = os.path.dirname(os.path.abspath(__file__))
    with tempfile.TemporaryDirectory() as tmp:
        so = _build_mutant(tmp, find, repl)
        code = _RUNNER.format(root=os.path.dirname(here), tests=here, so=so)
        proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if proc.returncode != 0:
        return
    res = json.loads(proc.stdout.strip().splitlines()[-1])
    failed = [k for k, ok in res.items() if not ok]
    assert failed, f"mutant {name} passed every pin"
