"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each with its own
batch (weak scaling), the step time is the maximum over ranks and the value
counts the points of every rank.  No GPU and no data-path collective."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    r, lr, ws = bench.dist_env()
    t = 1.0 + rank                      # rank 1 is the slow one
    tmax = bench.max_over_ranks(t, dist)
    seed = bench.rank_seed(1235, r)
    q.put((r, ws, tmax, seed, bench.aggregate(100, ws, tmax)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ws0, t0, s0, v0), (r1, ws1, t1, s1, v1) = res
    assert (r0, r1) == (0, 1) and ws0 == ws1 == 2
    assert t0 == t1 == 2.0                # the slowest rank sets the time
    assert s0 != s1                       # independent batches per rank
    assert v0 == v1 == pytest.approx(100 * 2 / 2.0)


def test_single_rank_defaults(monkeypatch):
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 0, 1)
    assert bench.max_over_ranks(3.5) == 3.5


def test_algorithmic_bytes_of_the_encoder_step():
    import workloads
    ab = bench.algorithmic_bytes(workloads.WORKLOADS["encoder_train"])
    # value 45.5 MB, locations 45.5 MB, weights 22.8 MB, output 45.5 MB
    assert ab["fwd"] == pytest.approx(159.3e6, rel=2e-3)
    assert ab["bwd"] == pytest.approx(273.1e6, rel=2e-3)


def test_roofline_follows_the_steps_own_kernels():
    """The roofline names the kernels of the step that was timed, with bytes of
    the same calls, and takes DRAM counts only on the workload they were
    captured on."""
    import workloads
    ms = {"fwd": 0.14, "bwd": 0.38, "fused_fwd": 0.15, "fused_bwd": 0.43}
    ab = bench.algorithmic_bytes(workloads.WORKLOADS["encoder_train"])
    for step, names in (("forward + backward", ("msda_forward_kernel", "msda_backward_kernel")),
                        ("fused", ("msda_forward_kernel_fused", "msda_backward_kernel_fused"))):
        kern = bench.step_kernels(step, ms)
        assert (kern["fwd"][0], kern["bwd"][0]) == names
        for call, (name, t, key) in kern.items():
            assert key in ab and t == ms[key]
    assert bench.step_kernels("fused", ms)["bwd"][2] == "fused_bwd"
    assert ab["fused_bwd"] > ab["bwd"]          # the fused backward also reads the reference points
    for name in ("msda_backward_kernel", "msda_backward_kernel_fused"):
        assert bench.roofline_traffic(name, "large") is None
        assert bench.roofline_traffic(name, bench.WORKLOAD) == bench.profiled_traffic(name)


def test_touched_value_bytes():
    """Byte accounting of sparse queries: whole 32-byte sectors of the rows
    the in-map corners reach, each counted once."""
    import numpy as np
    import workloads
    # 4 x 4 map, two heads of 16-byte bf16 rows (two rows per sector)
    w = workloads.custom(N=1, M=2, D=8, levels=[(4, 4)], K=1, Len_q=1, dtype="bf16")
    loc = np.array([0.5, 0.5, 0.1, 0.1], np.float32).reshape(1, 1, 2, 1, 1, 2)
    # head 0: px = py = 1.5, pixels 5, 6, 9, 10 -> rows 10, 12, 18, 20 -> sectors 5, 6, 9, 10;
    # head 1: px = py = -0.1, only pixel 0 inside -> row 1 -> sector 0
    assert bench.touched_value_bytes(w, loc) == 5 * 32
    # fp32 rows of 128 bytes: every query samples the centre of pixel (3, 2), so
    # px = 3, py = 2 exactly; its four corners (3..4, 2..3) are all in the map
    # (two with weight 0, loaded all the same): 4 rows per (batch, head)
    w = workloads.custom(N=2, M=3, D=32, levels=[(5, 7)], K=2, Len_q=4)
    loc = np.full((2, 4, 3, 1, 2, 2), 0.0, np.float32)
    loc[..., 0], loc[..., 1] = 3.5 / 7, 2.5 / 5
    assert bench.touched_value_bytes(w, loc) == 2 * 3 * 4 * 128


def test_reference_arm_line():
    """`bench.py --impl reference` runs the oracle on the host (no GPU) and
    prints the contract's line: the same metric and config as our arm, the
    oracle as its cpu_baseline, an e2e with no copies."""
    import json
    import subprocess
    import sys
    import types
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=bench.ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([x for x in r.stdout.splitlines() if x.startswith("{")][-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    args = types.SimpleNamespace(workload=bench.WORKLOAD, step="unfused")
    expect = bench.workload_config(args, bench.workloads.WORKLOADS[bench.WORKLOAD], 1)
    assert {k: line["config"][k] for k in expect} == expect


@pytest.mark.parametrize("name", ["tiny", "encoder"])
def test_location_inputs_of_both_kinds_of_draw(name):
    """The bench's input preparation: drawn references and offsets give
    ref + off / (W, H); directly drawn locations (tiny) give a reference and
    pixel offsets that rebuild them."""
    import numpy as np
    import torch
    import workloads
    w = workloads.WORKLOADS[name]
    raw = workloads.draw(w)
    sh = torch.from_numpy(raw["spatial_shapes"])
    loc, ref, off = bench.location_inputs(raw, sh)
    assert loc.dtype == torch.float32 and tuple(loc.shape) == (w.N, w.Lq, w.M, w.L, w.K, 2)
    assert tuple(ref.shape) == (w.N, w.Lq, w.L, 2) and tuple(off.shape) == tuple(loc.shape)
    wh = sh[:, [1, 0]].double()
    rebuilt = ref.double()[:, :, None, :, None, :] + off.double() / wh[None, None, None, :, None, :]
    assert np.allclose(rebuilt.numpy(), loc.double().numpy(), rtol=0, atol=1e-6)
    if "sampling_locations" in raw:
        assert np.array_equal(loc.numpy(), raw["sampling_locations"])


def test_oracle_on_all_cores_line(capsys):
    """bench.py --cpu-all-cores: the oracle over every host core, one JSON line."""
    import json
    bench.main(["--cpu-all-cores", "--workload", "tiny"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])["cpu_baseline_all_cores"]
    assert line["kind"] == "oracle" and line["cores"] >= 1 and line["value"] > 0 and line["unit"] == bench.UNIT
