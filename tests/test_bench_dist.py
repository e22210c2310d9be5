"""Host logic of bench.py's multi-rank (replica) path on CPU with gloo, and
the algorithmic-bytes model (no GPU)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    w, r, _ = bench.dist_env()
    active = bench.init_dist(w, "gloo")
    bench.barrier(active)
    got = bench.max_over_ranks(10.0 + 5.0 * r, active)
    q.put((r, got))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 15.0, 1: 15.0}


def test_single_rank_is_passthrough():
    assert bench.max_over_ranks(3.5, False) == 3.5


def test_b_alg_model():
    # N = 10: L = 4 levels, 3 sort levels
    assert bench.b_alg(10) == 10 * (20 * 3 + 12)
    assert bench.b_alg(100_000_000) == pytest.approx(53.2e9, rel=1e-3)
    assert bench.b_alg(1) == 12.0


def test_recorded_traffic_tracks_kernel_source(tmp_path, monkeypatch):
    import shutil
    # the table in profiles/ matches the committed sources
    for kern in ("finisher", "part"):
        v = bench.recorded_traffic(kern)
        assert v is None or v > 0
    assert bench.recorded_traffic("no_such_kernel") is None
    # a changed kernel source invalidates the recorded figure
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    shutil.copy(os.path.join(bench.ROOT, "profiles", "traffic_uniform_100m.txt"), root / "profiles")
    src = root / "balanced_tree_build_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "kdt_finisher_sorted.cu").write_text("// changed\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.recorded_traffic("finisher") is None


def test_reference_arm_json_line(capsys):
    # the reference arm (the oracle on the host cores) prints the contract's
    # one JSON line, on the bench workload's config, without a GPU
    import json
    rc = bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0", "--ref-sample", "4096"])
    assert rc == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "uniform_100m" and line["config"]["reference_sample_points"] == 4096
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_clock_samples_kept_inside_the_timed_region():
    # nvidia-smi lines: timestamp, sm, max sm, power, active mask, 4 reasons
    import datetime
    base = datetime.datetime(2026, 12, 2, 18, 0, 0)

    def line(ms, sm, reason=("Not Active",) * 4):
        ts = (base + datetime.timedelta(milliseconds=ms)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return ", ".join([ts, str(sm), "2070", "900.0", "0x0"] + list(reason))

    t0 = base.timestamp()
    lines = [line(0, 1200), line(500, 2070), line(520, 2070), line(540, 2070, ("Not Active", "Not Active",
             "Not Active", "Active")), line(900, 1500)]
    got = bench.ClockSampler.summarise(lines, (t0 + 0.49, t0 + 0.55))
    assert got["samples"] == 3 and got["window"] == "timed region"
    assert got["sm_mhz"] == 2070.0 and got["sm_max_mhz"] == 2070.0 and got["reasons"] == ["sw_power_cap"]
    # nothing inside: the two samples nearest to the window
    near = bench.ClockSampler.summarise(lines, (t0 + 0.7, t0 + 0.72))
    assert near["samples"] == 2 and near["window"] == "nearest to the timed region"
    # malformed lines are skipped; no usable line gives None
    assert bench.ClockSampler.summarise(["garbage", ""], None) is None
