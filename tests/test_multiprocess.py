"""The N > 1 host path of bench.py on CPU: two gloo ranks on 127.0.0.1.

Each rank holds its own step times; the whole job's time is the slowest
rank's (max over ranks), which every rank must receive.  The reference arm
runs on rank 0 only; other ranks return without work.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [1e-3 * (rank + 1), 2e-3 * (world - rank)]
    got = bench.max_over_ranks(mine, "cpu")
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    want = [1e-3 * world, 2e-3 * world]
    for r in range(world):
        assert out[r] == pytest.approx(want)


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"steps": 1, "warmup": 0, "gpus": 2})()
    bench.run_reference(args)
    assert capsys.readouterr().out == ""


def test_reference_arm_json_line():
    # the reference arm (the oracle on one host core) prints one JSON line
    # with the contract's keys; no GPU is touched
    import json
    import subprocess
    import sys
    from conftest import ROOT
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["config"]["workload"] == "qwen3-8b-layer-decode-100k"
    # ms_per_step is what a timed step measured; the whole-step figure the
    # value comes from is carried apart
    ex = line["extrapolation"]
    assert ex["measured_ms_per_sample_step"] == line["ms_per_step"]
    assert abs(ex["whole_step_ms"] - ex["factor"] * line["ms_per_step"]) <= 1e-6 * ex["whole_step_ms"]
    assert abs(line["value"] - 1e3 / ex["whole_step_ms"]) <= 1e-9 * line["value"]
    assert line["cpu_baseline"]["host_logical_cores"] >= 1 and line["cpu_baseline"]["host_cpu"]


def test_decode_bytes_match_the_oracle_accounting():
    # the roofline's algorithmic bytes per decode launch: INT2 history at the
    # oracle's per-token storage cost (codes + (scale, zero) per group), BF16
    # sink and recent K/V, page-table entries, q in and the fp32 output
    import bench
    import oracle as O
    w = bench.WORKLOAD
    keep = (w["group_k"], w["group_v"])
    try:
        for gk, gv in ((128, 128), (64, 64), (32, 128), (32, 32)):
            w["group_k"], w["group_v"] = gk, gv
            s, h, r = bench._split(w["ctx"])
            want = (h * O.kv_bytes_per_history_token(w["n_kv_heads"], group_k=gk, group_v=gv)
                    + (s + r) * w["n_kv_heads"] * 2 * 128 * 2 + -(-h // 16) * 4
                    + w["n_q_heads"] * 128 * (2 + 4))
            assert bench.bytes_per_decode() == want
            assert bench._hist_bytes_per_token(w["n_kv_heads"]) == O.kv_bytes_per_history_token(
                w["n_kv_heads"], group_k=gk, group_v=gv)
    finally:
        w["group_k"], w["group_v"] = keep
    assert bench.bytes_per_decode() == 58_775_896
