"""bench.py's multi-rank host logic on CPU: two gloo ranks agree on the
slowest rank's time, and the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 10.0 + 5.0 * rank
    got = bench.max_over_ranks(local_ms, "cpu")
    bench.barrier()
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
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


def test_single_process_max_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5


def test_reference_arm_skips_non_zero_ranks(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_step_bytes():
    import bench
    # forward 4*R*D*2 + D*2 and VJP 3*R*D*2 + D*2 + 4*D at R = 16384
    assert bench.fwd_bytes(16384, 4096) == 536879104
    assert bench.vjp_bytes(16384, 4096) == 402677760
    assert bench.fwd_bytes(16384, 8192) == 1073758208
    assert bench.vjp_bytes(16384, 8192) == 805355520
    assert bench.STEP_BYTES == 536879104 + 402677760 + 1073758208 + 805355520


def test_reference_arm_json_line(monkeypatch, capsys):
    """Rank 0 of the reference arm prints one JSON line with the contract's keys.  The timed
    oracle pass is stubbed (the oracle itself is checked by the pin tests); the sample sizing,
    timing and line assembly run as they are."""
    import json
    import bench
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.setattr(bench, "oracle_pass", lambda sample, threads=1, pool=None: (10 ** 6, {}))
    assert bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3
    assert line["unit"] == bench.UNIT and line["metric"] == bench.METRIC
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["cores"] == bench.host_cores() == line["cpu_baseline"]["host_cores"]
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": bench.UNIT, "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["value"] > 0


def test_all_core_oracle_pass_matches_one_thread():
    """The CPU baseline's all-core pass splits rows into contiguous blocks and
    adds the blocks' gw in block order: the same gw as one thread up to fp64
    reassociation, and the same bytes."""
    import concurrent.futures as cf
    import numpy as np
    import oracle
    import bench
    from rmsnorm_fwd_bwd_add_gb300 import workloads as W
    oracle.build()
    cases = {D: W.config4(D, 37) for D in bench.DS}
    sample = bench.oracle_sample(cases, 37)
    b1, gw1 = bench.oracle_pass(sample)
    with cf.ThreadPoolExecutor(max_workers=4) as pool:
        b4, gw4 = bench.oracle_pass(sample, 4, pool)
    assert b1 == b4 == sum(bench.fwd_bytes(37, D) + bench.vjp_bytes(37, D) for D in bench.DS)
    for D in bench.DS:
        np.testing.assert_allclose(gw4[D], gw1[D], rtol=1e-12, atol=1e-12)
        # and gw is the oracle's own VJP of the whole sample
        s = sample[D]
        _, h = oracle.fwd(s["x"], s["w"], s["eps"], 0.0, s["res"])
        np.testing.assert_array_equal(gw1[D], oracle.vjp(h, s["w"], s["g"], s["eps"], 0.0)[1])
