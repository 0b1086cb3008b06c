"""The bench's multi-process harness on CPU (gloo, world size 2): replicas
time independently and the reported time is the max over ranks."""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.rank_info()
    assert (r, w, lr) == (rank, world, rank)
    bench.barrier(w)
    out[rank] = bench.reduce_max(10.0 + 5.0 * rank, w)
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs)
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_process_reduce_is_identity():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5


def test_step_bytes_of_the_bench_workload():
    import numpy as np
    import bench
    import synth
    cfg = synth.QWEN3_8B_B1
    sb = bench.step_bytes(cfg, np.array([4096]), 5)
    # weights: eh 4096*8192, q 4096*4096, k/v 1024*4096 each, o 4096*4096,
    # gate/up/down 3*12288*4096, embedding/LM head 151936*4096, 5 norms of 4096
    w = (4096 * 8192 + 4096 * 4096 + 2 * 1024 * 4096 + 4096 * 4096 + 3 * 12288 * 4096 + 151936 * 4096
         + 5 * 4096) * 2
    assert sb["weights"] == w
    assert abs(sb["draft"] / 5 / 1e6 - 1715.09) < 0.5


def _reference_line(argv, capsys):
    import json
    import bench
    bench.main(argv)
    out = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(out) == 1
    return json.loads(out[0])


def test_reference_arm_follows_the_workload(capsys, monkeypatch):
    """The reference arm reports the metric, unit and config of the arm it
    stands beside: draft steps/s, loop tok/s (chain and tree)."""
    import bench
    monkeypatch.setenv("MTP_REFERENCE_BUDGET_S", "2")
    d = _reference_line(["--impl", "reference", "--workload", "tiny_f32_h256", "--steps", "1", "--warmup", "3"],
                        capsys)
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "steps/s"
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    d = _reference_line(["--impl", "reference", "--workload", "tiny_f32_h256", "--loop", "--steps", "2",
                         "--warmup", "3"], capsys)
    assert d["metric"] == bench.LOOP_METRIC and d["unit"] == "tok/s"
    assert d["config"]["workload"] == "spec_loop_tiny_f32_h256" and d["config"]["tree"] is None
    assert d["value"] > 0 and d["config"]["mean_emitted_per_step"] >= 1.0
    d = _reference_line(["--impl", "reference", "--workload", "tiny_f32_h256", "--loop", "--tree", "2,3,4",
                         "--steps", "1", "--warmup", "3"], capsys)
    assert d["config"]["tree"] == {"branching_factor": 2, "tree_depth": 3, "num_assistant_tokens": 4}
    assert d["value"] > 0
