"""The benchmark's multi-rank harness on CPU (gloo, world size 2): replicas
only, max-over-ranks timing and the whole-job aggregate; the reference arm
runs on rank 0 only."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    bench.init_dist(world, "gloo")
    t = bench.max_over_ranks(10.0 * (rank + 1), world)
    n = bench.sum_over_ranks(1.0, world)
    bench.barrier(world)
    rate = bench.whole_job_rate(world * 1000.0, t / 1e3)
    q.put((rank, t, n, rate))
    torch.distributed.destroy_process_group()


def test_two_rank_gloo_harness():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, n, rate in res:
        assert t == 20.0 and n == 2.0
        assert rate == pytest.approx(2000.0 / 0.020)


def test_reference_arm_nonzero_rank_does_no_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_decode_bytes_accounting():
    """Algorithmic bytes: real-channel codes + fp16 scale/zero of full blocks,
    fp32 tail latents, fp16 q and out."""
    import bench
    from rank_latent_kv_gb300 import synth
    w = synth.WORKLOADS["qwen7b"]
    b = bench.decode_bytes(w, 32, 8, 32, 8, 64, out_bytes=2)
    per_stream = 2 * (2 * 32 * (8 * 4 + 24 * 2) / 8 + 2 * 32 * 4)   # K and V, 2 full blocks, no tail
    assert b == w.batch * w.hkv * per_stream + w.batch * w.hq * 128 * 4
    b1 = bench.decode_bytes(w, 32, 8, 32, 8, 65, out_bytes=2)
    assert b1 - b == w.batch * w.hkv * 2 * 32 * 4                    # one fp32 tail token per tensor
