"""The multi-GPU (N > 1) path of the benchmark, on CPU with the gloo backend.

The path is data-parallel: each rank routes, lays out, dispatches and combines
its own batch and nothing crosses ranks except the benchmark's barrier and the
max-over-ranks of the timed region. Two ranks check that (a) their shards
differ, (b) routing the two shards together equals routing each shard alone
(tokens are independent, so sharding changes no result), and (c) the timing
reduction returns the slowest rank's time on every rank. The benchmark's own
reduction of a workload's timed totals (reduce_max_many, then whole_job) runs
on two and four ranks with different totals per rank, as its GPU arm calls it.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist

    import bench
    import ep_synth
    import oracle

    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = bench.rank_workload(ep_synth.CONFIGS["tiny"], rank)
    logits = ep_synth.gate_logits(w.seed, w.T, w.E, w.zipf_s)
    x = ep_synth.hidden_bf16_bits(w.seed, w.T, w.H)
    r = oracle.get().run_path(logits, x, E=w.E, R=w.R, k=w.k, W=8)

    # gather every rank's logits and routing
    all_logits = [torch.zeros_like(torch.from_numpy(logits)) for _ in range(world)]
    dist.all_gather(all_logits, torch.from_numpy(logits))
    all_idx = [torch.zeros((w.T, w.k), dtype=torch.int32) for _ in range(world)]
    dist.all_gather(all_idx, torch.from_numpy(r["idx"]))
    slowest = bench.reduce_max(float(rank + 1) * 1.5, world)
    bench.barrier(world)
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), slowest=slowest, seed=w.seed,
             logits=torch.stack(all_logits).numpy(), idx=torch.stack(all_idx).numpy(), out=r["out"])
    dist.destroy_process_group()


def test_two_rank_shards_gloo(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    import oracle

    res = [np.load(tmp_path / f"rank{r}.npz") for r in range(world)]
    assert all(float(r["slowest"]) == 3.0 for r in res)  # max over ranks, seen by every rank
    assert int(res[0]["seed"]) != int(res[1]["seed"])
    logits = res[0]["logits"]
    assert not np.array_equal(logits[0], logits[1]), "ranks must hold different batches"
    assert not np.array_equal(res[0]["out"], res[1]["out"])
    # routing the concatenated batch equals routing each shard alone
    both = np.concatenate([logits[0], logits[1]])
    idx_all, _ = oracle.get().route(both, 2)
    assert np.array_equal(idx_all, np.concatenate([res[0]["idx"][0], res[0]["idx"][1]]))


def _reduce_worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r: graph total 10 + r ms, stream total 30 - r ms, e2e 50 + 2 r, pipelined 40 - 3 r
    local = {"step": 10.0 + rank, "stream": 30.0 - rank, "e2e": 50.0 + 2 * rank, "pipe": 40.0 - 3 * rank}
    tot = bench.reduce_max_many(local, world)
    value, ms = bench.whole_job(1_000_000_000, world, 20, tot["step"])
    lat = bench.reduce_max_many({"median": 5.0 + 0.5 * rank, "mean": 7.0 - rank}, world)
    np.savez(os.path.join(out_dir, f"red{rank}.npz"), step=tot["step"], stream=tot["stream"], e2e=tot["e2e"],
             pipe=tot["pipe"], value=value, ms=ms, lat_median=lat["median"], lat_mean=lat["mean"])
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_bench_rank_reduction_gloo(tmp_path, world):
    mp.start_processes(_reduce_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    for r in range(world):
        res = np.load(tmp_path / f"red{r}.npz")
        assert float(res["step"]) == 10.0 + (world - 1)
        assert float(res["stream"]) == 30.0
        assert float(res["e2e"]) == 50.0 + 2 * (world - 1)
        assert float(res["pipe"]) == 40.0
        # every rank moved 1 GB per step, 20 steps, the slowest in 10 + world - 1 ms
        ms = (10.0 + world - 1) / 20
        assert float(res["ms"]) == pytest.approx(ms)
        assert float(res["value"]) == pytest.approx(world * 1.0 / (ms * 1e-3))
        assert float(res["lat_median"]) == 5.0 + 0.5 * (world - 1)
        assert float(res["lat_mean"]) == 7.0
