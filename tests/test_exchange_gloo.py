"""The expert-parallel exchange (combine_router_softmax_gb300.exchange) on CPU
processes with the gloo backend: 2 and 4 processes, each the expert-parallel
home of E / P experts.

Every process holds its own seeded batch. The oracle's path on that batch
stands in for the GPU's outputs (send buffer, counts, offsets, slots), so the
test needs no GPU; every process can recompute any other process's oracle path
from the seeds. Checked on every process:

* the dispatch exchange delivers, from each source s, exactly the oracle's
  send rows of s for this process's virtual ranks, in order, and the counts of
  this process's experts in them;
* the synthetic expert applied to the received rows (the oracle's expert
  function, per source segment) and sent back by the reverse exchange fills
  ``y`` with exactly the oracle's expert rows of this process's own batch;
* the oracle's combine of that ``y`` equals the oracle's output of the
  single-process path: the exchange changes no result.
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


def _source_path(orc, w0, s):
    import bench
    import ep_synth

    w = bench.rank_workload(w0, s)
    logits = ep_synth.gate_logits(w.seed, w.T, w.E, w.zipf_s)
    x = ep_synth.hidden_bf16_bits(w.seed, w.T, w.H)
    r = orc.run_path(logits, x, E=w.E, R=w.R, k=w.k, n_groups=w.n_groups, topk_groups=w.topk_groups,
                     renormalize=w.renormalize, ranks_per_node=w.ranks_per_node, self_rank=w.self_rank,
                     W=w.num_workers)
    return w, r


def _worker(rank, world, port, out_dir, w0):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist

    import oracle
    from combine_router_softmax_gb300 import EpConfig
    from combine_router_softmax_gb300.exchange import EpExchange

    dist.init_process_group("gloo", rank=rank, world_size=world)
    orc = oracle.get()
    w, mine = _source_path(orc, w0, rank)
    ex = EpExchange(EpConfig.from_workload(w))
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)  # noqa: E731
    rec = ex.dispatch(bf(mine["send"]), torch.from_numpy(mine["expert_count"]),
                      torch.from_numpy(mine["rank_offset"]))
    got = rec.rows.view(torch.int16).numpy().view(np.uint16)

    # (1) rows and counts from every source, against that source's oracle path
    Ep = w.E // world
    e0, e1 = rank * Ep, (rank + 1) * Ep
    r0, r1 = rank * (w.R // world), (rank + 1) * (w.R // world)
    at = 0
    ok_rows = ok_counts = True
    segments = []
    for s in range(world):
        _, src = _source_path(orc, w0, s)
        seg = src["send"][src["rank_offset"][r0]:src["rank_offset"][r1]]
        ok_rows &= np.array_equal(got[at:at + len(seg)], seg)
        ok_counts &= np.array_equal(rec.counts[s].numpy(), src["expert_count"][e0:e1])
        segments.append((at, len(seg)))
        at += len(seg)
    ok_rows &= at == got.shape[0]
    ids = rec.expert_ids.numpy()
    ok_ids = bool(((ids >= e0) & (ids < e1)).all()) and len(ids) == got.shape[0]

    # (2) the expert on the received rows, per source segment (rows ordered by expert)
    y_recv = np.empty_like(got)
    for s, (a, n) in enumerate(segments):
        off = np.zeros(w.E + 1, np.int32)
        off[e0 + 1:e1 + 1] = np.cumsum(rec.counts[s].numpy())
        off[e1 + 1:] = off[e1]
        y_recv[a:a + n] = orc.expert(got[a:a + n], off, w.E)
        ok_ids &= bool((ids[a:a + n] == np.repeat(np.arange(e0, e1), rec.counts[s].numpy())).all())
    y = torch.empty_like(bf(mine["send"]))
    ex.combine(bf(y_recv), rec, y)
    y_bits = y.view(torch.int16).numpy().view(np.uint16)
    ok_y = np.array_equal(y_bits, mine["y"])

    # (3) combine of the returned rows = the single-process output
    out = orc.combine(y_bits, mine["slot"], mine["w32"])
    ok_out = np.array_equal(out, mine["out"])
    np.savez(os.path.join(out_dir, f"x{rank}.npz"), rows=ok_rows, counts=ok_counts, ids=ok_ids, y=ok_y, out=ok_out,
             n_recv=got.shape[0], splits=np.array(rec.send_splits))
    dist.destroy_process_group()


def _shape(name, world):
    import ep_synth

    if name == "tiny":
        return ep_synth.CONFIGS["tiny"].with_(num_workers=8, ranks_per_node=2)
    # decode-like: E = 64 over R = 8 virtual ranks, top-8, Zipf-skewed popularity
    return ep_synth.Workload("small-decode", T=96, H=128, E=64, R=8, k=8, zipf_s=1.2, num_workers=16,
                             ranks_per_node=4)


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("name", ["tiny", "small-decode"])
def test_exchange_gloo(tmp_path, world, name):
    w0 = _shape(name, world)
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path), w0), nprocs=world, start_method="spawn")
    total_recv = 0
    for r in range(world):
        res = np.load(tmp_path / f"x{r}.npz")
        for key in ("rows", "counts", "ids", "y", "out"):
            assert bool(res[key]), f"process {r}: {key} differs"
        assert int(res["splits"].sum()) == w0.T * w0.k
        total_recv += int(res["n_recv"])
    assert total_recv == world * w0.T * w0.k  # every row of every process went to exactly one process


def test_exchange_rejects_uneven_split():
    from combine_router_softmax_gb300 import EpConfig
    from combine_router_softmax_gb300.exchange import EpExchange

    cfg = EpConfig.make(T=4, H=8, E=6, R=3, k=2, num_workers=2)
    ex = EpExchange(cfg, world=3, rank=1)
    assert ex.experts_per_proc == 2 and ex.ranks_per_proc == 1
    with pytest.raises(ValueError):  # 3 virtual ranks cannot be split over 2 processes
        EpExchange(cfg, world=2, rank=0)
