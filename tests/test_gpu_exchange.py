"""The expert-parallel exchange on the GPU with NCCL, in a one-process group
(the run has one GPU): the whole layer goes through the exchange -- the CUDA
path's dispatch, the count and row all-to-alls, the expert on the received
rows, the reverse all-to-all into ``y``, the CUDA combine -- and the output is
compared with the oracle's. With one process every row stays local, so this
checks the exchange's bookkeeping on device tensors and NCCL's handling of the
views it sends; the multi-process row routing is covered by the gloo tests.
"""
from __future__ import annotations

import socket

import numpy as np
import pytest
import torch

import ep_synth
from gpu_harness import bf16_from_dev, bf16_to_dev, bf16_ulp_distance, require_cuda

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_exchange_nccl_one_process(orc, name):
    require_cuda()
    import torch.distributed as dist

    import combine_router_softmax_gb300 as ep
    from combine_router_softmax_gb300.exchange import EpExchange

    w = ep_synth.CONFIGS[name]
    logits = ep_synth.gate_logits(w.seed, w.T, w.E, w.zipf_s)
    x = ep_synth.hidden_bf16_bits(w.seed, w.T, w.H)
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1,
                            device_id=torch.device("cuda", 0))
    try:
        cfg = ep.EpConfig.from_workload(w)
        b = ep.LayerBuffers.allocate(cfg)
        b.logits.copy_(torch.from_numpy(logits))
        b.x.copy_(bf16_to_dev(x))
        b.dispatch_fused()
        ex = EpExchange(cfg)
        rec = ex.dispatch(b.send, b.expert_count, b.rank_offset)
        e = rec.expert_ids
        y_recv = (rec.rows.float() * ((e + 1).float() / w.E)[:, None]).to(torch.bfloat16)
        b.y.view(torch.int16).fill_(-1)
        ex.combine(y_recv, rec, b.y)
        b.combine()
        torch.cuda.synchronize()
        assert rec.send_splits == [w.T * w.k] and rec.recv_splits == [w.T * w.k]
        assert torch.equal(rec.counts.reshape(-1), b.expert_count)
    finally:
        dist.destroy_process_group()
    r = orc.run_path(logits, x, E=w.E, R=w.R, k=w.k, n_groups=w.n_groups, topk_groups=w.topk_groups,
                     renormalize=w.renormalize, ranks_per_node=w.ranks_per_node, self_rank=w.self_rank,
                     W=w.num_workers)
    assert np.array_equal(bf16_from_dev(b.y), r["y"]), "expert rows returned by the exchange differ"
    assert bf16_ulp_distance(bf16_from_dev(b.out), r["out"]).max() <= 1
