"""Full-size workloads through the same calls and launch configuration the
benchmark times (GPU).

route, layout and the chunk schedule are compared with the oracle on every
token (cheap on the CPU). The send buffer and the combine output are checked
on sampled tokens, which the oracle computes one by one: a token's combine
output depends only on its own x row, experts and weights, so the oracle
solves the sub-problem made of the sampled tokens alone (its own route,
layout, dispatch, expert and combine) and that equals its full-size answer
for those tokens. Properties that hold at any size (slot_meta is a
permutation, the send rows of a token equal its x row) are checked in full.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ep_synth
from gpu_harness import bf16_from_dev, bf16_to_dev, bf16_ulp_distance, require_cuda, synthetic_expert
from test_gpu_parity import assert_layout, assert_route

pytestmark = pytest.mark.gpu

FULL = [
    ep_synth.CONFIGS["prefill"],
    ep_synth.CONFIGS["mid"],
    ep_synth.get_workload("sweep-zipf-T4096"),
    ep_synth.get_workload("sweep-uniform-T32768"),
    ep_synth.get_workload("sweep-zipf-T32768"),
]


@pytest.fixture(scope="module")
def ep():
    require_cuda()
    import combine_router_softmax_gb300 as m

    return m


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_fullsize(ep, orc, w):
    logits = ep_synth.gate_logits(w.seed, w.T, w.E, w.zipf_s)
    x = ep_synth.hidden_bf16_bits(w.seed, w.T, w.H)

    cfg = ep.EpConfig.from_workload(w)
    b = ep.LayerBuffers.allocate(cfg)
    b.logits.copy_(torch.from_numpy(logits))
    b.x.copy_(bf16_to_dev(x))
    b.route()
    b.layout()
    b.dispatch()
    synthetic_expert(b.send, b.expert_offset, w.E, out=b.y)
    b.combine()
    torch.cuda.synchronize()
    check_against_oracle(orc, w, b, logits, x)


# The benchmark's own launch configuration: ep_dispatch_fused + ep_combine
# captured once in a CUDA graph and replayed. Small T runs the single fused
# kernel (with and without its schedule CTA), large T the route, layout and
# dispatch kernels chained by programmatic dependent launch.
GRAPH = [
    ep_synth.get_workload("sweep-uniform-T1"),
    ep_synth.get_workload("sweep-zipf-T8"),
    ep_synth.get_workload("sweep-uniform-T64"),
    ep_synth.CONFIGS["decode"],
    ep_synth.get_workload("sweep-zipf-T512"),
    ep_synth.CONFIGS["prefill"],
    ep_synth.CONFIGS["mid"],
    ep_synth.get_workload("sweep-zipf-T32768"),
]


def poison_outputs(b):
    """Every buffer the step writes gets a value no correct step leaves there."""
    for t in (b.topk_idx, b.expert_count, b.expert_offset, b.rank_count, b.rank_offset, b.slot, b.chunks,
              b.n_chunks, b.worker_begin, b.slot_meta):
        t.fill_(-7)
    b.topk_w.fill_(float("nan"))
    b.send.view(torch.int16).fill_(-1)  # 0xFFFF: a bf16 NaN
    b.out.view(torch.int16).fill_(-1)


@pytest.mark.parametrize("w", GRAPH, ids=lambda w: w.name)
def test_fullsize_bench_graph(ep, orc, w):
    import bench

    logits = ep_synth.gate_logits(w.seed, w.T, w.E, w.zipf_s)
    x = ep_synth.hidden_bf16_bits(w.seed, w.T, w.H)
    cfg = ep.EpConfig.from_workload(w)
    b = ep.LayerBuffers.allocate(cfg)
    b.logits.copy_(torch.from_numpy(logits))
    b.x.copy_(bf16_to_dev(x))
    dev = torch.device("cuda", torch.cuda.current_device())
    # expert output of this batch, as the benchmark makes it before timing
    b.bind(torch.cuda.current_stream(dev)).dispatch_fused()
    synthetic_expert(b.send, b.expert_offset, w.E, out=b.y)
    torch.cuda.synchronize()

    g = bench.capture_step_graph(b, dev, fused=True)
    for _ in range(2):  # the second replay starts from what the first left in the workspace
        poison_outputs(b)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
    assert ep.ep_device_error() == 0
    check_against_oracle(orc, w, b, logits, x)


def check_against_oracle(orc, w, b, logits, x):
    # route + layout + schedule: every token
    idx, w64 = orc.route(logits, w.k, w.n_groups, w.topk_groups, w.renormalize)
    lay = orc.layout(idx, w.E, w.R)
    ch, wb = orc.schedule(lay["rank_offset"], w.ranks_per_node, w.self_rank, w.num_workers)
    n = int(b.n_chunks.item())
    g = dict(idx=b.topk_idx.cpu().numpy(), w=b.topk_w.cpu().numpy(),
             expert_count=b.expert_count.cpu().numpy(), expert_offset=b.expert_offset.cpu().numpy(),
             rank_count=b.rank_count.cpu().numpy(), rank_offset=b.rank_offset.cpu().numpy(),
             slot=b.slot.cpu().numpy(), chunks=b.chunks[:n].cpu().numpy(), worker_begin=b.worker_begin.cpu().numpy())
    assert_route(g, dict(idx=idx, w=w64), logits, w.renormalize)
    assert_layout(g, dict(chunks=ch, worker_begin=wb, **lay))

    # slot_meta is a permutation of 0 .. T k - 1 and agrees with slot
    meta = b.slot_meta
    assert torch.equal(torch.sort(meta).values, torch.arange(w.T * w.k, device="cuda", dtype=torch.int32))
    slot_flat = b.slot.view(-1).long()
    assert torch.equal(meta[slot_flat], torch.arange(w.T * w.k, device="cuda", dtype=torch.int32))

    # sampled tokens: send rows and combine output
    rng = np.random.default_rng(w.T)
    S = np.unique(np.concatenate([[0, 1, w.T // 2, w.T - 1], rng.integers(0, w.T, size=96)]))
    S = S[S < w.T]
    send_rows = bf16_from_dev(b.send[torch.from_numpy(lay["slot"][S].ravel()).long().cuda()])
    assert np.array_equal(send_rows, np.repeat(x[S], w.k, axis=0)), "send rows differ from x"

    sub = orc.run_path(logits[S], x[S], E=w.E, R=1, k=w.k, n_groups=w.n_groups, topk_groups=w.topk_groups,
                       renormalize=w.renormalize, ranks_per_node=1, self_rank=0, W=1)
    out_g = bf16_from_dev(b.out[torch.from_numpy(S).long().cuda()])
    d = bf16_ulp_distance(out_g, sub["out"])
    assert d.max() <= 1, f"combine differs by {d.max()} bf16 ulp on sampled tokens"
