"""Full-size workloads through the same calls and launch configuration the
benchmark times (GPU), compared with the oracle element by element.

* route, layout and the chunk schedule: every token (cheap on the CPU).
* dispatch: every element of the send buffer and every slot_meta entry
  against orc_dispatch. The dispatch copies whole rows, so restricting x to a
  block of columns restricts the send buffer to the same columns; the oracle
  dispatches blocks of COLS columns at a time, which bounds host memory at
  T = 32768 (3.8 GB of send rows), and each block of the GPU's send buffer is
  compared with its block.
* combine: every element of ``out`` within 1 bf16 ulp of orc_combine. A
  token's output depends only on its own logits and x row (its experts,
  weights and expert rows), so the oracle's whole path run on a chunk of
  CHUNK consecutive tokens gives the full-size answer for those tokens; the
  chunks cover every token.
"""
from __future__ import annotations

import concurrent.futures as cf

import numpy as np
import pytest
import torch

import ep_synth
from gpu_harness import bf16_from_dev, bf16_to_dev, bf16_ulp_distance, require_cuda, synthetic_expert
from test_gpu_parity import assert_layout, assert_route

pytestmark = pytest.mark.gpu

COLS = 1024     # columns of x per oracle dispatch block
CHUNK = 4096    # tokens per oracle combine chunk
ORACLE_THREADS = 4

FULL = [
    ep_synth.CONFIGS["prefill"],
    ep_synth.CONFIGS["mid"],
    ep_synth.get_workload("sweep-uniform-T4096"),
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
    poison_outputs(b)
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
# dispatch kernels chained by programmatic dependent launch. Every workload
# the benchmark times is here: the sweep's small-T latency points, decode,
# prefill, mid, both sweep T = 4096 points and the default T = 32768.
GRAPH = [
    ep_synth.get_workload("sweep-uniform-T1"),
    ep_synth.get_workload("sweep-zipf-T1"),
    ep_synth.get_workload("sweep-uniform-T8"),
    ep_synth.get_workload("sweep-zipf-T8"),
    ep_synth.get_workload("sweep-uniform-T64"),
    ep_synth.get_workload("sweep-zipf-T64"),
    ep_synth.CONFIGS["decode"].with_(name="decode-T160", T=160),  # the largest batch of the split form
    ep_synth.CONFIGS["decode"],
    ep_synth.get_workload("sweep-zipf-T512"),
    ep_synth.CONFIGS["prefill"],
    ep_synth.CONFIGS["mid"],
    ep_synth.get_workload("sweep-uniform-T4096"),
    ep_synth.get_workload("sweep-zipf-T4096"),
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
    T, H, k = w.T, w.H, w.k
    # route + layout + schedule: every token
    idx, w64 = orc.route(logits, k, w.n_groups, w.topk_groups, w.renormalize)
    lay = orc.layout(idx, w.E, w.R)
    ch, wb = orc.schedule(lay["rank_offset"], w.ranks_per_node, w.self_rank, w.num_workers, w.ranks_per_pod)
    n = int(b.n_chunks.item())
    g = dict(idx=b.topk_idx.cpu().numpy(), w=b.topk_w.cpu().numpy(),
             expert_count=b.expert_count.cpu().numpy(), expert_offset=b.expert_offset.cpu().numpy(),
             rank_count=b.rank_count.cpu().numpy(), rank_offset=b.rank_offset.cpu().numpy(),
             slot=b.slot.cpu().numpy(), chunks=b.chunks[:n].cpu().numpy(), worker_begin=b.worker_begin.cpu().numpy())
    assert_route(g, dict(idx=idx, w=w64), logits, w.renormalize)
    assert_layout(g, dict(chunks=ch, worker_begin=wb, **lay))

    # The oracle's blocks and chunks are independent calls into the C library
    # (ctypes releases the GIL), so a few run at once; each is the oracle as is.
    pool = cf.ThreadPoolExecutor(max_workers=ORACLE_THREADS)

    # dispatch: the whole send buffer and slot_meta, element by element
    blocks = [(c0, min(H, c0 + COLS)) for c0 in range(0, H, COLS)]
    refs = pool.map(lambda c: orc.dispatch(np.ascontiguousarray(x[:, c[0]:c[1]]), lay["slot"]), blocks)
    for (c0, c1), (send_ref, meta_ref) in zip(blocks, refs):
        got = bf16_from_dev(b.send[:, c0:c1].contiguous())
        assert np.array_equal(got, send_ref), f"send buffer differs in columns [{c0}, {c1})"
        if c0 == 0:
            assert np.array_equal(b.slot_meta.cpu().numpy(), meta_ref), "slot_meta differs"
        del send_ref, got

    # combine: every output element, token chunk by token chunk
    def chunk_out(t0):
        t1 = min(T, t0 + CHUNK)
        sub = orc.run_path(logits[t0:t1], x[t0:t1], E=w.E, R=1, k=k, n_groups=w.n_groups,
                           topk_groups=w.topk_groups, renormalize=w.renormalize, ranks_per_node=1, self_rank=0, W=1)
        return t0, t1, sub["idx"], sub["out"]

    worst = 0
    for t0, t1, sub_idx, sub_out in pool.map(chunk_out, range(0, T, CHUNK)):
        assert np.array_equal(sub_idx, idx[t0:t1])  # the chunk routes its tokens as the whole batch does
        d = bf16_ulp_distance(bf16_from_dev(b.out[t0:t1]), sub_out)
        worst = max(worst, int(d.max()))
    pool.shutdown()
    assert worst <= 1, f"combine differs by {worst} bf16 ulp"
