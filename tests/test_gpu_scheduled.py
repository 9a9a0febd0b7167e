"""Schedule-driven dispatch (GPU): ep_dispatch_scheduled against the oracle's
dispatch, bit for bit (send and slot_meta), with the chunk table from
ep_layout (checked against the oracle's first) and with other tables that
tile the rows once (one hop class; whole ranks per worker)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ep_synth
from gpu_harness import bf16_from_dev, bf16_to_dev, require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    require_cuda()
    import combine_router_softmax_gb300 as m

    return m


def setup(ep, orc, w):
    logits = ep_synth.gate_logits(w.seed, w.T, w.E, w.zipf_s)
    x = ep_synth.hidden_bf16_bits(w.seed, w.T, w.H)
    b = ep.LayerBuffers.allocate(ep.EpConfig.from_workload(w))
    b.logits.copy_(torch.from_numpy(logits))
    b.x.copy_(bf16_to_dev(x))
    b.route()
    b.layout()
    torch.cuda.synchronize()
    idx, _ = orc.route(logits, w.k, w.n_groups, w.topk_groups, w.renormalize)
    lay = orc.layout(idx, w.E, w.R)
    ch, wb = orc.schedule(lay["rank_offset"], w.ranks_per_node, w.self_rank, w.num_workers, w.ranks_per_pod)
    n = int(b.n_chunks.item())
    assert np.array_equal(b.slot.cpu().numpy(), lay["slot"])
    assert np.array_equal(b.chunks[:n].cpu().numpy(), ch)
    assert np.array_equal(b.worker_begin.cpu().numpy()[:w.num_workers + 1], wb)
    send, meta = orc.dispatch(x, lay["slot"])
    return b, send, meta


CASES = [
    ep_synth.CONFIGS["tiny"],
    ep_synth.CONFIGS["decode"],
    ep_synth.CONFIGS["decode"].with_(name="decode-T1", T=1),
    ep_synth.CONFIGS["prefill"].with_(name="prefill-T1000", T=1000),
    ep_synth.CONFIGS["mid"].with_(name="mid-T1100", T=1100),
    ep_synth.CONFIGS["prefill"].with_(name="prefill-T700-pods", T=700, ranks_per_node=4, ranks_per_pod=16,
                                      self_rank=21),
    ep_synth.CONFIGS["prefill"].with_(name="W1", T=300, num_workers=1),
    ep_synth.CONFIGS["decode"].with_(name="W5000", T=200, num_workers=5000, ranks_per_node=1, self_rank=63),
    ep_synth.Workload("short-rows-k3", T=513, H=64, E=32, R=4, k=3, num_workers=7),
    ep_synth.Workload("H8-k1", T=100, H=8, E=4, R=2, k=1, num_workers=3),
    ep_synth.Workload("E1024-k32", T=200, H=512, E=1024, R=32, k=32, n_groups=32, topk_groups=4, num_workers=152),
    ep_synth.Workload("rows-48KiB", T=40, H=24576, E=16, R=4, k=4, num_workers=152),
    ep_synth.CONFIGS["prefill"],
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_scheduled_dispatch_vs_oracle(ep, orc, w):
    b, send, meta = setup(ep, orc, w)
    b.send.view(torch.int16).fill_(0x7FC1)
    b.slot_meta.fill_(-9)
    ns = torch.zeros((ep.ep_dispatch_scheduled_ctas(b.cfg), 2), dtype=torch.int64, device="cuda")
    b.dispatch_scheduled(cta_ns=ns)
    torch.cuda.synchronize()
    assert ep.ep_device_error() == 0
    assert np.array_equal(b.slot_meta.cpu().numpy(), meta), "slot_meta differs"
    assert np.array_equal(bf16_from_dev(b.send), send), "send differs"
    t = ns.cpu().numpy()
    assert (t[:, 0] > 0).all() and (t[:, 1] >= t[:, 0]).all()


def _one_class_table(rank_offset, W):
    """Equal row shares of the whole buffer, ignoring hop classes."""
    N = int(rank_offset[-1])
    rows = []
    wb = [0]
    for w in range(W):
        lo, hi = N * w // W, N * (w + 1) // W
        for r in range(len(rank_offset) - 1):
            a, b = max(lo, rank_offset[r]), min(hi, rank_offset[r + 1])
            if b > a:
                rows.append([w, 0, r, a, b - a])
        wb.append(len(rows))
    return rows, wb


def _rank_static_table(rank_offset, W):
    """Worker r mod W takes the whole segment of rank r."""
    per = [[] for _ in range(W)]
    for r in range(len(rank_offset) - 1):
        n = int(rank_offset[r + 1] - rank_offset[r])
        if n:
            per[r % W].append([r % W, 0, r, int(rank_offset[r]), n])
    rows, wb = [], [0]
    for p in per:
        rows += p
        wb.append(len(rows))
    return rows, wb


@pytest.mark.parametrize("kind", ["one-class", "rank-static"])
def test_scheduled_dispatch_other_tables(ep, orc, kind):
    w = ep_synth.CONFIGS["prefill"].with_(name="prefill-T900", T=900)
    b, send, meta = setup(ep, orc, w)
    ro = b.rank_offset.cpu().numpy()
    rows, wb = (_one_class_table if kind == "one-class" else _rank_static_table)(ro, w.num_workers)
    b.chunks.zero_()
    b.chunks[:len(rows)] = torch.tensor(rows, dtype=torch.int32)
    b.worker_begin[:w.num_workers + 1] = torch.tensor(wb, dtype=torch.int32)
    b.n_chunks.fill_(len(rows))
    b.send.zero_()
    b.dispatch_scheduled()
    torch.cuda.synchronize()
    assert ep.ep_device_error() == 0
    assert np.array_equal(b.slot_meta.cpu().numpy(), meta)
    assert np.array_equal(bf16_from_dev(b.send), send)


def test_scheduled_dispatch_bad_table_flags_error(ep, orc):
    """A chunk past the end of the send buffer is caught by the kernel's own
    bounds check: nothing is written for it and error bit 3 is set."""
    w = ep_synth.CONFIGS["decode"].with_(name="decode-T50", T=50)
    b, _, _ = setup(ep, orc, w)
    b.chunks[0, 3] = w.T * w.k - 2  # row_begin
    b.chunks[0, 4] = 5              # row_count: runs past T k
    b.dispatch_scheduled()
    torch.cuda.synchronize()
    assert ep.ep_device_error() & 8
    assert ep.ep_device_error() == 0  # read and cleared


def test_scheduled_dispatch_unsupported_rows(ep):
    cfg = ep.EpConfig.make(T=4, H=32768, E=4, R=2, k=2, num_workers=4)
    b = ep.LayerBuffers.allocate(cfg)
    b.topk_idx.copy_(torch.tensor([[0, 1]] * 4, dtype=torch.int32))
    b.layout()
    with pytest.raises(ep.EpError) as ei:
        b.dispatch_scheduled()
    assert ei.value.status == ep.EP_ERR_UNSUPPORTED
