"""Data-as-Flag by sentinel polling (GPU): ep_dispatch_expert_sp against the
oracle's dispatch + expert, and the bulk-synchronous pair (ep_dispatch then
ep_expert_scale) against the same.

Bars: y (the expert output), slot_meta: bit-exact; send is the sentinel
everywhere after a sentinel-polling call (its payload was consumed and the
buffer re-armed); no device error flag. The layout tables the GPU kernels read
are first checked bit-exact against the oracle's, so both sides start from the
same slots and schedule.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ep_synth
from gpu_harness import bf16_from_dev, bf16_to_dev, require_cuda

pytestmark = pytest.mark.gpu

SENTINEL = 0xFFFF


@pytest.fixture(scope="module")
def ep():
    require_cuda()
    import combine_router_softmax_gb300 as m

    return m


def expert_scales(E: int) -> torch.Tensor:
    """fp32 (e + 1) / E, the scale the oracle's harness expert applies."""
    e = np.arange(E, dtype=np.float32)
    return torch.from_numpy((e + np.float32(1)) / np.float32(E)).cuda()


def setup_layer(ep, orc, w: ep_synth.Workload, x_seed_offset: int = 0):
    logits = ep_synth.gate_logits(w.seed, w.T, w.E, w.zipf_s)
    x = ep_synth.hidden_bf16_bits(w.seed + x_seed_offset, w.T, w.H)
    cfg = ep.EpConfig.from_workload(w)
    b = ep.LayerBuffers.allocate(cfg)
    b.logits.copy_(torch.from_numpy(logits))
    b.x.copy_(bf16_to_dev(x))
    b.route()
    b.layout()
    torch.cuda.synchronize()
    r = orc.run_path(logits, x, E=w.E, R=w.R, k=w.k, n_groups=w.n_groups, topk_groups=w.topk_groups,
                     renormalize=w.renormalize, ranks_per_node=w.ranks_per_node, self_rank=w.self_rank,
                     W=w.num_workers)
    n = int(b.n_chunks.item())
    assert np.array_equal(b.slot.cpu().numpy(), r["slot"])
    assert np.array_equal(b.expert_offset.cpu().numpy(), r["expert_offset"])
    assert np.array_equal(b.chunks[:n].cpu().numpy(), r["chunks"])
    assert np.array_equal(b.worker_begin.cpu().numpy(), r["worker_begin"])
    return b, r


SP = [
    ep_synth.CONFIGS["decode"],
    ep_synth.CONFIGS["decode"].with_(name="decode-T1", T=1),
    ep_synth.CONFIGS["decode"].with_(name="decode-T3-W7", T=3, num_workers=7),
    ep_synth.CONFIGS["prefill"].with_(name="prefill-T1000", T=1000),
    ep_synth.CONFIGS["mid"].with_(name="mid-T1100", T=1100),
    ep_synth.Workload("k4-H512", T=37, H=512, E=16, R=4, k=4, zipf_s=0.0, seed=21, num_workers=5),
    ep_synth.Workload("k4-H24576", T=200, H=24576, E=32, R=8, k=4, zipf_s=1.5, seed=22, num_workers=152),
    ep_synth.Workload("k12-2nodes", T=150, H=1024, E=64, R=16, k=12, zipf_s=0.8, seed=23, ranks_per_node=4,
                      self_rank=9, num_workers=40),
] + [w for w in ep_synth.sweep_workloads() if w.T == 512]


@pytest.mark.parametrize("w", SP, ids=lambda w: w.name)
def test_sentinel_polling_vs_oracle(ep, orc, w):
    b, r = setup_layer(ep, orc, w)
    scale = expert_scales(w.E)
    rows = w.T * w.k
    b.sentinel_arm()
    b.slot_meta.fill_(-7)
    b.y.fill_(0)
    b.dispatch_expert_sp(scale)
    torch.cuda.synchronize()
    assert ep.ep_device_error() == 0
    assert np.array_equal(bf16_from_dev(b.y), r["y"]), "expert output differs"
    assert np.array_equal(b.slot_meta.cpu().numpy(), r["meta"][:rows]), "slot_meta differs"
    assert (bf16_from_dev(b.send) == SENTINEL).all(), "send not re-armed"


@pytest.mark.parametrize("w", SP[:2] + SP[5:7], ids=lambda w: w.name)
def test_bsp_pair_vs_oracle(ep, orc, w):
    b, r = setup_layer(ep, orc, w)
    b.dispatch()
    b.expert_scale(expert_scales(w.E))
    torch.cuda.synchronize()
    assert np.array_equal(bf16_from_dev(b.send), r["send"])
    assert np.array_equal(bf16_from_dev(b.y), r["y"])


def test_sentinel_polling_rounds_rearm(ep, orc):
    """Back-to-back calls on new inputs need no arming in between: each call
    leaves send armed for the next."""
    w = ep_synth.CONFIGS["decode"].with_(name="decode-T64", T=64)
    b, _ = setup_layer(ep, orc, w)
    scale = expert_scales(w.E)
    b.sentinel_arm()
    for rnd in range(3):
        x = ep_synth.hidden_bf16_bits(w.seed + 100 + rnd, w.T, w.H)
        b.x.copy_(bf16_to_dev(x))
        b.dispatch_expert_sp(scale)
        torch.cuda.synchronize()
        assert ep.ep_device_error() == 0
        send_ref, _ = orc.dispatch(x, b.slot.cpu().numpy())
        y_ref = orc.expert(send_ref, b.expert_offset.cpu().numpy(), w.E)
        assert np.array_equal(bf16_from_dev(b.y), y_ref), f"round {rnd}"
        assert (bf16_from_dev(b.send) == SENTINEL).all()


def test_sentinel_polling_in_graph(ep, orc):
    """The call captured in a CUDA graph and replayed, as the benchmark runs it."""
    w = ep_synth.CONFIGS["prefill"].with_(name="prefill-T512", T=512)
    b, r = setup_layer(ep, orc, w)
    scale = expert_scales(w.E)
    b.sentinel_arm()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            b.dispatch_expert_sp(scale, stream=s)
    for _ in range(5):
        b.y.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert ep.ep_device_error() == 0
        assert np.array_equal(bf16_from_dev(b.y), r["y"])


def test_sentinel_polling_unsupported_shapes(ep):
    """k not a multiple of 4, or rows outside 1..48 KiB: EP_ERR_UNSUPPORTED, nothing launched."""
    for w in (ep_synth.Workload("k2", T=8, H=1024, E=8, R=2, k=2, zipf_s=0.0, seed=1),
              ep_synth.Workload("H256", T=8, H=256, E=8, R=2, k=4, zipf_s=0.0, seed=1),
              ep_synth.Workload("H32768", T=8, H=32768, E=8, R=2, k=4, zipf_s=0.0, seed=1)):
        b = ep.LayerBuffers.allocate(ep.EpConfig.from_workload(w))
        b.topk_idx.copy_(torch.arange(w.k, dtype=torch.int32).repeat(w.T, 1))
        b.layout()
        with pytest.raises(ep.EpError) as ei:
            b.dispatch_expert_sp(expert_scales(w.E))
        assert ei.value.status == ep.EP_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert ep.ep_device_error() == 0


# ---------------------------------------------------------------------------
# stop-and-wait baseline (per-row flags)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("w", SP, ids=lambda w: w.name)
def test_stop_and_wait_vs_oracle(ep, orc, w):
    b, r = setup_layer(ep, orc, w)
    rows = w.T * w.k
    flag = torch.zeros(rows, dtype=torch.int32, device="cuda")
    b.slot_meta.fill_(-7)
    b.y.fill_(0)
    b.send.fill_(0)
    b.dispatch_expert_sw(expert_scales(w.E), flag, 1)
    torch.cuda.synchronize()
    assert ep.ep_device_error() == 0
    assert np.array_equal(bf16_from_dev(b.y), r["y"]), "expert output differs"
    assert np.array_equal(bf16_from_dev(b.send), r["send"]), "send differs"
    assert np.array_equal(b.slot_meta.cpu().numpy(), r["meta"][:rows])
    assert (flag.cpu().numpy() == 1).all()


def test_stop_and_wait_epochs_and_graphs(ep, orc):
    """New inputs under new epochs; two captured graphs with alternating
    epochs replayed in turn, as the benchmark runs them."""
    w = ep_synth.CONFIGS["decode"].with_(name="decode-T64", T=64)
    b, _ = setup_layer(ep, orc, w)
    scale = expert_scales(w.E)
    flag = torch.zeros(w.T * w.k, dtype=torch.int32, device="cuda")
    offs = b.expert_offset.cpu().numpy()
    for epoch in (1, 2, 0xFFFFFFFF):
        x = ep_synth.hidden_bf16_bits(w.seed + epoch % 97, w.T, w.H)
        b.x.copy_(bf16_to_dev(x))
        b.dispatch_expert_sw(scale, flag, epoch)
        torch.cuda.synchronize()
        assert ep.ep_device_error() == 0
        send_ref, _ = orc.dispatch(x, b.slot.cpu().numpy())
        assert np.array_equal(bf16_from_dev(b.y), orc.expert(send_ref, offs, w.E)), f"epoch {epoch}"
    s = torch.cuda.Stream()
    graphs = []
    for epoch in (1, 2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                b.dispatch_expert_sw(scale, flag, epoch, stream=s)
        graphs.append(g)
    send_ref, _ = orc.dispatch(ep_synth.hidden_bf16_bits(w.seed + 2, w.T, w.H), b.slot.cpu().numpy())
    y_ref = orc.expert(send_ref, offs, w.E)
    b.x.copy_(bf16_to_dev(ep_synth.hidden_bf16_bits(w.seed + 2, w.T, w.H)))
    for i in range(6):
        b.y.fill_(0)
        graphs[i % 2].replay()
        torch.cuda.synchronize()
        assert ep.ep_device_error() == 0
        assert np.array_equal(bf16_from_dev(b.y), y_ref)
        assert (flag.cpu().numpy() == (1 if i % 2 == 0 else 2)).all()
