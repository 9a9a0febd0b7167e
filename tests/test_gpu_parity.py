"""CUDA path vs the CPU oracle, element by element (GPU).

Every input is seeded and synthetic (ep_synth) and goes, byte for byte, to both
sides; no oracle input comes from the GPU. Bars:

* topk_idx, counts, offsets, slot, chunk schedule, send buffer, slot_meta:
  bit-exact.
* topk_w (fp32 on the GPU, fp64 in the oracle): relative error within the
  bound derived from the fp32 arithmetic (``gpu_harness.route_weight_rtol``):
  the rounding of l - l_max (2^-24 |d|), expf (<= 2 ulp), the warp-tree sum
  and the division, with a 1.5x margin -- about 2^-18 here.
* combine fed the oracle's own slot / weights / expert rows: bit-exact (the
  same fp32 fma sequence and RNE rounding on both sides).
* the whole chain (GPU route weights differ from the oracle's by the bound
  above): combine output within 1 bf16 ulp of the oracle's.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import ep_synth
from gpu_harness import (bf16_from_dev, bf16_to_dev, bf16_ulp_distance, require_cuda, route_weight_rtol,
                         synthetic_expert)
from pins import check_schedule_invariants

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    require_cuda()
    import combine_router_softmax_gb300 as m

    return m


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def make_inputs(w: ep_synth.Workload):
    logits = ep_synth.gate_logits(w.seed, w.T, w.E, w.zipf_s)
    x = ep_synth.hidden_bf16_bits(w.seed, w.T, w.H)
    return logits, x


def run_gpu(ep, w, logits, x_bits, identity=False):
    cfg = ep.EpConfig.from_workload(w)
    b = ep.LayerBuffers.allocate(cfg)
    b.logits.copy_(torch.from_numpy(logits))
    b.x.copy_(bf16_to_dev(x_bits))
    b.send.fill_(0)
    b.slot_meta.fill_(-7)
    b.route()
    b.layout()
    b.dispatch()
    synthetic_expert(b.send, b.expert_offset, w.E, identity, out=b.y)
    b.combine()
    torch.cuda.synchronize()
    n = int(b.n_chunks.item())
    return b, dict(
        idx=b.topk_idx.cpu().numpy(), w=b.topk_w.cpu().numpy(),
        expert_count=b.expert_count.cpu().numpy(), expert_offset=b.expert_offset.cpu().numpy(),
        rank_count=b.rank_count.cpu().numpy(), rank_offset=b.rank_offset.cpu().numpy(),
        slot=b.slot.cpu().numpy(), chunks=b.chunks[:n].cpu().numpy(),
        worker_begin=b.worker_begin.cpu().numpy(), meta=b.slot_meta.cpu().numpy())


def run_oracle(orc, w, logits, x_bits, identity=False):
    return orc.run_path(logits, x_bits, E=w.E, R=w.R, k=w.k, n_groups=w.n_groups, topk_groups=w.topk_groups,
                        renormalize=w.renormalize, ranks_per_node=w.ranks_per_node, self_rank=w.self_rank,
                        W=w.num_workers, identity_expert=identity, ranks_per_pod=w.ranks_per_pod)


def assert_route(g, r, logits, renormalize):
    assert np.array_equal(g["idx"], r["idx"]), "topk_idx differs"
    rtol = route_weight_rtol(logits, r["idx"], renormalize)
    rel = np.abs(g["w"].astype(np.float64) - r["w"]) / r["w"]
    bad = rel > rtol[:, None]
    assert not bad.any(), f"topk_w beyond bound at {np.argwhere(bad)[:5]}: rel {rel[bad][:5]} tol {rtol[np.argwhere(bad)[:5, 0]]}"


def assert_layout(g, r):
    for key in ("expert_count", "expert_offset", "rank_count", "rank_offset", "slot"):
        assert np.array_equal(g[key], r[key]), f"{key} differs"
    assert np.array_equal(g["chunks"], r["chunks"]), "chunk table differs"
    assert np.array_equal(g["worker_begin"], r["worker_begin"]), "worker_begin differs"


# ---------------------------------------------------------------------------
# whole path, element by element, at sizes the oracle finishes in seconds
# ---------------------------------------------------------------------------

SMALL = [
    ep_synth.CONFIGS["tiny"],
    ep_synth.CONFIGS["decode"],
    ep_synth.CONFIGS["prefill"].with_(name="prefill-T1000", T=1000),
    ep_synth.CONFIGS["mid"].with_(name="mid-T1100", T=1100),
    ep_synth.CONFIGS["tiny"].with_(name="tiny-plain-softmax", renormalize=0),
    ep_synth.CONFIGS["mid"].with_(name="mid-T300-plain", T=300, renormalize=0),
    ep_synth.CONFIGS["tiny"].with_(name="tiny-2nodes", ranks_per_node=2, self_rank=3, num_workers=5),
    ep_synth.CONFIGS["tiny"].with_(name="tiny-3tiers", ranks_per_node=1, ranks_per_pod=2, self_rank=2, num_workers=5),
    ep_synth.CONFIGS["prefill"].with_(name="prefill-T1000-pods", T=1000, ranks_per_node=4, ranks_per_pod=16,
                                      self_rank=21),
] + [w for w in ep_synth.sweep_workloads() if w.T <= 512]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_path_parity(ep, orc, w):
    logits, x = make_inputs(w)
    b, g = run_gpu(ep, w, logits, x)
    r = run_oracle(orc, w, logits, x)
    assert_route(g, r, logits, w.renormalize)
    assert_layout(g, r)
    assert np.array_equal(bf16_from_dev(b.send), r["send"]), "send buffer differs"
    assert np.array_equal(g["meta"], r["meta"]), "slot_meta differs"
    d = bf16_ulp_distance(bf16_from_dev(b.out), r["out"])
    assert d.max() <= 1, f"combine differs by {d.max()} bf16 ulp"


def test_identity_expert_reconstructs_x(ep, orc):
    """dispatch -> identity expert -> combine with renormalised weights gives x back exactly."""
    w = ep_synth.CONFIGS["decode"].with_(T=300)
    logits, x = make_inputs(w)
    b, _ = run_gpu(ep, w, logits, x, identity=True)
    assert np.array_equal(bf16_from_dev(b.out), x)


# ---------------------------------------------------------------------------
# single calls fed the oracle's own intermediates: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("k,E,H,T", [(1, 8, 256, 100), (2, 8, 296, 129), (4, 64, 1032, 257), (6, 64, 4096, 70),
                                     (8, 256, 7168, 64), (3, 16, 520, 90), (12, 64, 264, 33), (32, 1024, 136, 20)])
def test_combine_bit_exact(ep, orc, k, E, H, T):
    """Oracle slot / fp32 weights / random mixed-sign expert rows into ep_combine."""
    logits = ep_synth.gate_logits(7, T, E)
    idx, w64 = orc.route(logits, k)
    lay = orc.layout(idx, E, 1)
    w32 = w64.astype(np.float32)
    y = ep_synth.random_rows_bf16_bits(11, T * k, H)
    ref = orc.combine(y, lay["slot"], w32)
    cfg = ep.EpConfig.make(T=T, H=H, E=E, R=1, k=k, num_workers=4)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    ep.ep_combine(cfg, bf16_to_dev(y), torch.from_numpy(lay["slot"]).cuda(), torch.from_numpy(w32).cuda(), out)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_from_dev(out), ref)


@pytest.mark.parametrize("k,E,H,T", [(1, 8, 8, 300), (2, 8, 296, 129), (8, 256, 7168, 40), (5, 32, 1024, 77),
                                     (32, 1024, 64, 9), (4, 64, 520, 1000), (8, 256, 4096, 2000),
                                     (12, 64, 2048, 333), (32, 1024, 1024, 31), (8, 128, 24576, 17)])
def test_dispatch_bit_exact(ep, orc, k, E, H, T):
    """Oracle slots into ep_dispatch; covers the vector path (short rows, k % 4 != 0)
    and the bulk-copy path (k % 4 == 0, rows >= 1 KiB), ragged T."""
    logits = ep_synth.gate_logits(8, T, E)
    idx, _ = orc.route(logits, k)
    lay = orc.layout(idx, E, 1)
    x = ep_synth.hidden_bf16_bits(8, T, H)
    send_ref, meta_ref = orc.dispatch(x, lay["slot"])
    cfg = ep.EpConfig.make(T=T, H=H, E=E, R=1, k=k, num_workers=4)
    send = torch.zeros((T * k, H), dtype=torch.bfloat16, device="cuda")
    meta = torch.full((T * k,), -1, dtype=torch.int32, device="cuda")
    ep.ep_dispatch(cfg, bf16_to_dev(x), torch.from_numpy(lay["slot"]).cuda(), send, meta)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_from_dev(send), send_ref)
    assert np.array_equal(meta.cpu().numpy(), meta_ref)


# ---------------------------------------------------------------------------
# route / layout / schedule edge cases
# ---------------------------------------------------------------------------

def _route_layout(ep, orc, w, logits):
    cfg = ep.EpConfig.from_workload(w)
    b = ep.LayerBuffers.allocate(cfg)
    b.logits.copy_(torch.from_numpy(logits))
    b.route()
    b.layout()
    torch.cuda.synchronize()
    n = int(b.n_chunks.item())
    g = dict(idx=b.topk_idx.cpu().numpy(), w=b.topk_w.cpu().numpy(),
             expert_count=b.expert_count.cpu().numpy(), expert_offset=b.expert_offset.cpu().numpy(),
             rank_count=b.rank_count.cpu().numpy(), rank_offset=b.rank_offset.cpu().numpy(),
             slot=b.slot.cpu().numpy(), chunks=b.chunks[:n].cpu().numpy(), worker_begin=b.worker_begin.cpu().numpy())
    idx, w64 = orc.route(logits, w.k, w.n_groups, w.topk_groups, w.renormalize)
    lay = orc.layout(idx, w.E, w.R)
    ch, wb = orc.schedule(lay["rank_offset"], w.ranks_per_node, w.self_rank, w.num_workers, w.ranks_per_pod)
    r = dict(idx=idx, w=w64, chunks=ch, worker_begin=wb, **lay)
    return g, r


EDGE = [
    ("T1", ep_synth.CONFIGS["decode"].with_(T=1), None),
    ("ties", ep_synth.CONFIGS["decode"].with_(T=700), "ties"),
    ("one-hot-expert", ep_synth.CONFIGS["decode"].with_(T=600, k=1), "hot"),
    ("hot-expert-k8", ep_synth.CONFIGS["prefill"].with_(T=513), "hot"),
    ("E1024-k32", ep_synth.Workload("max", T=300, H=64, E=1024, R=32, k=32, num_workers=152), None),
    ("E1024-k32-groups", ep_synth.Workload("maxg", T=97, H=64, E=1024, R=8, k=32, n_groups=32, topk_groups=3,
                                           num_workers=10), None),
    ("k12-groups", ep_synth.Workload("k12", T=257, H=64, E=96, R=6, k=12, n_groups=6, topk_groups=2,
                                     ranks_per_node=2, self_rank=5, num_workers=33), None),
    ("E8-k8-all", ep_synth.Workload("all", T=50, H=64, E=8, R=2, k=8, num_workers=3), None),
    ("W1", ep_synth.CONFIGS["prefill"].with_(T=300, num_workers=1), None),
    ("W1500", ep_synth.CONFIGS["prefill"].with_(T=300, num_workers=1500), None),
    ("W5000-rpn1", ep_synth.CONFIGS["decode"].with_(T=200, num_workers=5000, ranks_per_node=1, self_rank=63), None),
    ("rpn-ge-R", ep_synth.CONFIGS["decode"].with_(T=200, ranks_per_node=100, self_rank=10), None),
    ("zipf-empty-experts", ep_synth.CONFIGS["prefill"].with_(T=40, zipf_s=3.0), None),
    ("pods-W5000", ep_synth.CONFIGS["decode"].with_(T=200, num_workers=5000, ranks_per_node=2, ranks_per_pod=8,
                                                    self_rank=63), None),
    ("pods-W1", ep_synth.CONFIGS["prefill"].with_(T=300, num_workers=1, ranks_per_node=1, ranks_per_pod=4,
                                                  self_rank=6), None),
    ("pod-ge-R", ep_synth.CONFIGS["decode"].with_(T=200, ranks_per_node=4, ranks_per_pod=128, self_rank=10), None),
    ("pods-E1024", ep_synth.Workload("maxp", T=300, H=64, E=1024, R=1024, k=32, ranks_per_node=8, ranks_per_pod=64,
                                     self_rank=1000, num_workers=152), None),
    # group sizes around the shuffle path's limits: 24 and 64 experts per group (shared-memory path), one and two
    # experts per group (shuffle path)
    ("groups-of-24", ep_synth.Workload("g24", T=200, H=64, E=96, R=4, k=6, n_groups=4, topk_groups=2,
                                       num_workers=40), None),
    ("groups-of-64", ep_synth.Workload("g64", T=200, H=64, E=512, R=8, k=8, n_groups=8, topk_groups=3,
                                       num_workers=40), None),
    ("groups-of-1", ep_synth.Workload("g1", T=200, H=64, E=32, R=4, k=8, n_groups=32, topk_groups=8,
                                      num_workers=40), None),
    ("groups-of-2-ties", ep_synth.Workload("g2", T=300, H=64, E=64, R=4, k=4, n_groups=32, topk_groups=3,
                                           num_workers=40), "ties"),
]


@pytest.mark.parametrize("name,w,mode", EDGE, ids=[e[0] for e in EDGE])
def test_route_layout_edges(ep, orc, name, w, mode):
    logits = ep_synth.gate_logits(w.seed + 3, w.T, w.E, w.zipf_s)
    if mode == "ties":
        logits = (np.round(logits * 2) / 2).astype(np.float32)
    elif mode == "hot":
        logits[:, 5] += 40.0
    g, r = _route_layout(ep, orc, w, logits)
    assert_route(g, r, logits, w.renormalize)
    assert_layout(g, r)
    check_schedule_invariants(g["chunks"], g["worker_begin"], g["rank_offset"], w.ranks_per_node, w.self_rank,
                              w.num_workers, w.ranks_per_pod)


def test_layout_T0(ep):
    cfg = ep.EpConfig.make(T=0, H=64, E=16, R=4, k=2, num_workers=7)
    b = ep.LayerBuffers.allocate(cfg)
    for t in (b.expert_count, b.expert_offset, b.rank_count, b.rank_offset, b.worker_begin, b.n_chunks):
        t.fill_(-5)
    b.route()
    b.layout()
    b.dispatch()
    b.combine()
    torch.cuda.synchronize()
    for t in (b.expert_count, b.expert_offset, b.rank_count, b.rank_offset, b.worker_begin, b.n_chunks):
        assert (t == 0).all()


def test_invalid_slots_are_skipped(ep, orc):
    """Slots outside [0, T k) write nothing (dispatch) and add nothing (combine)."""
    T, H, E, k = 64, 256, 16, 4
    logits = ep_synth.gate_logits(2, T, E)
    idx, w64 = orc.route(logits, k)
    lay = orc.layout(idx, E, 1)
    slot = lay["slot"].copy()
    slot[3, 1] = -1
    slot[10, 0] = T * k + 5
    w32 = w64.astype(np.float32)
    x = ep_synth.hidden_bf16_bits(2, T, H)
    cfg = ep.EpConfig.make(T=T, H=H, E=E, R=1, k=k, num_workers=4)
    send = torch.full((T * k, H), 0x7FC1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    meta = torch.full((T * k,), -9, dtype=torch.int32, device="cuda")
    ep.ep_dispatch(cfg, bf16_to_dev(x), torch.from_numpy(slot).cuda(), send, meta)
    y = ep_synth.random_rows_bf16_bits(5, T * k, H)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    ep.ep_combine(cfg, bf16_to_dev(y), torch.from_numpy(slot).cuda(), torch.from_numpy(w32).cuda(), out)
    torch.cuda.synchronize()
    untouched = [lay["slot"][3, 1], lay["slot"][10, 0]]
    s_np = bf16_from_dev(send)
    for row in untouched:
        assert (s_np[row] == 0x7FC1).all() and meta[row].item() == -9
    # the oracle with those two weights zeroed (fma(0, y, acc) = acc for finite y)
    w_ref = w32.copy()
    w_ref[3, 1] = 0.0
    w_ref[10, 0] = 0.0
    slot_ref = lay["slot"]
    assert np.array_equal(bf16_from_dev(out), orc.combine(y, slot_ref, w_ref))


def test_argument_errors(ep):
    cfg = ep.EpConfig.make(T=16, H=12, E=8, R=4, k=2, num_workers=4)
    x = torch.zeros((16, 12), dtype=torch.bfloat16, device="cuda")
    slot = torch.zeros((16, 2), dtype=torch.int32, device="cuda")
    send = torch.zeros((32, 12), dtype=torch.bfloat16, device="cuda")
    meta = torch.zeros((32,), dtype=torch.int32, device="cuda")
    with pytest.raises(ep.EpError) as ei:
        ep.ep_dispatch(cfg, x, slot, send, meta)
    assert ei.value.status == ep.EP_ERR_UNSUPPORTED
    cfg = ep.EpConfig.make(T=16, H=16, E=8, R=4, k=2, num_workers=4)
    big = torch.zeros((16 * 16 + 8,), dtype=torch.bfloat16, device="cuda")
    lib = ep._lib
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.ep_dispatch(ctypes.byref(cfg), ctypes.c_void_p(big.data_ptr() + 2), ctypes.c_void_p(slot.data_ptr()),
                         ctypes.c_void_p(send.data_ptr()), ctypes.c_void_p(meta.data_ptr()), stream)
    assert rc == ep.EP_ERR_INVALID_ARG  # misaligned x
    bad = ep.EpConfig.make(T=16, H=16, E=8, R=3, k=2, num_workers=4)
    with pytest.raises(ep.EpError):
        ep.ep_route(bad, torch.zeros((16, 8), device="cuda"), slot, torch.zeros((16, 2), device="cuda"))
    b = ep.LayerBuffers.allocate(cfg)
    with pytest.raises(ep.EpError) as ei:
        ep.ep_layout(cfg, b.topk_idx, b.expert_count, b.expert_offset, b.rank_count, b.rank_offset, b.slot,
                     b.chunks[:3], b.n_chunks, b.worker_begin, b.workspace)
    assert ei.value.status == ep.EP_ERR_CAPACITY


def test_tensor_on_another_device_rejected(ep, monkeypatch):
    """The binding refuses tensors (and streams) of a device other than the
    current one before anything is launched; one GPU is enough to check it by
    making the binding believe another device is current."""
    cfg = ep.EpConfig.make(T=16, H=16, E=8, R=4, k=2, num_workers=4)
    b = ep.LayerBuffers.allocate(cfg)
    stream = torch.cuda.current_stream()
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 1)
    with pytest.raises(ValueError, match="current device is cuda:1"):
        ep.ep_dispatch(cfg, b.x, b.slot, b.send, b.slot_meta)
    with pytest.raises(ValueError, match="stream: on cuda:0"):
        ep._stream(stream)


@pytest.mark.parametrize("E,k,renorm", [(4, 1, 1), (4, 3, 0), (16, 5, 1), (32, 8, 1), (32, 2, 0), (64, 4, 1),
                                        (128, 8, 0), (512, 6, 1), (1024, 8, 1), (1024, 7, 0), (96, 8, 1)])
def test_route_shapes(ep, orc, E, k, renorm):
    """Every lanes-per-token variant of the route kernels (1 .. 32 lanes), ties included."""
    T = 333
    logits = ep_synth.gate_logits(17, T, E)
    logits[::3] = np.round(logits[::3] * 2) / 2  # every third token: coarse grid, many ties
    cfg = ep.EpConfig.make(T=T, H=8, E=E, R=1, k=k, renormalize=renorm, num_workers=2)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ep.ep_route(cfg, torch.from_numpy(logits).cuda(), idx, w)
    torch.cuda.synchronize()
    r_idx, r_w = orc.route(logits, k, renormalize=renorm)
    assert_route(dict(idx=idx.cpu().numpy(), w=w.cpu().numpy()), dict(idx=r_idx, w=r_w), logits, renorm)


def test_route_unaligned_logits(ep, orc):
    """A logits pointer that is not 16-byte aligned takes the general kernel."""
    T, E, k = 50, 256, 8
    logits = ep_synth.gate_logits(18, T, E)
    buf = torch.empty(T * E + 1, dtype=torch.float32, device="cuda")
    view = buf[1:].view(T, E)
    view.copy_(torch.from_numpy(logits))
    cfg = ep.EpConfig.make(T=T, H=8, E=E, R=1, k=k, num_workers=2)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ep.ep_route(cfg, view, idx, w)
    torch.cuda.synchronize()
    r_idx, r_w = orc.route(logits, k)
    assert_route(dict(idx=idx.cpu().numpy(), w=w.cpu().numpy()), dict(idx=r_idx, w=r_w), logits, 1)


@pytest.mark.parametrize("T,E,R,k,rpp", [(400_000, 256, 32, 8, 0), (160_000, 1024, 64, 32, 32),
                                          (100_000, 256, 32, 8, 0), (20_000, 1024, 64, 32, 0)])
def test_layout_many_ctas(ep, orc, T, E, R, k, rpp):
    """T beyond one co-resident grid: the three-kernel layout path (T = 400000, 160000). And single-kernel
    layouts of more than 64 CTAs, whose count table takes a thread several batches of polled loads: T = 100000
    (98 CTAs of 32 warps, 16 loads per batch) and T = 20000 at E = 1024 (79 CTAs of 8 warps, 4 columns and
    79 rows per thread, 32 loads per batch)."""
    rng = np.random.default_rng(T)
    base = rng.integers(0, E, size=(T, 1))
    step = rng.integers(1, E // k + 1, size=(T, 1))
    idx = ((base + step * np.arange(k)[None, :]) % E).astype(np.int32)  # k distinct experts per token
    assert (np.sort(idx, axis=1)[:, 1:] != np.sort(idx, axis=1)[:, :-1]).all()
    w = ep_synth.Workload("many", T=T, H=8, E=E, R=R, k=k, num_workers=152, ranks_per_pod=rpp, self_rank=R - 1)
    cfg = ep.EpConfig.from_workload(w)
    b = ep.LayerBuffers.allocate(cfg)
    b.topk_idx.copy_(torch.from_numpy(idx))
    b.layout()
    torch.cuda.synchronize()
    lay = orc.layout(idx, E, R)
    ch, wb = orc.schedule(lay["rank_offset"], w.ranks_per_node, w.self_rank, w.num_workers, w.ranks_per_pod)
    n = int(b.n_chunks.item())
    g = dict(expert_count=b.expert_count.cpu().numpy(), expert_offset=b.expert_offset.cpu().numpy(),
             rank_count=b.rank_count.cpu().numpy(), rank_offset=b.rank_offset.cpu().numpy(),
             slot=b.slot.cpu().numpy(), chunks=b.chunks[:n].cpu().numpy(), worker_begin=b.worker_begin.cpu().numpy())
    assert_layout(g, dict(chunks=ch, worker_begin=wb, **lay))


def test_no_device_error_flags(ep):
    """No kernel ran out of a bounded wait during the tests above."""
    assert ep.ep_device_error() == 0


@pytest.mark.parametrize("polls", [1, 1000, 100000])
def test_bounded_wait_gives_up(ep, polls):
    """A grid barrier that can never complete returns (both CTAs give up and say so, and a late arrival
    sees the failure), a wait on a ready flag that is never set returns too, and so does a count-table
    read whose row is published too late (the reader gives up, the late owner learns it failed)."""
    gave_up = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ep.ep_check_bounded_wait(polls, gave_up)
    torch.cuda.synchronize()
    # two barrier waiters, one flag waiter, the table reader and the late table owner; no late CTA went on
    assert int(gave_up.item()) == 5
    # the context is still usable afterwards
    z = torch.ones(4, device="cuda") * 2
    assert float(z.sum()) == 8.0


# ---------------------------------------------------------------------------
# ep_dispatch_fused: the same outputs as ep_route + ep_layout + ep_dispatch
# ---------------------------------------------------------------------------

FUSED = [
    ep_synth.CONFIGS["tiny"],
    ep_synth.CONFIGS["decode"],
    ep_synth.CONFIGS["prefill"],
    ep_synth.CONFIGS["mid"],
    ep_synth.CONFIGS["prefill"].with_(name="prefill-T1000", T=1000),
    ep_synth.CONFIGS["mid"].with_(name="mid-T300-plain", T=300, renormalize=0),
    ep_synth.CONFIGS["tiny"].with_(name="tiny-2nodes", ranks_per_node=2, self_rank=3, num_workers=5),
    ep_synth.Workload("k6-vector", T=777, H=1024, E=64, R=8, k=6, num_workers=20),
    ep_synth.Workload("short-rows", T=500, H=64, E=32, R=4, k=4, num_workers=7),
    ep_synth.Workload("E1024-k32", T=300, H=512, E=1024, R=32, k=32, n_groups=32, topk_groups=4, num_workers=152),
    ep_synth.Workload("k12-groups", T=257, H=2048, E=96, R=6, k=12, n_groups=6, topk_groups=2, ranks_per_node=2,
                      self_rank=5, num_workers=33),
    ep_synth.Workload("fallback-T80000", T=80000, H=256, E=256, R=32, k=8, num_workers=152),
    ep_synth.Workload("pods-T64", T=64, H=7168, E=256, R=64, k=8, ranks_per_node=4, ranks_per_pod=16, self_rank=33,
                      num_workers=152),
    ep_synth.Workload("pods-T4096", T=4096, H=1024, E=256, R=64, k=8, ranks_per_node=4, ranks_per_pod=16,
                      self_rank=5, num_workers=152),
    # the split form (T <= 160): one row per data CTA, or one token per data CTA when rows outnumber them
    ep_synth.Workload("split-k6", T=40, H=1024, E=64, R=8, k=6, num_workers=20),
    ep_synth.Workload("split-k32-E1024", T=50, H=512, E=1024, R=32, k=32, n_groups=32, topk_groups=4,
                      num_workers=152),
    ep_synth.Workload("split-k12-groups", T=57, H=2048, E=96, R=6, k=12, n_groups=6, topk_groups=2,
                      ranks_per_node=2, self_rank=5, num_workers=33),
    ep_synth.CONFIGS["prefill"].with_(name="split-T63-plain", T=63, renormalize=0),
    # tiles of 4 tokens up to T = 64, else 8: a single tile CTA of 3 tokens, tiles of 3 and 2, then 9 tiles of 8/7
    ep_synth.CONFIGS["decode"].with_(name="split-T3", T=3),
    ep_synth.CONFIGS["decode"].with_(name="split-T5", T=5),
    ep_synth.CONFIGS["decode"].with_(name="split-T65", T=65),
    ep_synth.CONFIGS["decode"].with_(name="split-T160", T=160),
    ep_synth.CONFIGS["decode"].with_(name="fused-T161", T=161),
    # either side of the small-batch kernel's upper bound (1760 tokens)
    ep_synth.CONFIGS["decode"].with_(name="fused-T1760", T=1760),
    ep_synth.CONFIGS["decode"].with_(name="three-kernels-T1761", T=1761),
    # above the small-batch kernel's range (route, layout and dispatch kernels; ragged last layout CTA)
    ep_synth.Workload("three-kernels-groups-T3001", T=3001, H=1024, E=128, R=16, k=8, n_groups=8, topk_groups=4,
                      num_workers=152),
    ep_synth.Workload("three-kernels-g24-T2500", T=2500, H=1024, E=96, R=6, k=6, n_groups=4, topk_groups=2,
                      ranks_per_node=2, self_rank=5, num_workers=33),
    ep_synth.Workload("three-kernels-E1024-T2600", T=2600, H=512, E=1024, R=32, k=32, num_workers=152),
    ep_synth.CONFIGS["prefill"].with_(name="three-kernels-plain-T4095", T=4095, renormalize=0),
] + [w for w in ep_synth.sweep_workloads() if w.T in (1, 8, 64, 512, 4096, 32768)]


@pytest.mark.parametrize("w", FUSED, ids=lambda w: w.name)
def test_dispatch_fused_matches_separate(ep, w):
    logits = torch.from_numpy(ep_synth.gate_logits(w.seed, w.T, w.E, w.zipf_s)).cuda()
    x = bf16_to_dev(ep_synth.hidden_bf16_bits(w.seed, w.T, w.H))
    cfg = ep.EpConfig.from_workload(w)
    a = ep.LayerBuffers.allocate(cfg)
    f = ep.LayerBuffers.allocate(cfg)
    for b_ in (a, f):
        b_.logits.copy_(logits)
        b_.x.copy_(x)
    a.send.fill_(0)
    f.send.view(torch.int16).fill_(0x7FC1)
    f.slot_meta.fill_(-9)
    a.route(); a.layout(); a.dispatch()
    f.dispatch_fused()
    torch.cuda.synchronize()
    assert ep.ep_device_error() == 0
    for name in ("topk_idx", "topk_w", "expert_count", "expert_offset", "rank_count", "rank_offset", "slot",
                 "worker_begin", "send", "slot_meta", "n_chunks"):
        ga, gf = getattr(a, name), getattr(f, name)
        if name == "worker_begin":
            W = w.num_workers
            ga, gf = ga[:W + 1], gf[:W + 1]
        assert torch.equal(ga.view(torch.int32) if ga.dtype == torch.float32 else ga,
                           gf.view(torch.int32) if gf.dtype == torch.float32 else gf), f"{name} differs"
    n = int(a.n_chunks.item())
    assert torch.equal(a.chunks[:n], f.chunks[:n])


def test_dispatch_fused_vs_oracle(ep, orc):
    """The fused call against the oracle directly (prefill shape, T = 2000)."""
    w = ep_synth.CONFIGS["prefill"].with_(T=2000)
    logits, x = make_inputs(w)
    cfg = ep.EpConfig.from_workload(w)
    b = ep.LayerBuffers.allocate(cfg)
    b.logits.copy_(torch.from_numpy(logits))
    b.x.copy_(bf16_to_dev(x))
    b.dispatch_fused()
    synthetic_expert(b.send, b.expert_offset, w.E, out=b.y)
    b.combine()
    torch.cuda.synchronize()
    r = run_oracle(orc, w, logits, x)
    n = int(b.n_chunks.item())
    g = dict(idx=b.topk_idx.cpu().numpy(), w=b.topk_w.cpu().numpy(),
             expert_count=b.expert_count.cpu().numpy(), expert_offset=b.expert_offset.cpu().numpy(),
             rank_count=b.rank_count.cpu().numpy(), rank_offset=b.rank_offset.cpu().numpy(),
             slot=b.slot.cpu().numpy(), chunks=b.chunks[:n].cpu().numpy(), worker_begin=b.worker_begin.cpu().numpy())
    assert_route(g, r, logits, w.renormalize)
    assert_layout(g, r)
    assert np.array_equal(bf16_from_dev(b.send), r["send"])
    assert np.array_equal(b.slot_meta.cpu().numpy(), r["meta"])
    assert bf16_ulp_distance(bf16_from_dev(b.out), r["out"]).max() <= 1


# ---------------------------------------------------------------------------
# tiling boundaries: where the layout's tokens per warp change (its grid is
# kept near 64 CTAs of 16 warps) and where the fused dispatch kernel's range
# ends (at most 8 tokens per tile, one resident slot kept for the schedule CTA)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T", [1023, 1024, 1025, 2047, 2049, 4095, 4097, 8191, 8193, 16385, 32769])
def test_layout_tiling_boundaries(ep, orc, T):
    w = ep_synth.CONFIGS["prefill"].with_(name=f"prefill-T{T}", T=T)
    logits = ep_synth.gate_logits(w.seed + 7, w.T, w.E, w.zipf_s)
    g, r = _route_layout(ep, orc, w, logits)
    assert_route(g, r, logits, w.renormalize)
    assert_layout(g, r)


# either side of the small-batch kernel's upper bound (1760 tokens; above it the call runs the route, layout
# and dispatch kernels), and 16 tokens per CTA on 152 SMs and one more
@pytest.mark.parametrize("T", [1759, 1760, 1761, 1762, 2432, 2433])
def test_dispatch_fused_form_boundary(ep, T):
    w = ep_synth.CONFIGS["prefill"].with_(name=f"prefill-T{T}", T=T)
    logits = torch.from_numpy(ep_synth.gate_logits(w.seed, w.T, w.E, w.zipf_s)).cuda()
    x = bf16_to_dev(ep_synth.hidden_bf16_bits(w.seed, w.T, w.H))
    cfg = ep.EpConfig.from_workload(w)
    a = ep.LayerBuffers.allocate(cfg)
    f = ep.LayerBuffers.allocate(cfg)
    for b_ in (a, f):
        b_.logits.copy_(logits)
        b_.x.copy_(x)
    a.route(); a.layout(); a.dispatch()
    f.dispatch_fused()
    torch.cuda.synchronize()
    assert ep.ep_device_error() == 0
    for name in ("topk_idx", "expert_offset", "rank_offset", "slot", "send", "slot_meta", "n_chunks"):
        assert torch.equal(getattr(a, name), getattr(f, name)), f"{name} differs"
    n = int(a.n_chunks.item())
    assert torch.equal(a.chunks[:n], f.chunks[:n])
    assert torch.equal(a.worker_begin[:w.num_workers + 1], f.worker_begin[:w.num_workers + 1])
