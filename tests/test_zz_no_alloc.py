"""ep_layout_static: the layout entry point for callers that cannot allocate.

Some callers cannot allocate device memory when they run the layout (an engine
that owns all of its device memory and hands a library only the inputs and
outputs, or code running where allocation is not allowed), so they cannot pass
ep_layout's workspace. ep_layout_static takes its scratch from a fixed device
array inside the library instead. This test calls it through the C ABI twice in
a row, on different inputs, and checks every output against ep_layout's on the
same inputs (layout results are integers: bit-exact), then checks that a shape
needing more than the array is rejected before anything is launched.

The file sorts last so that a run stopping at the first failure has run every
other test first; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import ep_synth
from gpu_harness import require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    require_cuda()
    import combine_router_softmax_gb300 as m

    return m


def _outputs(ep, cfg, device="cuda"):
    T, E, R, k = cfg.T, cfg.E, cfg.R, cfg.k
    cap = ep.ep_schedule_capacity(cfg)
    W = (cap - R) // 2
    i32 = dict(dtype=torch.int32, device=device)
    return dict(expert_count=torch.full((E,), -3, **i32), expert_offset=torch.full((E + 1,), -3, **i32),
                rank_count=torch.full((R,), -3, **i32), rank_offset=torch.full((R + 1,), -3, **i32),
                slot=torch.full((T, k), -3, **i32), chunks=torch.full((cap, 5), -3, **i32),
                n_chunks=torch.full((1,), -3, **i32), worker_begin=torch.full((W + 1,), -3, **i32))


def _static_call(ep, cfg, idx, o):
    """ep_layout_static through the raw C ABI (ctypes), current stream."""
    vp = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = ep._lib.ep_layout_static(ctypes.byref(cfg), vp(idx), vp(o["expert_count"]), vp(o["expert_offset"]),
                                  vp(o["rank_count"]), vp(o["rank_offset"]), vp(o["slot"]), vp(o["chunks"]),
                                  ctypes.c_int32(o["chunks"].shape[0]), vp(o["n_chunks"]), vp(o["worker_begin"]),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc


def _route(ep, w, seed):
    cfg = ep.EpConfig.from_workload(w)
    logits = torch.from_numpy(ep_synth.gate_logits(seed, w.T, w.E, w.zipf_s)).cuda()
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    wts = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    ep.ep_route(cfg, logits, idx, wts)
    return cfg, idx


def test_static_layout_matches_workspace_layout_twice(ep):
    cases = [ep_synth.CONFIGS["prefill"].with_(T=3000), ep_synth.CONFIGS["mid"].with_(T=777, num_workers=40)]
    for call, (w, seed) in enumerate(zip(cases, (5, 6))):
        cfg, idx = _route(ep, w, seed)
        ref = _outputs(ep, cfg)
        ws = torch.empty((max(ep.ep_layout_workspace_size(cfg), 256),), dtype=torch.uint8, device="cuda")
        ep.ep_layout(cfg, idx, ref["expert_count"], ref["expert_offset"], ref["rank_count"], ref["rank_offset"],
                     ref["slot"], ref["chunks"], ref["n_chunks"], ref["worker_begin"], ws)
        got = _outputs(ep, cfg)
        rc = _static_call(ep, cfg, idx, got)
        assert rc == ep.EP_OK, f"call {call}: {ep.ep_status_string(rc)}"
        torch.cuda.synchronize()
        n = int(ref["n_chunks"].item())
        assert int(got["n_chunks"].item()) == n
        for key in ("expert_count", "expert_offset", "rank_count", "rank_offset", "slot", "worker_begin"):
            assert torch.equal(got[key], ref[key]), f"call {call}: {key} differs"
        assert torch.equal(got["chunks"][:n], ref["chunks"][:n]), f"call {call}: chunk table differs"
        # and the slots are a permutation of the send rows
        s = np.sort(got["slot"].cpu().numpy().ravel())
        assert np.array_equal(s, np.arange(w.T * w.k))


def test_static_layout_rejects_shapes_beyond_its_array(ep):
    # E = 1024 experts need 4 KiB of scratch per 256 tokens: 1 MiB covers T <= 65536
    w = ep_synth.Workload("big", T=65536 + 256, H=64, E=1024, R=8, k=2, num_workers=8)
    cfg = ep.EpConfig.from_workload(w)
    assert ep.ep_layout_workspace_size(cfg) > ep.EP_LAYOUT_STATIC_SCRATCH_BYTES
    o = _outputs(ep, ep.EpConfig.from_workload(w.with_(T=1)))
    idx = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    assert _static_call(ep, cfg, idx, o) == ep.EP_ERR_CAPACITY
    ok = ep.EpConfig.from_workload(w.with_(T=65536))
    assert ep.ep_layout_workspace_size(ok) <= ep.EP_LAYOUT_STATIC_SCRATCH_BYTES
