"""Token-Flag Fusion block codec (GPU): ep_tff_encode / ep_tff_decode against
the oracle's codec, byte for byte (metadata, payload and zero fill), and the
rejection of stale blocks. The rows encoded are the send buffer the oracle's
dispatch produces for the workload."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ep_synth
from gpu_harness import bf16_to_dev, require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    require_cuda()
    import combine_router_softmax_gb300 as m

    return m


def send_rows(orc, w):
    logits = ep_synth.gate_logits(w.seed, w.T, w.E, w.zipf_s)
    x = ep_synth.hidden_bf16_bits(w.seed, w.T, w.H)
    idx, _ = orc.route(logits, w.k, w.n_groups, w.topk_groups, w.renormalize)
    lay = orc.layout(idx, w.E, w.R)
    send, _ = orc.dispatch(x, lay["slot"])
    return send  # uint16 bits [T k, H]


CASES = [
    ep_synth.CONFIGS["tiny"],                                   # 512-byte rows: 2 blocks, the second 32 bytes
    ep_synth.CONFIGS["decode"].with_(name="decode-T16", T=16),  # 14336-byte rows: 30 blocks, the last 416 bytes
    ep_synth.Workload("H240", T=33, H=240, E=8, R=2, k=3),       # exactly one full block
    ep_synth.Workload("H8", T=5, H=8, E=4, R=2, k=2),            # 16-byte rows
    ep_synth.Workload("H24576", T=7, H=24576, E=16, R=4, k=4),  # 48 KiB rows
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_tff_encode_decode_vs_oracle(ep, orc, w):
    cfg = ep.EpConfig.from_workload(w)
    send = send_rows(orc, w)
    rows = bf16_to_dev(send)
    nbytes = ep.ep_tff_framed_bytes(cfg)
    framed = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device="cuda")
    epoch = 0x9E3779B9
    ep.ep_tff_encode(cfg, rows, framed, epoch)
    torch.cuda.synchronize()
    ref = orc.tff_encode(send.view(np.uint8).reshape(send.shape[0], -1), epoch)
    assert np.array_equal(framed.cpu().numpy(), ref.reshape(-1)), "framed bytes differ"
    out = torch.zeros_like(rows)
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_tff_decode(cfg, framed, epoch, out, bad)
    torch.cuda.synchronize()
    assert int(bad.item()) == 0
    assert torch.equal(out.view(torch.int16), rows.view(torch.int16))


def test_tff_decode_rejects_stale_blocks(ep, orc):
    w = ep_synth.CONFIGS["decode"].with_(name="decode-T4", T=4)
    cfg = ep.EpConfig.from_workload(w)
    send = send_rows(orc, w)
    rows = bf16_to_dev(send)
    framed = torch.empty((ep.ep_tff_framed_bytes(cfg),), dtype=torch.uint8, device="cuda")
    ep.ep_tff_encode(cfg, rows, framed, 3)
    torch.cuda.synchronize()
    host = framed.cpu().numpy().copy()
    nblk = -(-w.H * 2 // 480)
    hits = [(0, 0, 0), (5, 29, 4), (17, 3, 8), (31, 10, 12)]  # (row, block, metadata byte)
    for r, b, byte in hits:
        host[(r * nblk + b) * 512 + byte] ^= 0x40
    framed.copy_(torch.from_numpy(host))
    out = torch.full_like(rows, 7.0)  # rejected blocks must leave these bytes as they are
    init_rows = out.view(torch.int16).cpu().numpy().view(np.uint8).reshape(send.shape[0], -1).copy()
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_tff_decode(cfg, framed, 3, out, bad)
    torch.cuda.synchronize()
    assert int(bad.item()) == len(hits)
    want, nbad = orc.tff_decode(host.reshape(send.shape[0], -1), w.H * 2, 3, out=init_rows)
    assert nbad == len(hits)
    got = out.view(torch.int16).cpu().numpy().view(np.uint8).reshape(send.shape[0], -1)
    assert np.array_equal(got, want)
