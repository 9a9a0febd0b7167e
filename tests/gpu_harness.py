"""Test harness around the CUDA path: device transfers, the synthetic expert and
comparison helpers. The expert (an FFN in a real MoE layer) is not part of the
library; here it is a torch op on the GPU that scales each send row by
(e + 1) / E, e the expert owning the row, or the identity."""
from __future__ import annotations

import numpy as np
import pytest
import torch


def require_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def bf16_to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def bf16_from_dev(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def synthetic_expert(send: torch.Tensor, expert_offset: torch.Tensor, E: int, identity: bool = False,
                     out: torch.Tensor | None = None) -> torch.Tensor:
    """y[s] = bf16(float(send[s]) * ((e + 1) / E)) with e the expert owning row s."""
    if identity:
        y = send.clone() if out is None else out.copy_(send)
        return y
    rows = torch.arange(send.shape[0], device=send.device, dtype=torch.int32)
    e = torch.searchsorted(expert_offset, rows, right=True) - 1
    scale = (e + 1).to(torch.float32) / float(E)
    y = (send.float() * scale[:, None]).to(torch.bfloat16)
    if out is not None:
        out.copy_(y)
        return out
    return y


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in representable bf16 steps (signed-magnitude mapped to an ordered line)."""
    def ordered(b):
        b = b.astype(np.int32)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def route_weight_rtol(logits: np.ndarray, idx: np.ndarray, renormalize: int) -> np.ndarray:
    """Per-token relative tolerance of the fp32 GPU weights against the fp64 oracle.

    Derived from the fp32 arithmetic (see the parity test docstring):
      d = fl(l - l_max) carries <= 2^-24 |d| absolute error -> <= 2^-24 D relative after exp,
      expf <= 2 ulp (2^-22 relative), the warp-tree sum of positive terms <= (depth) 2^-24,
      the division 2^-24; with a 1.5x margin.
    """
    T, E = logits.shape
    lmax = logits.max(axis=1).astype(np.float64)
    sel = np.take_along_axis(logits, idx, axis=1).astype(np.float64)
    d_sel = np.abs(sel - lmax[:, None]).max(axis=1)
    u = 2.0**-24
    if renormalize:
        bound = 2 * (d_sel * u + 4 * u) + 6 * u
    else:
        d_all = np.abs(logits.astype(np.float64) - lmax[:, None]).max(axis=1)
        vpl = (E + 31) // 32
        bound = (d_sel * u + 4 * u) + (d_all * u + 4 * u) + (vpl + 4) * u + u
    return 1.5 * bound
