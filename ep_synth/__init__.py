"""Seeded synthetic inputs for the MoE route -> layout -> dispatch -> combine path.

This module is shared by the tests, the benchmark and the smoke check. It holds
the *input recipe* only: the counter-based random streams, the normal and Zipf
draws and the workload catalogue. It does no routing, layout, dispatch or
combine arithmetic, so both the CPU oracle and the CUDA path can be fed the
same bytes without either depending on the other.

Random numbers
--------------
Every tensor has its own stream ``(seed, tensor_id)``. Element ``i`` of a
stream is the SplitMix64 output for counter ``i``: the generator state is
``base + (i + 1) * 0x9E3779B97F4A7C15`` with ``base`` itself a SplitMix64 mix
of ``seed ^ (tensor_id << 32)``, and the output is the SplitMix64 finaliser of
that state (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014; constants as published by Vigna). Because element
``i`` depends only on ``i``, a workload with ``T`` tokens is a prefix of the
same workload with more tokens, which the CPU baseline's token samples use.

Normals come from the Box-Muller transform in float64 (two uniforms per pair,
both outputs used), then are cast to float32; bf16 activations are the
round-to-nearest-even bf16 of that float32.
"""
from __future__ import annotations

import math

import numpy as np

from .configs import CONFIGS, Workload, get_workload, sweep_workloads  # noqa: F401

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22  # elements generated per numpy pass (bounds host memory)

TENSOR_LOGITS = 1
TENSOR_X = 2
TENSOR_WEIGHTS = 3
TENSOR_ROWS = 4


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _stream_base(seed: int, tensor_id: int) -> np.uint64:
    s = np.array([(seed ^ (tensor_id << 32)) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return _mix(s)[0]


def uint64_stream(seed: int, tensor_id: int, n: int, offset: int = 0) -> np.ndarray:
    """``n`` consecutive SplitMix64 outputs of stream ``(seed, tensor_id)``."""
    base = _stream_base(seed, tensor_id)
    ctr = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = base + ctr * _GOLDEN
    return _mix(state)


def uniform_f64(seed: int, tensor_id: int, n: int, offset: int = 0) -> np.ndarray:
    """Uniforms in [0, 1) with 53 random bits."""
    return (uint64_stream(seed, tensor_id, n, offset) >> np.uint64(11)).astype(np.float64) * 2.0**-53


def _normal_chunk(out: np.ndarray, seed: int, tensor_id: int, pos: int, m: int, offset: int) -> None:
    g0 = offset + pos  # global index of the first normal in this chunk
    p0, p1 = g0 // 2, (g0 + m + 1) // 2  # pair range covering [g0, g0 + m)
    u = uint64_stream(seed, tensor_id, 2 * (p1 - p0), 2 * p0)
    u1 = ((u[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0**-53  # (0, 1]
    u2 = (u[1::2] >> np.uint64(11)).astype(np.float64) * 2.0**-53  # [0, 1)
    r = np.sqrt(-2.0 * np.log(u1))
    th = 2.0 * math.pi * u2
    pair = np.empty(2 * (p1 - p0), dtype=np.float64)
    pair[0::2] = r * np.cos(th)
    pair[1::2] = r * np.sin(th)
    s = g0 - 2 * p0
    out[pos:pos + m] = pair[s:s + m]


def normal_f64(seed: int, tensor_id: int, n: int, offset: int = 0) -> np.ndarray:
    """``n`` standard normals (Box-Muller), element ``i`` fixed by ``offset + i``.

    Chunks are independent (each element depends only on its index), so large
    draws are spread over a thread pool; numpy releases the GIL in its array
    loops. The result does not depend on the number of threads."""
    out = np.empty(n, dtype=np.float64)
    starts = list(range(0, n, _CHUNK))
    if len(starts) <= 1:
        for pos in starts:
            _normal_chunk(out, seed, tensor_id, pos, min(_CHUNK, n - pos), offset)
        return out
    import concurrent.futures as cf
    import os

    workers = min(len(starts), os.cpu_count() or 1, 16)
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(lambda pos: _normal_chunk(out, seed, tensor_id, pos, min(_CHUNK, n - pos), offset), starts))
    return out


def zipf_log_bias(E: int, s: float) -> np.ndarray:
    """ln p_e with p_e proportional to (e + 1)^-s: expert 0 is the most popular."""
    logw = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    return logw - np.log(np.exp(logw).sum())


def gate_logits(seed: int, T: int, E: int, zipf_s: float | None = None, t0: int = 0) -> np.ndarray:
    """fp32 gate logits [T, E]: N(0, 1), plus ln p_e for a Zipf(s) expert popularity.

    ``t0`` selects tokens ``t0 .. t0+T-1`` of the same stream.
    """
    z = normal_f64(seed, TENSOR_LOGITS, T * E, offset=t0 * E).reshape(T, E)
    if zipf_s is not None:
        z = z + zipf_log_bias(E, zipf_s)[None, :]
    return z.astype(np.float32)


def hidden_bf16_bits(seed: int, T: int, H: int, t0: int = 0) -> np.ndarray:
    """Token activations x [T, H] as bf16 bit patterns (uint16), N(0, 1) rounded RNE."""
    import torch

    f32 = normal_f64(seed, TENSOR_X, T * H, offset=t0 * H).astype(np.float32)
    bits = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return bits.reshape(T, H)


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """RNE bf16 bit patterns of a float32 array (input-recipe helper, via torch)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact float32 values of bf16 bit patterns."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def random_rows_bf16_bits(seed: int, n_rows: int, H: int, tensor_id: int = TENSOR_ROWS) -> np.ndarray:
    """Arbitrary bf16 rows (N(0,1)) for combine tests that need y unrelated to x."""
    f32 = normal_f64(seed, tensor_id, n_rows * H).astype(np.float32)
    return bf16_bits_from_f32(f32).reshape(n_rows, H)


def random_topk_weights(seed: int, T: int, k: int) -> np.ndarray:
    """Positive fp32 weights [T, k] (uniform in (0, 1]) for combine-only tests."""
    u = uniform_f64(seed, TENSOR_WEIGHTS, T * k)
    return (1.0 - u).astype(np.float32).reshape(T, k)
