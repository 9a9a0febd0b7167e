"""Python binding of the GB300 MoE expert-parallel hot path (``libep_gb300.so``).

The functions here have the names of the C entry points in ``include/ep.h``
(``ep_route``, ``ep_layout``, ``ep_dispatch``, ``ep_combine`` and the size
queries) and only marshal arguments: they check that each torch tensor has
the dtype, shape and device the C ABI expects, pass raw device pointers and
the current CUDA stream, and raise :class:`EpError` on a non-zero status.
Every step of the path runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback. Importing this package loads the library and fails if it
has not been built (``python combine_router_softmax_gb300/build.py``).

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import pathlib
from dataclasses import dataclass

import torch

_PKG = pathlib.Path(__file__).resolve().parent
LIB_PATH = _PKG / "libep_gb300.so"

EP_OK, EP_ERR_INVALID_ARG, EP_ERR_UNSUPPORTED, EP_ERR_CUDA, EP_ERR_CAPACITY = range(5)

# Entry points declared in include/ep.h (checked by the ABI test).
EXPORTS = ("ep_status_string", "ep_version", "ep_device_error", "ep_step_kernel_count", "ep_fused_step_kernel_count",
           "ep_layout_workspace_size", "ep_dispatch_fused_workspace_size", "ep_schedule_capacity",
           "ep_dispatch_fused", "ep_check_bounded_wait", "ep_sentinel_arm", "ep_expert_scale",
           "ep_dispatch_expert_sp", "ep_dispatch_expert_sw", "ep_dispatch_scheduled_ctas", "ep_dispatch_scheduled",
           "ep_tff_framed_bytes", "ep_tff_encode", "ep_tff_decode",
           "ep_route", "ep_layout", "ep_dispatch", "ep_combine", "ep_layout_static")
# Size of the device array ep_layout_static uses instead of a workspace (include/ep.h).
EP_LAYOUT_STATIC_SCRATCH_BYTES = 1 << 20


class EpError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_status_string(status)}")


class EpConfig(ctypes.Structure):
    """``ep_config`` of include/ep.h."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "T", "H", "E", "R", "k", "n_groups", "topk_groups", "renormalize",
        "ranks_per_node", "self_rank", "num_workers", "ranks_per_pod")]

    @classmethod
    def make(cls, *, T, H, E, R, k, n_groups=1, topk_groups=1, renormalize=1, ranks_per_node=16,
             self_rank=0, num_workers=0, ranks_per_pod=0) -> "EpConfig":
        return cls(T, H, E, R, k, n_groups, topk_groups, renormalize, ranks_per_node, self_rank, num_workers,
                   ranks_per_pod)

    @property
    def hop_classes(self) -> int:
        return 3 if self.ranks_per_pod > 0 else 2

    @classmethod
    def from_workload(cls, w, **over) -> "EpConfig":
        kw = dict(T=w.T, H=w.H, E=w.E, R=w.R, k=w.k, n_groups=w.n_groups, topk_groups=w.topk_groups,
                  renormalize=w.renormalize, ranks_per_node=w.ranks_per_node, self_rank=w.self_rank,
                  num_workers=w.num_workers, ranks_per_pod=w.ranks_per_pod)
        kw.update(over)
        return cls.make(**kw)


class EpChunk(ctypes.Structure):
    """``ep_chunk`` of include/ep.h (5 x int32)."""
    _fields_ = [(n, ctypes.c_int32) for n in ("worker", "hop_class", "dst_rank", "row_begin", "row_count")]


def _load() -> ctypes.CDLL:
    if not LIB_PATH.exists():
        raise ImportError(
            f"{LIB_PATH.name} is not built; run `python combine_router_softmax_gb300/build.py` "
            "(nvcc for sm_103a). There is no fallback path.")
    lib = ctypes.CDLL(str(LIB_PATH))
    P, vp = ctypes.POINTER, ctypes.c_void_p
    cfgp = P(EpConfig)
    lib.ep_status_string.argtypes = [ctypes.c_int]
    lib.ep_status_string.restype = ctypes.c_char_p
    lib.ep_version.argtypes = []
    lib.ep_version.restype = ctypes.c_int
    lib.ep_device_error.argtypes = [P(ctypes.c_int32)]
    lib.ep_check_bounded_wait.argtypes = [ctypes.c_int32, vp, vp]
    lib.ep_sentinel_arm.argtypes = [cfgp, vp, vp]
    lib.ep_expert_scale.argtypes = [cfgp, vp, vp, vp, vp, vp]
    lib.ep_dispatch_expert_sp.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.ep_dispatch_expert_sw.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_uint32, vp]
    lib.ep_dispatch_scheduled_ctas.argtypes = [cfgp, P(ctypes.c_int32)]
    lib.ep_tff_framed_bytes.argtypes = [cfgp, P(ctypes.c_size_t)]
    lib.ep_tff_encode.argtypes = [cfgp, vp, vp, ctypes.c_uint32, vp]
    lib.ep_tff_decode.argtypes = [cfgp, vp, ctypes.c_uint32, vp, vp, vp]
    lib.ep_dispatch_scheduled.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.ep_step_kernel_count.argtypes = [cfgp, P(ctypes.c_int32)]
    lib.ep_fused_step_kernel_count.argtypes = [cfgp, P(ctypes.c_int32)]
    lib.ep_layout_workspace_size.argtypes = [cfgp, P(ctypes.c_size_t)]
    lib.ep_schedule_capacity.argtypes = [cfgp, P(ctypes.c_int32)]
    lib.ep_route.argtypes = [cfgp, vp, vp, vp, vp]
    lib.ep_layout.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int32, vp, vp, vp, ctypes.c_size_t, vp]
    lib.ep_layout_static.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int32, vp, vp, vp]
    lib.ep_dispatch.argtypes = [cfgp, vp, vp, vp, vp, vp]
    lib.ep_dispatch_fused_workspace_size.argtypes = [cfgp, P(ctypes.c_size_t)]
    lib.ep_dispatch_fused.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int32, vp, vp, vp, vp, vp,
                                      ctypes.c_size_t, vp]
    lib.ep_combine.argtypes = [cfgp, vp, vp, vp, vp, vp]
    for f in ("ep_dispatch_fused_workspace_size", "ep_dispatch_fused", "ep_fused_step_kernel_count",
              "ep_check_bounded_wait", "ep_sentinel_arm", "ep_expert_scale", "ep_dispatch_expert_sp",
              "ep_dispatch_scheduled_ctas", "ep_dispatch_scheduled", "ep_dispatch_expert_sw",
              "ep_tff_framed_bytes", "ep_tff_encode", "ep_tff_decode",
              "ep_device_error", "ep_step_kernel_count", "ep_layout_workspace_size", "ep_schedule_capacity", "ep_route", "ep_layout",
              "ep_dispatch", "ep_combine", "ep_layout_static"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


_lib = _load()


def _status_string(status: int) -> str:
    return _lib.ep_status_string(int(status)).decode()


def ep_status_string(status: int) -> str:
    return _status_string(status)


def ep_version() -> int:
    return int(_lib.ep_version())


def _check(status: int, what: str):
    if status != EP_OK:
        raise EpError(status, what)


def _ptr(t: torch.Tensor | None, dtype: torch.dtype, shape: tuple | None, name: str):
    """Device pointer of a contiguous CUDA tensor of the expected dtype/shape (None -> NULL)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    cur = torch.cuda.current_device()
    if t.device.index != cur:
        # the kernels run on the current device and would dereference another device's memory
        raise ValueError(f"{name}: on {t.device}, but the current device is cuda:{cur}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    elif stream.device.index != torch.cuda.current_device():
        raise ValueError(f"stream: on {stream.device}, but the current device is cuda:{torch.cuda.current_device()}")
    return ctypes.c_void_p(stream.cuda_stream)


def ep_device_error() -> int:
    """Device-side error flags of the current device (read and cleared; synchronous)."""
    v = ctypes.c_int32(0)
    _check(_lib.ep_device_error(ctypes.byref(v)), "ep_device_error")
    return int(v.value)


def ep_check_bounded_wait(max_polls: int, gave_up, stream=None) -> None:
    """Run the library's bounded-wait self-check; gave_up: int32 [1] CUDA tensor (ends at 2)."""
    _check(_lib.ep_check_bounded_wait(int(max_polls), _ptr(gave_up, torch.int32, (1,), "gave_up"), _stream(stream)),
           "ep_check_bounded_wait")


def ep_step_kernel_count(cfg: EpConfig, fused: bool = False) -> int:
    """Kernels one pass enqueues on the current device: route + layout + dispatch
    + combine, or (fused=True) dispatch_fused + combine."""
    v = ctypes.c_int32(0)
    f = _lib.ep_fused_step_kernel_count if fused else _lib.ep_step_kernel_count
    _check(f(ctypes.byref(cfg), ctypes.byref(v)), "ep_step_kernel_count")
    return int(v.value)


def ep_layout_workspace_size(cfg: EpConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.ep_layout_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "ep_layout_workspace_size")
    return int(n.value)


def ep_schedule_capacity(cfg: EpConfig) -> int:
    n = ctypes.c_int32(0)
    _check(_lib.ep_schedule_capacity(ctypes.byref(cfg), ctypes.byref(n)), "ep_schedule_capacity")
    return int(n.value)


def ep_route(cfg: EpConfig, logits, topk_idx, topk_w, stream=None) -> None:
    """logits fp32 [T, E] -> topk_idx int32 [T, k], topk_w fp32 [T, k]."""
    T, E, k = cfg.T, cfg.E, cfg.k
    _check(_lib.ep_route(ctypes.byref(cfg), _ptr(logits, torch.float32, (T, E), "logits"),
                         _ptr(topk_idx, torch.int32, (T, k), "topk_idx"),
                         _ptr(topk_w, torch.float32, (T, k), "topk_w"), _stream(stream)), "ep_route")


def ep_layout(cfg: EpConfig, topk_idx, expert_count, expert_offset, rank_count, rank_offset, slot, chunks,
              n_chunks, worker_begin, workspace, stream=None) -> None:
    """Counts, offsets, slots and chunk schedule; ``chunks`` is int32 [capacity, 5]
    (one ``ep_chunk`` per row) and ``workspace`` a uint8 tensor."""
    T, E, R, k = cfg.T, cfg.E, cfg.R, cfg.k
    if chunks.dim() != 2 or chunks.shape[1] != 5:
        raise ValueError("chunks: expected int32 [capacity, 5]")
    W = (ep_schedule_capacity(cfg) - R) // cfg.hop_classes
    if worker_begin.dim() != 1 or worker_begin.numel() < W + 1:
        raise ValueError(f"worker_begin: expected int32 [>= {W + 1}]")
    if workspace is not None and workspace.dtype != torch.uint8:
        raise TypeError("workspace: expected a uint8 tensor")
    ws_ptr = _ptr(workspace, torch.uint8, None, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() if workspace is not None else 0
    _check(_lib.ep_layout(ctypes.byref(cfg), _ptr(topk_idx, torch.int32, (T, k), "topk_idx"),
                          _ptr(expert_count, torch.int32, (E,), "expert_count"),
                          _ptr(expert_offset, torch.int32, (E + 1,), "expert_offset"),
                          _ptr(rank_count, torch.int32, (R,), "rank_count"),
                          _ptr(rank_offset, torch.int32, (R + 1,), "rank_offset"),
                          _ptr(slot, torch.int32, (T, k), "slot"),
                          _ptr(chunks, torch.int32, None, "chunks"), ctypes.c_int32(chunks.shape[0]),
                          _ptr(n_chunks, torch.int32, (1,), "n_chunks"),
                          _ptr(worker_begin, torch.int32, None, "worker_begin"),
                          ws_ptr, ctypes.c_size_t(ws_bytes), _stream(stream)), "ep_layout")


def ep_layout_static(cfg: EpConfig, topk_idx, expert_count, expert_offset, rank_count, rank_offset, slot, chunks,
                     n_chunks, worker_begin, stream=None) -> None:
    """``ep_layout`` without a workspace argument: the library's fixed device
    scratch array stands in for it (for callers that cannot allocate; see
    include/ep.h). The first call on a device should precede any stream capture."""
    T, E, R, k = cfg.T, cfg.E, cfg.R, cfg.k
    if chunks.dim() != 2 or chunks.shape[1] != 5:
        raise ValueError("chunks: expected int32 [capacity, 5]")
    W = (ep_schedule_capacity(cfg) - R) // cfg.hop_classes
    if worker_begin.dim() != 1 or worker_begin.numel() < W + 1:
        raise ValueError(f"worker_begin: expected int32 [>= {W + 1}]")
    _check(_lib.ep_layout_static(ctypes.byref(cfg), _ptr(topk_idx, torch.int32, (T, k), "topk_idx"),
                                 _ptr(expert_count, torch.int32, (E,), "expert_count"),
                                 _ptr(expert_offset, torch.int32, (E + 1,), "expert_offset"),
                                 _ptr(rank_count, torch.int32, (R,), "rank_count"),
                                 _ptr(rank_offset, torch.int32, (R + 1,), "rank_offset"),
                                 _ptr(slot, torch.int32, (T, k), "slot"),
                                 _ptr(chunks, torch.int32, None, "chunks"), ctypes.c_int32(chunks.shape[0]),
                                 _ptr(n_chunks, torch.int32, (1,), "n_chunks"),
                                 _ptr(worker_begin, torch.int32, None, "worker_begin"), _stream(stream)),
           "ep_layout_static")


def ep_dispatch_fused_workspace_size(cfg: EpConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.ep_dispatch_fused_workspace_size(ctypes.byref(cfg), ctypes.byref(n)),
           "ep_dispatch_fused_workspace_size")
    return int(n.value)


def ep_dispatch_fused(cfg: EpConfig, logits, x, topk_idx, topk_w, expert_count, expert_offset, rank_count,
                      rank_offset, slot, chunks, n_chunks, worker_begin, send, slot_meta, workspace,
                      stream=None) -> None:
    """ep_route + ep_layout + ep_dispatch in one call (same outputs)."""
    T, H, E, R, k = cfg.T, cfg.H, cfg.E, cfg.R, cfg.k
    if chunks.dim() != 2 or chunks.shape[1] != 5:
        raise ValueError("chunks: expected int32 [capacity, 5]")
    W = (ep_schedule_capacity(cfg) - R) // cfg.hop_classes
    if worker_begin.dim() != 1 or worker_begin.numel() < W + 1:
        raise ValueError(f"worker_begin: expected int32 [>= {W + 1}]")
    if workspace.dtype != torch.uint8:
        raise TypeError("workspace: expected a uint8 tensor")
    _check(_lib.ep_dispatch_fused(ctypes.byref(cfg), _ptr(logits, torch.float32, (T, E), "logits"),
                                  _ptr(x, torch.bfloat16, (T, H), "x"),
                                  _ptr(topk_idx, torch.int32, (T, k), "topk_idx"),
                                  _ptr(topk_w, torch.float32, (T, k), "topk_w"),
                                  _ptr(expert_count, torch.int32, (E,), "expert_count"),
                                  _ptr(expert_offset, torch.int32, (E + 1,), "expert_offset"),
                                  _ptr(rank_count, torch.int32, (R,), "rank_count"),
                                  _ptr(rank_offset, torch.int32, (R + 1,), "rank_offset"),
                                  _ptr(slot, torch.int32, (T, k), "slot"),
                                  _ptr(chunks, torch.int32, None, "chunks"), ctypes.c_int32(chunks.shape[0]),
                                  _ptr(n_chunks, torch.int32, (1,), "n_chunks"),
                                  _ptr(worker_begin, torch.int32, None, "worker_begin"),
                                  _ptr(send, torch.bfloat16, (T * k, H), "send"),
                                  _ptr(slot_meta, torch.int32, (T * k,), "slot_meta"),
                                  _ptr(workspace, torch.uint8, None, "workspace"), ctypes.c_size_t(workspace.numel()),
                                  _stream(stream)), "ep_dispatch_fused")


def ep_dispatch_scheduled_ctas(cfg: EpConfig) -> int:
    """CTAs of ep_dispatch_scheduled (rows of its optional cta_ns output)."""
    n = ctypes.c_int32(0)
    _check(_lib.ep_dispatch_scheduled_ctas(ctypes.byref(cfg), ctypes.byref(n)), "ep_dispatch_scheduled_ctas")
    return n.value


def ep_dispatch_scheduled(cfg: EpConfig, x, slot, chunks, n_chunks, worker_begin, send, slot_meta, cta_ns=None,
                          stream=None) -> None:
    """Dispatch pulled by the chunk schedule (same send / slot_meta as ep_dispatch)."""
    T, H, k = cfg.T, cfg.H, cfg.k
    ns = None
    if cta_ns is not None:
        ns = _ptr(cta_ns, torch.int64, (ep_dispatch_scheduled_ctas(cfg), 2), "cta_ns")
    _check(_lib.ep_dispatch_scheduled(ctypes.byref(cfg), _ptr(x, torch.bfloat16, (T, H), "x"),
                                      _ptr(slot, torch.int32, (T, k), "slot"),
                                      _ptr(chunks, torch.int32, None, "chunks"),
                                      _ptr(n_chunks, torch.int32, (1,), "n_chunks"),
                                      _ptr(worker_begin, torch.int32, None, "worker_begin"),
                                      _ptr(send, torch.bfloat16, (T * k, H), "send"),
                                      _ptr(slot_meta, torch.int32, (T * k,), "slot_meta"), ns, _stream(stream)),
           "ep_dispatch_scheduled")


EP_TFF_BLOCK_BYTES = 512


def ep_tff_framed_bytes(cfg: EpConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.ep_tff_framed_bytes(ctypes.byref(cfg), ctypes.byref(n)), "ep_tff_framed_bytes")
    return n.value


def ep_tff_encode(cfg: EpConfig, rows, framed, epoch: int, stream=None) -> None:
    """rows bf16 [T*k, H] -> framed uint8 [ep_tff_framed_bytes] of 512-byte blocks."""
    _check(_lib.ep_tff_encode(ctypes.byref(cfg), _ptr(rows, torch.bfloat16, (cfg.T * cfg.k, cfg.H), "rows"),
                              _ptr(framed, torch.uint8, (ep_tff_framed_bytes(cfg),), "framed"),
                              ctypes.c_uint32(epoch & 0xFFFFFFFF), _stream(stream)), "ep_tff_encode")


def ep_tff_decode(cfg: EpConfig, framed, epoch: int, rows, bad_blocks, stream=None) -> None:
    """framed -> rows bf16 [T*k, H]; rejected blocks are added to bad_blocks (int32 [1])."""
    _check(_lib.ep_tff_decode(ctypes.byref(cfg), _ptr(framed, torch.uint8, (ep_tff_framed_bytes(cfg),), "framed"),
                              ctypes.c_uint32(epoch & 0xFFFFFFFF),
                              _ptr(rows, torch.bfloat16, (cfg.T * cfg.k, cfg.H), "rows"),
                              _ptr(bad_blocks, torch.int32, (1,), "bad_blocks"), _stream(stream)), "ep_tff_decode")


EP_SENTINEL_BF16 = 0xFFFF


def ep_sentinel_arm(cfg: EpConfig, send, stream=None) -> None:
    """Fill send [T*k, H] with the bf16 sentinel 0xFFFF."""
    _check(_lib.ep_sentinel_arm(ctypes.byref(cfg), _ptr(send, torch.bfloat16, (cfg.T * cfg.k, cfg.H), "send"),
                                _stream(stream)), "ep_sentinel_arm")


def ep_expert_scale(cfg: EpConfig, send, expert_offset, expert_scale, y, stream=None) -> None:
    """y[s] = bf16(send[s] * expert_scale[e(s)])."""
    T, H, E, k = cfg.T, cfg.H, cfg.E, cfg.k
    _check(_lib.ep_expert_scale(ctypes.byref(cfg), _ptr(send, torch.bfloat16, (T * k, H), "send"),
                                _ptr(expert_offset, torch.int32, (E + 1,), "expert_offset"),
                                _ptr(expert_scale, torch.float32, (E,), "expert_scale"),
                                _ptr(y, torch.bfloat16, (T * k, H), "y"), _stream(stream)), "ep_expert_scale")


def ep_dispatch_expert_sp(cfg: EpConfig, x, slot, expert_offset, expert_scale, chunks, n_chunks, worker_begin,
                          send, slot_meta, y, stream=None) -> None:
    """Dispatch + scale expert in one kernel, rows handed over by sentinel polling."""
    T, H, E, k = cfg.T, cfg.H, cfg.E, cfg.k
    _check(_lib.ep_dispatch_expert_sp(ctypes.byref(cfg), _ptr(x, torch.bfloat16, (T, H), "x"),
                                      _ptr(slot, torch.int32, (T, k), "slot"),
                                      _ptr(expert_offset, torch.int32, (E + 1,), "expert_offset"),
                                      _ptr(expert_scale, torch.float32, (E,), "expert_scale"),
                                      _ptr(chunks, torch.int32, None, "chunks"),
                                      _ptr(n_chunks, torch.int32, (1,), "n_chunks"),
                                      _ptr(worker_begin, torch.int32, None, "worker_begin"),
                                      _ptr(send, torch.bfloat16, (T * k, H), "send"),
                                      _ptr(slot_meta, torch.int32, (T * k,), "slot_meta"),
                                      _ptr(y, torch.bfloat16, (T * k, H), "y"), _stream(stream)),
           "ep_dispatch_expert_sp")


def ep_dispatch_expert_sw(cfg: EpConfig, x, slot, expert_offset, expert_scale, chunks, n_chunks, worker_begin,
                          send, slot_meta, y, row_flag, epoch: int, stream=None) -> None:
    """Stop-and-wait handoff: per-row flag released after the row lands (row_flag int32 [T*k])."""
    T, H, E, k = cfg.T, cfg.H, cfg.E, cfg.k
    _check(_lib.ep_dispatch_expert_sw(ctypes.byref(cfg), _ptr(x, torch.bfloat16, (T, H), "x"),
                                      _ptr(slot, torch.int32, (T, k), "slot"),
                                      _ptr(expert_offset, torch.int32, (E + 1,), "expert_offset"),
                                      _ptr(expert_scale, torch.float32, (E,), "expert_scale"),
                                      _ptr(chunks, torch.int32, None, "chunks"),
                                      _ptr(n_chunks, torch.int32, (1,), "n_chunks"),
                                      _ptr(worker_begin, torch.int32, None, "worker_begin"),
                                      _ptr(send, torch.bfloat16, (T * k, H), "send"),
                                      _ptr(slot_meta, torch.int32, (T * k,), "slot_meta"),
                                      _ptr(y, torch.bfloat16, (T * k, H), "y"),
                                      _ptr(row_flag, torch.int32, (T * k,), "row_flag"),
                                      ctypes.c_uint32(epoch & 0xFFFFFFFF), _stream(stream)), "ep_dispatch_expert_sw")


def ep_dispatch(cfg: EpConfig, x, slot, send, slot_meta, stream=None) -> None:
    """x bf16 [T, H] -> send bf16 [T*k, H], slot_meta int32 [T*k]."""
    T, H, k = cfg.T, cfg.H, cfg.k
    _check(_lib.ep_dispatch(ctypes.byref(cfg), _ptr(x, torch.bfloat16, (T, H), "x"),
                            _ptr(slot, torch.int32, (T, k), "slot"),
                            _ptr(send, torch.bfloat16, (T * k, H), "send"),
                            _ptr(slot_meta, torch.int32, (T * k,), "slot_meta"), _stream(stream)), "ep_dispatch")


def ep_combine(cfg: EpConfig, y, slot, topk_w, out, stream=None) -> None:
    """y bf16 [T*k, H] (slot order), slot, topk_w -> out bf16 [T, H]."""
    T, H, k = cfg.T, cfg.H, cfg.k
    _check(_lib.ep_combine(ctypes.byref(cfg), _ptr(y, torch.bfloat16, (T * k, H), "y"),
                           _ptr(slot, torch.int32, (T, k), "slot"),
                           _ptr(topk_w, torch.float32, (T, k), "topk_w"),
                           _ptr(out, torch.bfloat16, (T, H), "out"), _stream(stream)), "ep_combine")


@dataclass
class LayerBuffers:
    """Every device buffer one layer of the path reads or writes (allocated by torch)."""
    cfg: EpConfig
    logits: torch.Tensor
    x: torch.Tensor
    topk_idx: torch.Tensor
    topk_w: torch.Tensor
    expert_count: torch.Tensor
    expert_offset: torch.Tensor
    rank_count: torch.Tensor
    rank_offset: torch.Tensor
    slot: torch.Tensor
    chunks: torch.Tensor
    n_chunks: torch.Tensor
    worker_begin: torch.Tensor
    workspace: torch.Tensor
    send: torch.Tensor
    slot_meta: torch.Tensor
    y: torch.Tensor
    out: torch.Tensor

    @classmethod
    def allocate(cls, cfg: EpConfig, device="cuda", y_is_send: bool = False) -> "LayerBuffers":
        T, H, E, R, k = cfg.T, cfg.H, cfg.E, cfg.R, cfg.k
        cap = ep_schedule_capacity(cfg)
        W = (cap - R) // cfg.hop_classes
        i32 = dict(dtype=torch.int32, device=device)
        send = torch.empty((T * k, H), dtype=torch.bfloat16, device=device)
        return cls(
            cfg=cfg,
            logits=torch.empty((T, E), dtype=torch.float32, device=device),
            x=torch.empty((T, H), dtype=torch.bfloat16, device=device),
            topk_idx=torch.empty((T, k), **i32),
            topk_w=torch.empty((T, k), dtype=torch.float32, device=device),
            expert_count=torch.empty((E,), **i32),
            expert_offset=torch.empty((E + 1,), **i32),
            rank_count=torch.empty((R,), **i32),
            rank_offset=torch.empty((R + 1,), **i32),
            slot=torch.empty((T, k), **i32),
            chunks=torch.empty((cap, 5), **i32),
            n_chunks=torch.empty((1,), **i32),
            worker_begin=torch.empty((W + 1,), **i32),
            workspace=torch.empty((max(ep_layout_workspace_size(cfg), ep_dispatch_fused_workspace_size(cfg), 256),),
                                  dtype=torch.uint8, device=device),
            send=send,
            slot_meta=torch.empty((T * k,), **i32),
            y=send if y_is_send else torch.empty((T * k, H), dtype=torch.bfloat16, device=device),
            out=torch.empty((T, H), dtype=torch.bfloat16, device=device),
        )

    def route(self, stream=None):
        ep_route(self.cfg, self.logits, self.topk_idx, self.topk_w, stream)

    def layout(self, stream=None):
        ep_layout(self.cfg, self.topk_idx, self.expert_count, self.expert_offset, self.rank_count,
                  self.rank_offset, self.slot, self.chunks, self.n_chunks, self.worker_begin, self.workspace,
                  stream)

    def dispatch(self, stream=None):
        ep_dispatch(self.cfg, self.x, self.slot, self.send, self.slot_meta, stream)

    def combine(self, stream=None):
        ep_combine(self.cfg, self.y, self.slot, self.topk_w, self.out, stream)

    def dispatch_fused(self, stream=None):
        """route + layout + dispatch in one call."""
        ep_dispatch_fused(self.cfg, self.logits, self.x, self.topk_idx, self.topk_w, self.expert_count,
                          self.expert_offset, self.rank_count, self.rank_offset, self.slot, self.chunks,
                          self.n_chunks, self.worker_begin, self.send, self.slot_meta, self.workspace, stream)

    def dispatch_scheduled(self, cta_ns=None, stream=None):
        ep_dispatch_scheduled(self.cfg, self.x, self.slot, self.chunks, self.n_chunks, self.worker_begin, self.send,
                              self.slot_meta, cta_ns, stream)

    def sentinel_arm(self, stream=None):
        ep_sentinel_arm(self.cfg, self.send, stream)

    def expert_scale(self, expert_scale, stream=None):
        ep_expert_scale(self.cfg, self.send, self.expert_offset, expert_scale, self.y, stream)

    def dispatch_expert_sp(self, expert_scale, stream=None):
        """dispatch + per-expert scale in one kernel; send must be armed."""
        ep_dispatch_expert_sp(self.cfg, self.x, self.slot, self.expert_offset, expert_scale, self.chunks,
                              self.n_chunks, self.worker_begin, self.send, self.slot_meta, self.y, stream)

    def dispatch_expert_sw(self, expert_scale, row_flag, epoch: int, stream=None):
        """dispatch + per-expert scale in one kernel, rows handed over by per-row flags."""
        ep_dispatch_expert_sw(self.cfg, self.x, self.slot, self.expert_offset, expert_scale, self.chunks,
                              self.n_chunks, self.worker_begin, self.send, self.slot_meta, self.y, row_flag, epoch,
                              stream)

    def bind(self, stream=None) -> "BoundLayer":
        """Pre-marshalled C calls on this layer's buffers (same entry points,
        argument checks done once), for launch-rate-sensitive loops."""
        return BoundLayer(self, stream)

    def step(self, stream=None):
        """route -> layout -> dispatch -> combine (the expert between dispatch and
        combine is the caller's: ``y`` is whatever it holds)."""
        self.route(stream)
        self.layout(stream)
        self.dispatch(stream)
        self.combine(stream)


class BoundLayer:
    """The four C entry points with their ctypes arguments built once.

    Shapes and dtypes are checked when binding (through the same helpers as the
    functions above); each call then goes straight to the C ABI and raises
    :class:`EpError` on a non-zero status.
    """

    def __init__(self, b: LayerBuffers, stream=None):
        cfg = b.cfg
        T, H, E, R, k = cfg.T, cfg.H, cfg.E, cfg.R, cfg.k
        self._cfg = ctypes.byref(cfg)
        self._keep = (b, cfg)
        st = _stream(stream)
        cap = ep_schedule_capacity(cfg)
        W = (cap - R) // cfg.hop_classes
        if b.chunks.shape[0] < cap or b.worker_begin.numel() < W + 1:
            raise ValueError("chunk table or worker_begin too small")
        self._route = (self._cfg, _ptr(b.logits, torch.float32, (T, E), "logits"),
                       _ptr(b.topk_idx, torch.int32, (T, k), "topk_idx"),
                       _ptr(b.topk_w, torch.float32, (T, k), "topk_w"), st)
        self._layout = (self._cfg, _ptr(b.topk_idx, torch.int32, (T, k), "topk_idx"),
                        _ptr(b.expert_count, torch.int32, (E,), "expert_count"),
                        _ptr(b.expert_offset, torch.int32, (E + 1,), "expert_offset"),
                        _ptr(b.rank_count, torch.int32, (R,), "rank_count"),
                        _ptr(b.rank_offset, torch.int32, (R + 1,), "rank_offset"),
                        _ptr(b.slot, torch.int32, (T, k), "slot"),
                        _ptr(b.chunks, torch.int32, None, "chunks"), ctypes.c_int32(b.chunks.shape[0]),
                        _ptr(b.n_chunks, torch.int32, (1,), "n_chunks"),
                        _ptr(b.worker_begin, torch.int32, None, "worker_begin"),
                        _ptr(b.workspace, torch.uint8, None, "workspace"), ctypes.c_size_t(b.workspace.numel()), st)
        self._dispatch = (self._cfg, _ptr(b.x, torch.bfloat16, (T, H), "x"), _ptr(b.slot, torch.int32, (T, k), "slot"),
                          _ptr(b.send, torch.bfloat16, (T * k, H), "send"),
                          _ptr(b.slot_meta, torch.int32, (T * k,), "slot_meta"), st)
        self._combine = (self._cfg, _ptr(b.y, torch.bfloat16, (T * k, H), "y"), _ptr(b.slot, torch.int32, (T, k), "slot"),
                         _ptr(b.topk_w, torch.float32, (T, k), "topk_w"),
                         _ptr(b.out, torch.bfloat16, (T, H), "out"), st)
        self._fused = (self._cfg, self._route[1], self._dispatch[1], self._route[2], self._route[3],
                       *self._layout[2:7], self._layout[7], self._layout[8], self._layout[9], self._layout[10],
                       self._dispatch[3], self._dispatch[4], self._layout[11], self._layout[12], st)
        self._f = (_lib.ep_route, _lib.ep_layout, _lib.ep_dispatch, _lib.ep_combine, _lib.ep_dispatch_fused)

    def route(self):
        rc = self._f[0](*self._route)
        if rc:
            raise EpError(rc, "ep_route")

    def layout(self):
        rc = self._f[1](*self._layout)
        if rc:
            raise EpError(rc, "ep_layout")

    def dispatch(self):
        rc = self._f[2](*self._dispatch)
        if rc:
            raise EpError(rc, "ep_dispatch")

    def combine(self):
        rc = self._f[3](*self._combine)
        if rc:
            raise EpError(rc, "ep_combine")

    def dispatch_fused(self):
        rc = self._f[4](*self._fused)
        if rc:
            raise EpError(rc, "ep_dispatch_fused")
