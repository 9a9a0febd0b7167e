"""CPU oracle for the MoE route -> layout -> dispatch -> combine path.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm may import this package. The product
path (``combine_router_softmax_gb300``) never imports it and shares no code
with it.

The arithmetic lives in ``ep_oracle.c`` (plain single-threaded C, fp64 except
for the fp32 combine the path fixes); this module only builds that file with
gcc and marshals numpy arrays through ctypes. Each wrapper names the C function
whose comment cites the passage it follows.

Parity status of each function (what pins it is listed in the tests):
  route     pinned (brute-force sort, full-softmax and equal-logit cases)
  layout    pinned (brute-force counting, stable-sort special case, invariants)
  schedule  pinned (hand-enumerated tables, tiling and balance invariants)
  dispatch  pinned (row-permutation and provenance invariants)
  combine   pinned (exact reconstruction, dyadic-weight exactness, fp64 bound)
"""
from __future__ import annotations

import ctypes
import os
import pathlib
import subprocess
import threading

import numpy as np

_HERE = pathlib.Path(__file__).resolve().parent
SOURCE = _HERE / "ep_oracle.c"
DEFAULT_LIB = _HERE / "libep_oracle.so"
# ISO C mode and no contraction: gcc must not fuse a*b+c on its own (it does by
# default on aarch64 in GNU mode); the only fused multiply-adds are the explicit
# fmaf calls of the combine.
CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall"]

_lock = threading.Lock()


class OracleError(RuntimeError):
    pass


def build(source: os.PathLike = SOURCE, out: os.PathLike = DEFAULT_LIB, force: bool = False) -> pathlib.Path:
    """Compile the oracle with gcc (idempotent unless ``force``)."""
    source, out = pathlib.Path(source), pathlib.Path(out)
    with _lock:
        if not force and out.exists() and out.stat().st_mtime >= source.stat().st_mtime:
            return out
        tmp = out.with_name(out.name + f".tmp{os.getpid()}")
        cmd = ["gcc", *CFLAGS, str(source), "-o", str(tmp), "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise OracleError(f"oracle build failed: {' '.join(cmd)}\n{r.stderr}")
        os.replace(tmp, out)
    return out


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """ctypes handle on one build of ``ep_oracle.c``."""

    def __init__(self, lib_path: os.PathLike | None = None):
        path = pathlib.Path(lib_path) if lib_path is not None else build()
        self.lib = ctypes.CDLL(str(path))
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        P = ctypes.POINTER
        L = self.lib
        L.orc_route.argtypes = [i64, i32, i32, i32, i32, i32, P(ctypes.c_float), P(i32), P(ctypes.c_double)]
        L.orc_layout.argtypes = [i64, i32, i32, i32, P(i32), P(i32), P(i32), P(i32), P(i32), P(i32)]
        L.orc_schedule.argtypes = [i32, i32, i32, i32, i32, P(i32), P(i32), i32, P(i32), P(i32)]
        L.orc_dispatch.argtypes = [i64, i32, i32, P(ctypes.c_uint16), P(i32), P(ctypes.c_uint16), P(i32)]
        L.orc_combine.argtypes = [i64, i32, i32, P(ctypes.c_uint16), P(i32), P(ctypes.c_float), P(ctypes.c_uint16)]
        L.orc_expert_scale.argtypes = [i64, i32, i32, P(i32), i32, P(ctypes.c_uint16), P(ctypes.c_uint16)]
        L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        L.orc_f32_to_bf16.restype = ctypes.c_uint16
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f32.restype = ctypes.c_float
        L.orc_tff_encode.argtypes = [i64, i64, P(ctypes.c_uint8), ctypes.c_uint32, P(ctypes.c_uint8)]
        L.orc_tff_decode.argtypes = [i64, i64, P(ctypes.c_uint8), ctypes.c_uint32, P(ctypes.c_uint8), P(i64)]
        L.orc_tff_blocks_per_row.argtypes = [i64]
        L.orc_tff_blocks_per_row.restype = i64
        for f in ("orc_route", "orc_layout", "orc_schedule", "orc_dispatch", "orc_combine", "orc_expert_scale",
                  "orc_tff_encode", "orc_tff_decode"):
            getattr(L, f).restype = ctypes.c_int

    @staticmethod
    def _check(rc: int, what: str):
        if rc != 0:
            raise OracleError(f"{what} returned {rc}")

    # -- route (orc_route) -------------------------------------------------
    def route(self, logits: np.ndarray, k: int, n_groups: int = 1, topk_groups: int = 1,
              renormalize: int = 1):
        """idx int32 [T, k], w float64 [T, k] for fp32 logits [T, E]."""
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        T, E = logits.shape
        idx = np.zeros((T, k), dtype=np.int32)
        w = np.zeros((T, k), dtype=np.float64)
        self._check(self.lib.orc_route(T, E, k, n_groups, topk_groups, renormalize,
                                       _ptr(logits, ctypes.c_float), _ptr(idx, ctypes.c_int32),
                                       _ptr(w, ctypes.c_double)), "orc_route")
        return idx, w

    # -- layout (orc_layout) -----------------------------------------------
    def layout(self, idx: np.ndarray, E: int, R: int) -> dict:
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        T, k = idx.shape
        out = {
            "expert_count": np.zeros(E, np.int32), "expert_offset": np.zeros(E + 1, np.int32),
            "rank_count": np.zeros(R, np.int32), "rank_offset": np.zeros(R + 1, np.int32),
            "slot": np.zeros((T, k), np.int32),
        }
        self._check(self.lib.orc_layout(T, E, R, k, _ptr(idx, ctypes.c_int32),
                                        *(_ptr(out[n], ctypes.c_int32) for n in
                                          ("expert_count", "expert_offset", "rank_count", "rank_offset", "slot"))),
                    "orc_layout")
        return out

    # -- schedule (orc_schedule) -------------------------------------------
    def schedule(self, rank_offset: np.ndarray, ranks_per_node: int, self_rank: int, W: int,
                 ranks_per_pod: int = 0):
        """(chunks int32 [n, 5], worker_begin int32 [W + 1])."""
        rank_offset = np.ascontiguousarray(rank_offset, dtype=np.int32)
        R = rank_offset.shape[0] - 1
        cap = 3 * W + R
        chunks = np.zeros((cap, 5), np.int32)
        wb = np.zeros(W + 1, np.int32)
        n = ctypes.c_int32(0)
        self._check(self.lib.orc_schedule(R, ranks_per_node, ranks_per_pod, self_rank, W,
                                          _ptr(rank_offset, ctypes.c_int32),
                                          _ptr(chunks, ctypes.c_int32), cap, ctypes.byref(n),
                                          _ptr(wb, ctypes.c_int32)), "orc_schedule")
        return chunks[:n.value].copy(), wb

    # -- dispatch (orc_dispatch) -------------------------------------------
    def dispatch(self, x_bits: np.ndarray, slot: np.ndarray):
        """(send bf16 bits [T*k, H], meta int32 [T*k])."""
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
        slot = np.ascontiguousarray(slot, dtype=np.int32)
        T, H = x_bits.shape
        k = slot.shape[1]
        send = np.zeros((T * k, H), np.uint16)
        meta = np.full(T * k, -1, np.int32)
        self._check(self.lib.orc_dispatch(T, H, k, _ptr(x_bits, ctypes.c_uint16), _ptr(slot, ctypes.c_int32),
                                          _ptr(send, ctypes.c_uint16), _ptr(meta, ctypes.c_int32)), "orc_dispatch")
        return send, meta

    # -- combine (orc_combine) ---------------------------------------------
    def combine(self, y_bits: np.ndarray, slot: np.ndarray, w32: np.ndarray) -> np.ndarray:
        """out bf16 bits [T, H] from expert rows y [T*k, H] in slot order."""
        y_bits = np.ascontiguousarray(y_bits, dtype=np.uint16)
        slot = np.ascontiguousarray(slot, dtype=np.int32)
        w32 = np.ascontiguousarray(w32, dtype=np.float32)
        T, k = slot.shape
        H = y_bits.shape[1]
        out = np.zeros((T, H), np.uint16)
        self._check(self.lib.orc_combine(T, H, k, _ptr(y_bits, ctypes.c_uint16), _ptr(slot, ctypes.c_int32),
                                         _ptr(w32, ctypes.c_float), _ptr(out, ctypes.c_uint16)), "orc_combine")
        return out

    # -- synthetic expert of the harness (orc_expert_scale) -----------------
    def expert(self, send_bits: np.ndarray, expert_offset: np.ndarray, E: int, identity: bool = False):
        send_bits = np.ascontiguousarray(send_bits, dtype=np.uint16)
        expert_offset = np.ascontiguousarray(expert_offset, dtype=np.int32)
        rows, H = send_bits.shape
        y = np.zeros_like(send_bits)
        self._check(self.lib.orc_expert_scale(rows, H, E, _ptr(expert_offset, ctypes.c_int32), int(identity),
                                              _ptr(send_bits, ctypes.c_uint16), _ptr(y, ctypes.c_uint16)),
                    "orc_expert_scale")
        return y

    # -- Token-Flag Fusion block codec (orc_tff_encode / orc_tff_decode) ----
    def tff_blocks_per_row(self, row_bytes: int) -> int:
        return int(self.lib.orc_tff_blocks_per_row(row_bytes))

    def tff_encode(self, rows_u8: np.ndarray, epoch: int) -> np.ndarray:
        """rows uint8 [R, row_bytes] -> framed uint8 [R, blocks * 512]."""
        rows_u8 = np.ascontiguousarray(rows_u8, dtype=np.uint8)
        R, nbytes = rows_u8.shape
        framed = np.full((R, self.tff_blocks_per_row(nbytes) * 512), 0xAB, np.uint8)
        self._check(self.lib.orc_tff_encode(R, nbytes, _ptr(rows_u8, ctypes.c_uint8), epoch & 0xFFFFFFFF,
                                            _ptr(framed, ctypes.c_uint8)), "orc_tff_encode")
        return framed

    def tff_decode(self, framed: np.ndarray, row_bytes: int, epoch: int, out: np.ndarray | None = None):
        """framed uint8 [R, blocks * 512] -> (rows uint8 [R, row_bytes], bad block count)."""
        framed = np.ascontiguousarray(framed, dtype=np.uint8)
        R = framed.shape[0]
        out = np.zeros((R, row_bytes), np.uint8) if out is None else np.ascontiguousarray(out, dtype=np.uint8)
        bad = ctypes.c_int64(0)
        self._check(self.lib.orc_tff_decode(R, row_bytes, _ptr(framed, ctypes.c_uint8), epoch & 0xFFFFFFFF,
                                            _ptr(out, ctypes.c_uint8), ctypes.byref(bad)), "orc_tff_decode")
        return out, bad.value

    def f32_to_bf16(self, f: float) -> int:
        return int(self.lib.orc_f32_to_bf16(ctypes.c_float(f)))

    def bf16_to_f32(self, b: int) -> float:
        return float(self.lib.orc_bf16_to_f32(ctypes.c_uint16(b)))

    # -- the whole path on one workload ------------------------------------
    def run_path(self, logits, x_bits, *, E, R, k, n_groups=1, topk_groups=1, renormalize=1,
                 ranks_per_node=16, self_rank=0, W=152, identity_expert=False, ranks_per_pod=0) -> dict:
        """route -> layout -> schedule -> dispatch -> expert -> combine, all on the CPU."""
        idx, w = self.route(logits, k, n_groups, topk_groups, renormalize)
        lay = self.layout(idx, E, R)
        chunks, wb = self.schedule(lay["rank_offset"], ranks_per_node, self_rank, W, ranks_per_pod)
        send, meta = self.dispatch(x_bits, lay["slot"])
        y = self.expert(send, lay["expert_offset"], E, identity=identity_expert)
        w32 = w.astype(np.float32)
        out = self.combine(y, lay["slot"], w32)
        return dict(idx=idx, w=w, w32=w32, chunks=chunks, worker_begin=wb, send=send, meta=meta, y=y,
                    out=out, **lay)


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from ``ep_oracle.c`` in this directory (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
