"""Expert-parallel exchange of one MoE layer across processes (one GPU each).

The UBEP article's subject is this exchange: every token row goes to the
device that holds each expert chosen for it, and the experts' outputs come back
to the token's device in the Combine step (opening section; "Communication-Level
Performance"). On one GPU the library models the R expert-parallel ranks as
contiguous partitions of one send buffer: ep_layout orders the rows by
(destination rank, expert, source token), so rank r's rows are the segment
[rank_offset[r], rank_offset[r + 1]). Across P processes, process p holds the
experts of virtual ranks [p R / P, (p + 1) R / P) -- E / P consecutive experts
-- and the exchange is:

1. counts: every process sends each process the counts of that process's
   experts in its own send buffer (an all-to-all of E / P ints per pair);
2. rows: one all-to-all-v of the send buffer's process segments; process p
   receives, from each source s in turn, the rows s holds for p's experts,
   ordered by expert and then by source token (the order ep_layout gave them);
3. expert: the caller runs its experts on the received rows
   (``Received.expert_ids`` names the expert of every row);
4. reverse: one all-to-all-v of the expert outputs back along the same
   segments, which puts every output row into the source's ``y`` at the
   send-buffer row it was dispatched from; ep_combine then reduces them.

Nothing here computes: the two all-to-alls move bytes only, through
torch.distributed (NCCL between GPUs, gloo between CPU processes in the
tests). The split sizes of an all-to-all-v are host integers, so step 1 ends
with a device-to-host copy of the counts (one synchronisation per layer).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch
import torch.distributed as dist


@dataclass
class Received:
    """What one process receives in the dispatch exchange."""

    rows: torch.Tensor          # bf16 [n_recv, H]: by source process, then expert, then source token
    counts: torch.Tensor        # int32 [P, E / P]: rows of each of this process's experts from each source
    send_splits: list           # rows this process sent to each process (its send-buffer segments)
    recv_splits: list           # rows it received from each process
    first_expert: int           # global id of this process's first expert

    @property
    def expert_ids(self) -> torch.Tensor:
        """Global expert id of every received row (int64 [n_recv])."""
        P, Ep = self.counts.shape
        ids = self.first_expert + torch.arange(Ep, device=self.counts.device, dtype=torch.int64).repeat(P)
        return torch.repeat_interleave(ids, self.counts.reshape(-1).to(torch.int64))


def _as_words(rows: torch.Tensor) -> torch.Tensor:
    """bf16 [n, H] viewed as int32 [n, H / 2]: the collective moves the bytes as they are."""
    return rows.view(torch.int32)


class EpExchange:
    """The dispatch and combine exchanges of one layer shape over a process group.

    ``cfg.R`` must be a multiple of the group size: each process holds R / P
    virtual ranks, i.e. E / P consecutive experts.
    """

    def __init__(self, cfg, group=None, world: int | None = None, rank: int | None = None):
        self.cfg = cfg
        self.group = group
        self.world = dist.get_world_size(group) if world is None else world
        self.rank = dist.get_rank(group) if rank is None else rank
        if cfg.R % self.world != 0:
            raise ValueError(f"R = {cfg.R} virtual ranks cannot be split over {self.world} processes")
        self.experts_per_proc = cfg.E // self.world
        self.ranks_per_proc = cfg.R // self.world

    def send_splits(self, rank_offset: torch.Tensor) -> list:
        """Rows of the send buffer bound for each process (host ints)."""
        bounds = rank_offset[::self.ranks_per_proc].to("cpu", torch.int64)
        return (bounds[1:] - bounds[:-1]).tolist()

    def dispatch(self, send: torch.Tensor, expert_count: torch.Tensor, rank_offset: torch.Tensor) -> Received:
        """Steps 1 and 2: exchange the counts, then the rows (send: [T k, H] bf16
        in ep_layout's order; expert_count [E], rank_offset [R + 1] as ep_layout
        wrote them)."""
        P, Ep = self.world, self.experts_per_proc
        counts_out = expert_count.to(torch.int32).reshape(P, Ep).contiguous()
        counts_in = torch.empty_like(counts_out)
        dist.all_to_all_single(counts_in, counts_out, group=self.group)
        send_splits = self.send_splits(rank_offset)
        recv_splits = counts_in.sum(dim=1).to("cpu", torch.int64).tolist()
        H = send.shape[1]
        rows = torch.empty((sum(recv_splits), H), dtype=send.dtype, device=send.device)
        n_send = sum(send_splits)
        dist.all_to_all_single(_as_words(rows), _as_words(send[:n_send]), recv_splits, send_splits, group=self.group)
        return Received(rows=rows, counts=counts_in, send_splits=send_splits, recv_splits=recv_splits,
                        first_expert=self.rank * Ep)

    def combine(self, y_recv: torch.Tensor, received: Received, y: torch.Tensor) -> torch.Tensor:
        """Step 4: send the expert outputs (y_recv, in ``received.rows`` order)
        back; each lands in ``y`` [T k, H] at the send-buffer row it came
        from, ready for ep_combine."""
        n = sum(received.send_splits)
        dist.all_to_all_single(_as_words(y[:n]), _as_words(y_recv), received.send_splits, received.recv_splits,
                               group=self.group)
        return y
