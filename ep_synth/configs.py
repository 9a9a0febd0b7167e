"""Workload catalogue: the five synthetic MoE shapes the path is tested and timed on.

Shapes follow the decode / prefill / mid-size MoE workloads of the UBEP
evaluation ("NJU x Huawei UBEP: Reengineering MoE Expert Parallelism",
Experimental Evaluation: Qwen3-30B, GLM-4.7, DeepSeek-R1 and DeepSeek-V3.2 on
CloudMatrix384). No model weights or traces are used: every tensor is drawn
from the seeded streams in :mod:`ep_synth`.

``ranks_per_node`` = 16 follows the testbed of the same section (256 NPU dies in
16 servers). ``num_workers`` = 152 is one chunk-schedule worker per GB300 SM.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tokens
    H: int            # hidden size (bf16 elements per row)
    E: int            # experts
    R: int            # virtual expert-parallel ranks (E % R == 0)
    k: int            # experts per token
    n_groups: int = 1        # expert groups for group-limited routing (1 = off)
    topk_groups: int = 1     # groups kept per token
    renormalize: int = 1     # top-k weights renormalised to sum to 1
    zipf_s: float | None = None  # Zipf exponent of the expert-popularity bias (None = uniform)
    seed: int = 0
    ranks_per_node: int = 16
    self_rank: int = 0
    num_workers: int = 152
    ranks_per_pod: int = 0   # 0: no pod tier (two hop classes)
    note: str = ""

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def pairs(self) -> int:
        return self.T * self.k

    def algorithmic_bytes(self) -> dict:
        """Bytes each step must move at least once (read + write), per kernel call.

        route    : logits T*E*4 in, idx + w T*k*8 out
        layout   : idx T*k*4 in, slot T*k*4 out, counts/offsets (2E+2R+2)*4
        dispatch : x T*H*2 in, send T*k*H*2 out, slot T*k*4 in, meta T*k*4 out
        combine  : y T*k*H*2 in, out T*H*2 out, slot + w T*k*8 in
        """
        T, H, E, R, k = self.T, self.H, self.E, self.R, self.k
        return {
            "route": T * E * 4 + T * k * 8,
            "layout": T * k * 8 + (2 * E + 2 * R + 2) * 4,
            "dispatch": T * H * 2 + T * k * H * 2 + T * k * 8,
            "combine": T * k * H * 2 + T * k * 8 + T * H * 2,
        }

    def total_bytes(self) -> int:
        return sum(self.algorithmic_bytes().values())


CONFIGS = {
    "tiny": Workload("tiny", T=128, H=256, E=8, R=4, k=2,
                     note="tiny: T=128, H=256, E=8 over R=4, top-2; experts scale rows by (e+1)/8"),
    "decode": Workload("decode", T=256, H=7168, E=256, R=64, k=8,
                       note="decode-shaped: T=256, H=7168, E=256 over R=64, top-8, N(0,1) logits"),
    "prefill": Workload("prefill", T=4096, H=7168, E=256, R=32, k=8, zipf_s=1.2,
                        note="prefill-shaped, skewed: T=4096, H=7168, E=256 over R=32, top-8, Zipf s=1.2 popularity"),
    "mid": Workload("mid", T=16384, H=4096, E=128, R=16, k=8, n_groups=8, topk_groups=4,
                    note="mid-size MoE: T=16384, H=4096, E=128 over R=16, top-8 within top-4 of 8 groups"),
}

SWEEP_T = (1, 8, 64, 512, 4096, 32768)


def sweep_workloads() -> list[Workload]:
    """The sweep: T in SWEEP_T x {uniform, Zipf 1.2}, H=7168, E=256 over R=64, top-8."""
    out = []
    for dist, s in (("uniform", None), ("zipf", 1.2)):
        for T in SWEEP_T:
            out.append(Workload(f"sweep-{dist}-T{T}", T=T, H=7168, E=256, R=64, k=8, zipf_s=s,
                                note=f"sweep: T={T}, H=7168, E=256 over R=64, top-8, {dist} routing"))
    return out


def get_workload(name: str) -> Workload:
    if name in CONFIGS:
        return CONFIGS[name]
    for w in sweep_workloads():
        if w.name == name:
            return w
    raise KeyError(f"unknown workload {name!r}; known: {sorted(CONFIGS)} + sweep-<uniform|zipf>-T<n>")
