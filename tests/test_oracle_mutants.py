"""Planted mistakes in the oracle must fail at least one pin.

Each case copies ``oracle/ep_oracle.c`` to a temporary directory, applies one
textual change that models a plausible slip (a flipped comparison, a dropped
term, a wrong index or sign, a transposed operand), builds it with gcc and runs
the whole pin battery of ``pins.py`` against it. A pin battery that lets a
mutant through is not pinning that part of the oracle. CPU only.
"""
import pathlib

import pytest

import oracle
import pins

MUTANTS = [
    ("topk tie goes to the higher index",
     "(best < 0 || l[e] > l[best])) best = e;", "(best < 0 || l[e] >= l[best])) best = e;"),
    ("group score is the minimum",
     "if (l[g * gsize + i] > s) s = l[g * gsize + i];", "if (l[g * gsize + i] < s) s = l[g * gsize + i];"),
    ("group ranking tie to the higher group",
     "(best < 0 || gscore[g] > gscore[best])) best = g;", "(best < 0 || gscore[g] >= gscore[best])) best = g;"),
    ("softmax exponent sign flipped",
     "p[e] = exp((double)l[e] - m);", "p[e] = exp(m - (double)l[e]);"),
    ("renormalisation dropped",
     "w[t * k + j] = renormalize ? p[idx[t * k + j]] / s : p[idx[t * k + j]];",
     "w[t * k + j] = p[idx[t * k + j]];"),
    ("softmax denominator not shifted by the max",
     "            S += p[e];", "            S += exp((double)l[e]);"),
    ("softmax exponent in fp32",
     "p[e] = exp((double)l[e] - m);", "p[e] = (double)expf((float)((double)l[e] - m));"),
    ("group score is the sum",
     "if (l[g * gsize + i] > s) s = l[g * gsize + i];", "s += l[g * gsize + i];"),
    ("softmax over the eligible experts only",
     "p[e] = exp((double)l[e] - m);", "p[e] = eligible[e] ? exp((double)l[e] - m) : 0.0;"),
    ("renormalisation over all E",
     "for (int32_t j = 0; j < k; ++j) s += p[idx[t * k + j]];", "for (int32_t j = 0; j < E; ++j) s += p[j];"),
    ("rank count taken from the rank's first expert",
     "for (int32_t r = 0; r < R; ++r) rank_count[r] = rank_offset[r + 1] - rank_offset[r];",
     "for (int32_t r = 0; r < R; ++r) rank_count[r] = expert_count[r * epr];"),
    ("rank offset indexed by rank, not by first expert",
     "rank_offset[r] = expert_offset[r * epr];", "rank_offset[r] = expert_offset[r];"),
    ("offset scan off by one expert",
     "expert_offset[e + 1] = expert_offset[e] + expert_count[e];",
     "expert_offset[e + 1] = expert_offset[e] + expert_count[e + (e + 1 < E)];"),
    ("tokens walked in reverse (unstable order)",
     "    for (int64_t t = 0; t < T; ++t)\n        for (int32_t j = 0; j < k; ++j) {\n            int32_t e = idx[t * k + j];\n            slot[t * k + j] = cursor[e];",
     "    for (int64_t t = T - 1; t >= 0; --t)\n        for (int32_t j = 0; j < k; ++j) {\n            int32_t e = idx[t * k + j];\n            slot[t * k + j] = cursor[e];"),
    ("near traffic scheduled first",
     "for (int c = 2; c >= 0; --c) {", "for (int c = 0; c <= 2; ++c) {"),
    ("chunk row_begin missing the rank base",
     "rec[3] = (int32_t)(rank_offset[r] + (a - seg_lo));", "rec[3] = (int32_t)(a - seg_lo);"),
    ("worker share rounded up",
     "int64_t hi = N[c] * (w + 1) / W;", "int64_t hi = (N[c] * (w + 1) + W - 1) / W;"),
    ("hop class from the rank, not the node",
     "if (r / ranks_per_node == self_rank / ranks_per_node) return 0;", "if (r == self_rank) return 0;"),
    ("pod tier tested with the node size",
     "r / ranks_per_pod != self_rank / ranks_per_pod) return 2;",
     "r / ranks_per_node != self_rank / ranks_per_pod) return 2;"),
    ("pod tier folded into the node tier",
     "self_rank / ranks_per_pod) return 2;", "self_rank / ranks_per_pod) return 1;"),
    ("schedule chunk at position 0 one row long",
     "rec[4] = (int32_t)(b - a);", "rec[4] = (int32_t)(b - a + (a == 0));"),
    ("schedule worker_begin[W] one short",
     "    worker_begin[W] = n;\n", "    worker_begin[W] = n - (n > 0);\n"),
    ("meta drops the top-k position",
     "meta[s] = (int32_t)(t * k + j);", "meta[s] = (int32_t)(t * k);"),
    ("meta transposed",
     "meta[s] = (int32_t)(t * k + j);", "meta[s] = (int32_t)(j * T + t);"),
    ("combine weight operand transposed",
     "acc = fmaf(w[t * k + j], orc_bf16_to_f32(y[s * H + h]), acc);",
     "acc = fmaf(w[j * T + t], orc_bf16_to_f32(y[s * H + h]), acc);"),
    ("combine drops the last term",
     "            for (int32_t j = 0; j < k; ++j) {\n                int64_t s = slot[t * k + j];\n                if (s < 0 || s >= T * k) return ORC_EINVAL;\n                acc",
     "            for (int32_t j = 0; j < k - 1; ++j) {\n                int64_t s = slot[t * k + j];\n                if (s < 0 || s >= T * k) return ORC_EINVAL;\n                acc"),
    ("combine sums the terms in reverse order",
     "                int64_t s = slot[t * k + j];\n                if (s < 0 || s >= T * k) return ORC_EINVAL;\n"
     "                acc = fmaf(w[t * k + j], orc_bf16_to_f32(y[s * H + h]), acc);",
     "                int64_t s = slot[t * k + (k - 1 - j)];\n                if (s < 0 || s >= T * k) return ORC_EINVAL;\n"
     "                acc = fmaf(w[t * k + (k - 1 - j)], orc_bf16_to_f32(y[s * H + h]), acc);"),
    ("combine rounds the product before the add",
     "acc = fmaf(w[t * k + j], orc_bf16_to_f32(y[s * H + h]), acc);",
     "acc = w[t * k + j] * orc_bf16_to_f32(y[s * H + h]) + acc;"),
    ("combine accumulates in double",
     "            float acc = 0.0f;\n            for (int32_t j = 0; j < k; ++j) {\n"
     "                int64_t s = slot[t * k + j];\n                if (s < 0 || s >= T * k) return ORC_EINVAL;\n"
     "                acc = fmaf(w[t * k + j], orc_bf16_to_f32(y[s * H + h]), acc);",
     "            double acc = 0.0;\n            for (int32_t j = 0; j < k; ++j) {\n"
     "                int64_t s = slot[t * k + j];\n                if (s < 0 || s >= T * k) return ORC_EINVAL;\n"
     "                acc = fma((double)w[t * k + j], (double)orc_bf16_to_f32(y[s * H + h]), acc);"),
    ("expert scale e / E",
     "float scale = (float)(e + 1) / (float)E;", "float scale = (float)e / (float)E;"),
    ("expert ownership boundary off by one",
     "while (e < E - 1 && s >= expert_offset[e + 1]) ++e;", "while (e < E - 1 && s > expert_offset[e + 1]) ++e;"),
    ("TFF decoder ignores the epoch",
     "if (orc_get_u32(blk + 0) != epoch ||", "if (0 ||"),
    ("TFF decoder ignores the block index",
     "orc_get_u32(blk + 8) != (uint32_t)b ||", "0 ||"),
    ("TFF decoder ignores the length",
     "orc_get_u32(blk + 12) != (uint32_t)n) {", "0) {"),
    ("TFF payload not zero-filled",
     "            memset(blk, 0, ORC_TFF_BLOCK);\n", "            memset(blk, 0, ORC_TFF_META);\n"),
    ("TFF payload written over the metadata",
     "memcpy(blk + ORC_TFF_META, in + r * row_bytes + off, (size_t)n);", "memcpy(blk, in + r * row_bytes + off, (size_t)n);"),
    ("TFF last block claims a full payload",
     "            orc_put_u32(blk + 12, (uint32_t)n);", "            orc_put_u32(blk + 12, (uint32_t)ORC_TFF_PAYLOAD);"),
    ("TFF decoder ignores the row field",
     "orc_get_u32(blk + 4) != (uint32_t)r ||", "0 ||"),
    ("TFF block index off by one",
     "            orc_put_u32(blk + 8, (uint32_t)b);", "            orc_put_u32(blk + 8, (uint32_t)(b + 1));"),
    ("bf16 ties rounded away from zero",
     "if (low > 0x8000u || (low == 0x8000u && (keep & 1u)))", "if (low >= 0x8000u)"),
    ("bf16 truncation",
     "        keep += 1u;                      /* carries into the exponent: ok  */", "        keep += 0u;"),
]


def _battery(o):
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(o)
        except (AssertionError, oracle.OracleError, IndexError, ValueError) as exc:  # noqa: PERF203
            failed.append((pin.__name__, type(exc).__name__))
    return failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path: pathlib.Path, name, old, new):
    src = oracle.SOURCE.read_text()
    assert src.count(old) == 1, f"mutation site not unique/absent: {name}"
    mutated = tmp_path / "ep_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.build(mutated, tmp_path / "libmutant.so", force=True)
    failed = _battery(oracle.Oracle(lib))
    assert failed, f"no pin caught the mutant: {name}"
