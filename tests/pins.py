"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an :class:`oracle.Oracle` and raises
``AssertionError`` when the oracle disagrees with what the problem statement
and the mathematics fix: brute-force enumeration on tiny inputs, library
routines for special cases (``scipy.special.softmax``, ``numpy`` stable sort,
torch's bf16 rounding), closed forms, hand-worked tables under
``tests/golden/`` and invariants (counts sum to T*k, every pair exactly once,
rows are a permutation, identity experts reconstruct the input).

The same functions run against planted-mistake builds of the oracle in
``test_oracle_mutants.py``, which shows that each plausible slip fails at least
one pin.
"""
from __future__ import annotations

import itertools
import json
import math
import pathlib

import numpy as np
import scipy.special
import torch

import ep_synth

GOLDEN = pathlib.Path(__file__).resolve().parent / "golden"


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits; normal range)."""
    a = np.maximum(np.abs(v), 2.0**-126)
    return np.exp2(np.floor(np.log2(a)) - 7)


# ---------------------------------------------------------------------------
# route
# ---------------------------------------------------------------------------

def _sorted_topk(l, k, eligible=None):
    E = len(l)
    cand = [e for e in range(E) if eligible is None or eligible[e]]
    return sorted(cand, key=lambda e: (-float(l[e]), e))[:k]


def pin_route_bruteforce(o):
    """idx = the first k of all experts sorted by (-logit, index); many ties."""
    g = _rng(1)
    for E, k in ((8, 1), (8, 2), (13, 5), (64, 8), (256, 8)):
        l = (np.round(g.normal(size=(40, E)) * 2) / 2).astype(np.float32)  # coarse grid: ties
        idx, _ = o.route(l, k)
        for t in range(l.shape[0]):
            assert list(idx[t]) == _sorted_topk(l[t], k), (E, k, t)


def pin_route_group_bruteforce(o):
    """Group-limited top-k: group score = max logit; keep the best groups; top-k inside."""
    g = _rng(2)
    for E, ng, tg, k in ((16, 4, 2, 3), (128, 8, 4, 8), (32, 8, 3, 4)):
        gs = E // ng
        l = (np.round(g.normal(size=(30, E)) * 3) / 3).astype(np.float32)
        idx, _ = o.route(l, k, ng, tg)
        for t in range(l.shape[0]):
            score = [max(float(v) for v in l[t, q * gs:(q + 1) * gs]) for q in range(ng)]
            kept = sorted(range(ng), key=lambda q: (-score[q], q))[:tg]
            elig = [(e // gs) in kept for e in range(E)]
            assert list(idx[t]) == _sorted_topk(l[t], k, elig), (E, ng, tg, k, t)
        # unrenormalised weights are entries of the softmax over ALL E experts
        # (the group limit restricts the choice, not the softmax)
        idx_raw, w_raw = o.route(l, k, ng, tg, renormalize=0)
        full = scipy.special.softmax(l.astype(np.float64), axis=1)
        assert np.array_equal(idx_raw, idx)
        assert np.allclose(w_raw, np.take_along_axis(full, idx_raw.astype(np.int64), axis=1), rtol=1e-12, atol=0)
        # keeping every group is no limit at all
        idx_all, w_all = o.route(l, k, ng, ng)
        idx_plain, w_plain = o.route(l, k, 1, 1)
        assert np.array_equal(idx_all, idx_plain) and np.array_equal(w_all, w_plain)


def pin_route_full_softmax(o):
    """k = E: every expert chosen and the weights are the full softmax."""
    l = _rng(3).normal(size=(25, 8)).astype(np.float32)
    for renorm in (0, 1):
        idx, w = o.route(l, 8, renormalize=renorm)
        p = scipy.special.softmax(l.astype(np.float64), axis=1)
        for t in range(l.shape[0]):
            assert sorted(idx[t]) == list(range(8))
            np.testing.assert_allclose(w[t], p[t, idx[t]], rtol=1e-13, atol=0)


def pin_route_weights(o):
    """Renormalised weights = softmax of the chosen logits alone (the full
    denominator cancels); plain weights = full-softmax entries."""
    g = _rng(4)
    for E, k, bias in ((256, 8, None), (256, 8, 1.2), (128, 8, None), (8, 2, None)):
        l = g.normal(size=(50, E))
        if bias is not None:
            l = l + ep_synth.zipf_log_bias(E, bias)
        l = l.astype(np.float32)
        idx, wr = o.route(l, k, renormalize=1)
        _, wp = o.route(l, k, renormalize=0)
        p = scipy.special.softmax(l.astype(np.float64), axis=1)
        for t in range(l.shape[0]):
            sel = l[t, idx[t]].astype(np.float64)
            np.testing.assert_allclose(wr[t], scipy.special.softmax(sel), rtol=1e-12, atol=0)
            np.testing.assert_allclose(wp[t], p[t, idx[t]], rtol=1e-12, atol=0)
        np.testing.assert_allclose(wr.sum(axis=1), 1.0, rtol=0, atol=1e-12)


def pin_route_equal_logits(o):
    """Equal logits: experts 0..k-1 in order, weights 1/k (renorm) or 1/E."""
    l = np.full((3, 16), 0.25, np.float32)
    idx, wr = o.route(l, 4)
    _, wp = o.route(l, 4, renormalize=0)
    assert (idx == np.arange(4)).all()
    np.testing.assert_allclose(wr, 0.25, rtol=1e-15)
    np.testing.assert_allclose(wp, 1.0 / 16, rtol=1e-15)


def pin_route_golden(o):
    """Hand-worked routing cases (tests/golden/route_small.json)."""
    data = json.loads((GOLDEN / "route_small.json").read_text())
    env = {"exp": math.exp}
    for c in data["cases"]:
        l = np.array(c["logits"], np.float32)
        idx, wr = o.route(l, c["k"], c["n_groups"], c["topk_groups"], 1)
        assert idx.tolist() == c["idx"], c["name"]
        exp_r = np.array([[eval(s, env) for s in row] for row in c["w_renorm"]])
        np.testing.assert_allclose(wr, exp_r, rtol=1e-14, err_msg=c["name"])
        if c["w_plain"] is not None:
            _, wp = o.route(l, c["k"], c["n_groups"], c["topk_groups"], 0)
            exp_p = np.array([[eval(s, env) for s in row] for row in c["w_plain"]])
            np.testing.assert_allclose(wp, exp_p, rtol=1e-14, err_msg=c["name"])


# ---------------------------------------------------------------------------
# layout
# ---------------------------------------------------------------------------

def _random_idx(g, T, E, k):
    return np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


def pin_layout_bruteforce(o):
    """T <= 8: slot[t, j] = number of pairs ordered before it by (rank, expert, token),
    counted pair by pair (no scan)."""
    g = _rng(5)
    for T, E, R, k in ((1, 2, 1, 1), (3, 4, 2, 2), (8, 8, 4, 3), (8, 6, 3, 2), (5, 8, 2, 3)):
        idx = _random_idx(g, T, E, k)
        lay = o.layout(idx, E, R)
        epr = E // R
        pairs = [(t, j) for t in range(T) for j in range(k)]
        key = {p: (int(idx[p]) // epr, int(idx[p]), p[0]) for p in pairs}
        for p in pairs:
            expect = sum(1 for q in pairs if key[q] < key[p])
            assert lay["slot"][p] == expect, (T, E, R, k, p)
        for e in range(E):
            assert lay["expert_count"][e] == sum(1 for p in pairs if idx[p] == e)
        for r in range(R):
            assert lay["rank_count"][r] == sum(1 for p in pairs if idx[p] // epr == r)


def pin_layout_counts(o):
    """Counts, offsets and rank offsets against numpy bincount / cumsum."""
    g = _rng(6)
    for T, E, R, k in ((500, 64, 8, 4), (257, 256, 64, 8), (100, 8, 8, 2), (64, 16, 1, 16)):
        idx = _random_idx(g, T, E, k)
        lay = o.layout(idx, E, R)
        cnt = np.bincount(idx.ravel(), minlength=E)
        assert (lay["expert_count"] == cnt).all()
        assert lay["expert_offset"][-1] == T * k
        assert (lay["expert_offset"] == np.concatenate([[0], np.cumsum(cnt)])).all()
        rc = np.bincount(idx.ravel() // (E // R), minlength=R)
        assert (lay["rank_count"] == rc).all()
        assert (lay["rank_offset"] == np.concatenate([[0], np.cumsum(rc)])).all()


def pin_layout_stable_sort(o):
    """k = 1 and R = 1: the slots are a stable counting sort by expert id."""
    g = _rng(7)
    e = g.integers(0, 16, size=777).astype(np.int32)
    lay = o.layout(e[:, None], 16, 1)
    order = np.argsort(e, kind="stable")
    assert (lay["slot"][order, 0] == np.arange(777)).all()


def pin_layout_bijection_stable(o):
    """Every pair gets its own row; within an expert, rows increase with t."""
    g = _rng(8)
    T, E, R, k = 1000, 64, 16, 6
    idx = _random_idx(g, T, E, k)
    lay = o.layout(idx, E, R)
    s = lay["slot"].ravel()
    assert np.array_equal(np.sort(s), np.arange(T * k))
    for ex in range(E):
        rows = lay["slot"][idx == ex]  # boolean mask walks tokens in ascending order
        assert (np.diff(rows) > 0).all()
        lo, hi = lay["expert_offset"][ex], lay["expert_offset"][ex + 1]
        assert rows.min(initial=lo) >= lo and rows.max(initial=lo) < max(hi, lo + 1)


def pin_layout_golden(o):
    d = json.loads((GOLDEN / "layout_small.json").read_text())
    idx = np.array(d["idx"], np.int32)
    lay = o.layout(idx, d["E"], d["R"])
    for key in ("expert_count", "expert_offset", "rank_count", "rank_offset", "slot"):
        assert lay[key].tolist() == d[key], key
    x = np.arange(idx.shape[0] * 8, dtype=np.uint16).reshape(idx.shape[0], 8)
    _, meta = o.dispatch(x, lay["slot"])
    assert meta.tolist() == d["meta"]


# ---------------------------------------------------------------------------
# schedule
# ---------------------------------------------------------------------------

def pin_schedule_golden(o):
    d = json.loads((GOLDEN / "schedule_small.json").read_text())
    for c in d["cases"]:
        ch, wb = o.schedule(np.array(c["rank_offset"], np.int32), c["ranks_per_node"], c["self_rank"], c["W"],
                            c.get("ranks_per_pod", 0))
        assert ch.tolist() == c["chunks"], c["name"]
        assert wb.tolist() == c["worker_begin"], c["name"]


def hop_class(r, rpn, self_rank, rpp=0):
    """0: the sending rank's node; 2: another pod (when pods are given); 1: another node."""
    if r // rpn == self_rank // rpn:
        return 0
    if rpp > 0 and r // rpp != self_rank // rpp:
        return 2
    return 1


def check_schedule_invariants(chunks, wb, rank_offset, rpn, self_rank, W, rpp=0):
    """Tiling, balance and order of a chunk table (also used on GPU output)."""
    R = len(rank_offset) - 1
    total = int(rank_offset[-1])
    n_classes = 3 if rpp > 0 else 2
    assert len(chunks) <= n_classes * W + R
    assert wb[0] == 0 and wb[-1] == len(chunks) and (np.diff(wb) >= 0).all()
    cover = np.zeros(total, np.int32)
    share = np.zeros((W, 3), np.int64)
    for i, (w, c, r, b, n) in enumerate(chunks):
        assert wb[w] <= i < wb[w + 1]
        assert n > 0 and c == hop_class(r, rpn, self_rank, rpp)
        assert rank_offset[r] <= b and b + n <= rank_offset[r + 1]
        cover[b:b + n] += 1
        share[w, c] += n
    assert (cover == 1).all(), "rows not covered exactly once"
    for c in range(3):
        assert share[:, c].max() - share[:, c].min() <= 1, "class shares unbalanced"
    for w in range(W):
        rows = [tuple(chunks[i]) for i in range(wb[w], wb[w + 1])]
        keys = [(-r[1], r[2]) for r in rows]
        assert keys == sorted(keys) and len(set(keys)) == len(keys), "order within a worker"


def pin_schedule_invariants(o):
    g = _rng(9)
    for R, rpn, self_rank, W, rpp in ((64, 16, 0, 152, 0), (32, 16, 17, 7, 0), (16, 16, 3, 40, 0), (8, 1, 5, 3, 0),
                                      (5, 2, 4, 11, 0), (64, 4, 37, 19, 16), (64, 1, 0, 152, 8), (30, 2, 29, 7, 6),
                                      (12, 3, 5, 1, 6)):
        counts = g.integers(0, 30, size=R)
        counts[g.integers(0, R)] = 0
        ro = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        ch, wb = o.schedule(ro, rpn, self_rank, W, rpp)
        check_schedule_invariants(ch, wb, ro, rpn, self_rank, W, rpp)


def pin_schedule_one_pod_is_two_tiers(o):
    """A pod that holds every rank adds no tier: the table equals the two-tier one."""
    g = _rng(15)
    for R, rpn, self_rank, W in ((16, 4, 6, 9), (64, 16, 40, 152)):
        ro = np.concatenate([[0], np.cumsum(g.integers(0, 40, size=R))]).astype(np.int32)
        two = o.schedule(ro, rpn, self_rank, W)
        for rpp in (R, 2 * R):
            three = o.schedule(ro, rpn, self_rank, W, rpp)
            assert np.array_equal(two[0], three[0]) and np.array_equal(two[1], three[1])


# ---------------------------------------------------------------------------
# dispatch / combine / bf16
# ---------------------------------------------------------------------------

def pin_dispatch_provenance(o):
    """send row s is x[meta[s] // k]; meta is a bijection; slot and meta agree."""
    g = _rng(10)
    T, E, R, k, H = 200, 32, 8, 4, 24
    idx = _random_idx(g, T, E, k)
    lay = o.layout(idx, E, R)
    x = g.integers(0, 65536, size=(T, H)).astype(np.uint16)
    send, meta = o.dispatch(x, lay["slot"])
    assert np.array_equal(np.sort(meta), np.arange(T * k))
    assert np.array_equal(send, x[meta // k])
    flat = lay["slot"].ravel()
    assert np.array_equal(meta[flat], np.arange(T * k))
    # multiset of rows = each x row k times
    assert np.array_equal(np.sort(send.view(np.dtype((np.void, 2 * H))).ravel()),
                          np.sort(np.repeat(x, k, axis=0).view(np.dtype((np.void, 2 * H))).ravel()))


def pin_combine_identity(o):
    """Identity experts + renormalised weights reproduce x exactly (the fp32
    error is ~2^-21 relative, far below half a bf16 ulp)."""
    for T, H, E, R, k, seed in ((128, 256, 8, 4, 2, 0), (64, 64, 256, 64, 8, 1)):
        l = ep_synth.gate_logits(seed, T, E)
        x = ep_synth.hidden_bf16_bits(seed, T, H)
        r = o.run_path(l, x, E=E, R=R, k=k, W=8, identity_expert=True)
        assert np.array_equal(r["out"], x)


def pin_combine_k1_dyadic(o):
    """k = 1 with weights of few bits: out = bf16(w * y) exactly (torch rounding)."""
    g = _rng(11)
    T, H = 50, 40
    y = ep_synth.random_rows_bf16_bits(3, T, H)
    slot = g.permutation(T).astype(np.int32)[:, None]
    w = g.choice(np.array([0.5, 0.75, 1.0, 1.5, -0.25, 3.0], np.float32), size=(T, 1))
    out = o.combine(y, slot, w)
    prod = (ep_synth.bf16_bits_to_f32(y)[slot[:, 0]] * w).astype(np.float32)  # exact in fp32
    assert np.array_equal(out, ep_synth.bf16_bits_from_f32(prod))


def pin_combine_fp64_bound(o):
    """|out - sum_j w_j y_j| <= fp32 accumulation bound + half a bf16 ulp of the fp32 sum,
    with the exact sum in fp64; mixed signs."""
    g = _rng(12)
    T, H, k = 60, 48, 8
    y = ep_synth.random_rows_bf16_bits(4, T * k, H)
    slot = g.permutation(T * k).astype(np.int32).reshape(T, k)
    w = ep_synth.random_topk_weights(5, T, k)
    out = ep_synth.bf16_bits_to_f32(o.combine(y, slot, w)).astype(np.float64)
    yf = ep_synth.bf16_bits_to_f32(y).astype(np.float64)
    terms = w.astype(np.float64)[:, :, None] * yf[slot]          # [T, k, H]
    exact = terms.sum(axis=1)
    accb = k * 2.0**-24 * np.abs(terms).sum(axis=1) * (1 + 2.0**-7)
    bound = accb + 0.5 * _bf16_ulp(np.abs(exact) + accb)
    assert (np.abs(out - exact) <= bound).all()


def _round_to_bits(q, mant_bits: int):
    """The rational q rounded to the nearest binary number of `mant_bits`
    significant bits, ties to the even one (normal range, exponent >= -126)."""
    from fractions import Fraction

    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()  # 2^(e-1) < a < 2^(e+1)
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)  # now 2^e <= a < 2^(e+1)
    ulp = Fraction(2) ** (e - (mant_bits - 1))
    n, rem = divmod(a / ulp, 1)
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * ulp


def _fma_chain_bf16(w_row, y_cols, order):
    """acc = 0; acc = fp32(w_j * y_j + acc) for j in `order` (one rounding of the
    exact product-sum per term, as a fused multiply-add does); bf16 RNE of acc.
    Exact rational arithmetic throughout."""
    from fractions import Fraction

    acc = Fraction(0)
    for j in order:
        acc = _round_to_bits(Fraction(float(w_row[j])) * Fraction(float(y_cols[j])) + acc, 24)
    out = np.float32(float(_round_to_bits(acc, 8)))
    return np.uint16(out.view(np.uint32) >> np.uint32(16))


def pin_combine_exact_fma_chain(o):
    """The combine equals its definition computed exactly: one fused multiply-add
    per term in j = 0 .. k-1 order (exact product plus accumulator, rounded once to
    fp32), then bf16 round-to-nearest-even. Half of the tokens are built so that
    the order and the single rounding decide the result: their first two terms
    cancel exactly (w_1 = -w_0, y_1 = y_0, large) and the last two are small, so a
    sum in another order, or with the product rounded before the add, leaves a
    different residue; the pin checks that those alternatives do differ here."""
    g = _rng(21)
    T, H, k = 48, 24, 4
    w = np.empty((T, k), np.float32)
    yv = np.empty((T, k, H), np.float32)
    for t in range(T):
        if t % 2 == 0:  # cancelling pair, then two small terms
            w0 = np.float32(g.uniform(0.5, 1.0))
            w[t] = [w0, -w0, g.uniform(-1, 1), g.uniform(-1, 1)]
            big = np.ldexp(g.uniform(1, 2, H), g.integers(0, 7, H)) * g.choice([-1, 1], H)
            yv[t, 0] = yv[t, 1] = big
            yv[t, 2:] = np.ldexp(g.uniform(1, 2, (2, H)), g.integers(-14, -9, (2, H))) * g.choice([-1, 1], (2, H))
        else:  # arbitrary terms, mixed signs
            w[t] = g.uniform(-1, 1, k)
            yv[t] = g.normal(size=(k, H)) * 4
    ybits_t = ep_synth.bf16_bits_from_f32(yv.reshape(-1)).reshape(T, k, H)
    slot = g.permutation(T * k).astype(np.int32).reshape(T, k)
    y = np.zeros((T * k, H), np.uint16)
    y[slot.reshape(-1)] = ybits_t.reshape(T * k, H)
    out = o.combine(y, slot, w)
    yf = ep_synth.bf16_bits_to_f32(ybits_t)

    def sign_free(b):
        return np.where(b == 0x8000, 0, b)

    forward = reverse = 0
    two_roundings = 0
    for t in range(T):
        for h in range(H):
            ref = _fma_chain_bf16(w[t], yf[t, :, h], range(k))
            assert sign_free(out[t, h]) == sign_free(ref), (t, h, hex(out[t, h]), hex(ref))
            forward += 1
            if t % 2 == 0:
                reverse += int(_fma_chain_bf16(w[t], yf[t, :, h], range(k - 1, -1, -1)) != ref)
                # product rounded to fp32 first, then the add rounded again
                from fractions import Fraction

                acc = Fraction(0)
                for j in range(k):
                    p = _round_to_bits(Fraction(float(w[t, j])) * Fraction(float(yf[t, j, h])), 24)
                    acc = _round_to_bits(p + acc, 24)
                alt = np.uint16(np.float32(float(_round_to_bits(acc, 8))).view(np.uint32) >> np.uint32(16))
                two_roundings += int(alt != ref)
    assert forward == T * H
    assert reverse > 0 and two_roundings > 0, (reverse, two_roundings)


def pin_bf16_rounding(o):
    """The oracle's float -> bf16 rounding equals torch's (RNE) on ties, carries,
    overflow, subnormals and signed zeros."""
    g = _rng(13)
    bits = np.concatenate([
        g.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32),
        np.array([0x3F808000, 0x3F818000, 0x3F80FFFF, 0x7F7FFFFF, 0x7F7F8000, 0x00008000,
                  0x00018000, 0x80000000, 0x00000000, 0xBF808000, 0x7F800000, 0xFF800000], np.uint32)])
    f = bits.view(np.float32)
    f = f[~np.isnan(f)]
    ours = np.array([o.f32_to_bf16(float(v)) for v in f], np.uint16)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    # and back: bf16 -> f32 is exact
    for b in (0x3F80, 0xC2F7, 0x0001, 0x8000, 0x7F7F):
        assert np.float32(o.bf16_to_f32(b)).view(np.uint32) == np.uint32(b) << np.uint32(16)


def pin_expert_scale(o):
    """The harness expert: row s belongs to the expert e with offset[e] <= s <
    offset[e + 1] (found here by brute force over all experts, empty ones
    included) and y = bf16(float(send) * fp32((e + 1) / E)), rounded by torch."""
    g = _rng(14)
    E, H = 9, 24
    counts = g.integers(0, 6, size=E)
    counts[[0, 4, 8]] = 0  # empty experts at both ends and inside
    offset = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(offset[-1])
    send = ep_synth.random_rows_bf16_bits(6, rows, H)
    y = o.expert(send, offset, E)
    owner = np.array([[e for e in range(E) if offset[e] <= s < offset[e + 1]][0] for s in range(rows)])
    scale = (np.float32(1) + owner.astype(np.float32)) / np.float32(E)
    prod = (ep_synth.bf16_bits_to_f32(send) * scale[:, None].astype(np.float32)).astype(np.float32)
    ref = torch.from_numpy(prod).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(y, ref)
    assert np.array_equal(o.expert(send, offset, E, identity=True), send)


# ---------------------------------------------------------------------------
# Token-Flag Fusion block codec
# ---------------------------------------------------------------------------

def _tff_rows(case):
    if "rows_hex" in case:
        return np.stack([np.frombuffer(bytes.fromhex(h), np.uint8) for h in case["rows_hex"]])
    n = case["row_bytes"]
    return (np.arange(n) % 251).astype(np.uint8)[None, :]


def pin_tff_golden(o):
    """Hand-worked frames (tests/golden/tff_small.json): metadata words, payload, zero fill."""
    d = json.loads((GOLDEN / "tff_small.json").read_text())
    for c in d["cases"]:
        rows = _tff_rows(c)
        framed = o.tff_encode(rows, c["epoch"])
        nblk = len([b for b in c["blocks"] if b["row"] == 0])
        assert framed.shape == (rows.shape[0], 512 * nblk), c["name"]
        for b in c["blocks"]:
            blk = framed[b["row"], 512 * b["block"]:512 * (b["block"] + 1)]
            assert blk[:32].tobytes() == bytes.fromhex(b["meta_hex"]), (c["name"], b)
            pay = bytes.fromhex(b["payload_hex"]) if "payload_hex" in b else \
                rows[b["row"], b["payload_from"]:b["payload_from"] + b["payload_len"]].tobytes()
            assert blk[32:32 + len(pay)].tobytes() == pay, (c["name"], b)
            assert not blk[32 + len(pay):].any(), (c["name"], b)
        back, bad = o.tff_decode(framed, c["row_bytes"], c["epoch"])
        assert bad == 0 and np.array_equal(back, rows)


def pin_tff_roundtrip_and_size(o):
    """decode(encode(rows)) == rows with no bad block; a row takes the fewest
    480-byte payloads that hold it (one fewer would not)."""
    g = _rng(16)
    for n in (2, 16, 478, 480, 482, 960, 14336, 4096 * 2, 24576 * 2):
        rows = g.integers(0, 256, size=(3, n), dtype=np.uint8)
        framed = o.tff_encode(rows, 0xFFFFFFFF)
        nblk = framed.shape[1] // 512
        assert framed.shape[1] % 512 == 0 and nblk * 480 >= n and (nblk - 1) * 480 < n
        back, bad = o.tff_decode(framed, n, 0xFFFFFFFF)
        assert bad == 0 and np.array_equal(back, rows)


def pin_tff_rejects_stale_blocks(o):
    """A block whose epoch, row, block index or length does not match is
    counted and its bytes are not copied; every other block still is."""
    g = _rng(17)
    n = 1000  # 3 blocks per row
    rows = g.integers(0, 256, size=(4, n), dtype=np.uint8)
    framed = o.tff_encode(rows, 9)
    hits = [(0, 0, 0, 8), (1, 2, 4, 3), (2, 1, 8, 7), (3, 2, 12, 1)]  # (row, block, metadata byte, new value)
    for r, b, byte, v in hits:
        framed[r, 512 * b + byte] = v
    sentinel = np.full((4, n), 0xEE, np.uint8)
    back, bad = o.tff_decode(framed, n, 9, out=sentinel)
    assert bad == len(hits)
    for r in range(4):
        for b in range(3):
            lo, hi = 480 * b, min(480 * (b + 1), n)
            want = sentinel[r, lo:hi] if any(h[0] == r and h[1] == b for h in hits) else rows[r, lo:hi]
            if any(h[0] == r and h[1] == b for h in hits):
                assert (back[r, lo:hi] == 0xEE).all()
            else:
                assert np.array_equal(back[r, lo:hi], want)
    _, bad_epoch = o.tff_decode(o.tff_encode(rows, 9), n, 10)
    assert bad_epoch == 4 * 3


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
