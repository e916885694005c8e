"""Pins for the oracle's Top-K, renormalisation, capacity dropping and the
permutation map, by brute force on tiny inputs and by the invariants the
dispatcher must keep (counts, capacity bound, bijection)."""
import itertools
import math

import numpy as np
import pytest

from oracle import moe_oracle as O


def _beats(p_row, a, b):
    """Total order of the Top-K rule: higher p first, then lower expert index."""
    return p_row[a] > p_row[b] or (p_row[a] == p_row[b] and a < b)


@pytest.mark.parametrize("E,K", [(4, 1), (4, 2), (6, 3), (8, 2), (8, 4), (5, 5)])
@pytest.mark.parametrize("ties", [False, True])
def test_topk_brute_force(E, K, ties):
    rng = np.random.default_rng(E * 10 + K)
    T = 64
    if ties:  # few distinct values force ties
        p = rng.integers(0, 3, (T, E)).astype(np.float32) / np.float32(4)
    else:
        p = O.softmax_f32(rng.standard_normal((T, E)).astype(np.float32))
    idx, prob = O.topk(p, K)
    for t in range(T):
        winners = [set(S) for S in itertools.combinations(range(E), K)
                   if all(_beats(p[t], a, b) for a in S for b in range(E) if b not in S)]
        assert len(winners) == 1
        assert set(idx[t].tolist()) == winners[0]
        # selection order follows the same total order
        for k in range(K - 1):
            assert _beats(p[t], idx[t, k], idx[t, k + 1])
        assert np.array_equal(prob[t], p[t, idx[t]])


def test_renorm_weights():
    rng = np.random.default_rng(0)
    p = O.softmax_f32(rng.standard_normal((500, 8)).astype(np.float32))
    idx, prob = O.topk(p, 2)
    w = O.renorm_weights(prob, True)
    assert w.dtype == np.float32
    s = w.astype(np.float64).sum(axis=1)
    assert np.all(np.abs(s - 1.0) <= 4 * 2.0**-24)
    ratio = w.astype(np.float64) / prob.astype(np.float64)
    assert np.allclose(ratio, ratio[:, :1], rtol=3e-7)
    assert np.array_equal(O.renorm_weights(prob, False), prob)


def test_capacity_formula():
    # ceil(CF * S * K / E): cases from the benchmark shapes and a ragged one.
    assert O.capacity(1.0, 4096, 2, 8) == 1024
    assert O.capacity(1.0, 4096, 8, 64) == 512
    assert O.capacity(1.0, 10, 2, 4) == 5
    assert O.capacity(1.0, 11, 2, 4) == 6
    assert O.capacity(1.25, 100, 2, 8) == 32      # 31.25 -> 32
    assert O.capacity(0.5, 7, 1, 4) == 1          # 0.875 -> 1


def _brute_keep(idx, prob, E, cf, S):
    """O(n^2) definition: an assignment is kept when fewer than cap other
    assignments of the same (sub-sequence, expert) beat it under
    (prob descending, token ascending)."""
    T, K = idx.shape
    keep = np.zeros((T, K), dtype=np.uint8)
    for lo in range(0, T, S):
        hi = min(T, lo + S)
        cap = math.ceil(float(np.float32(cf)) * (hi - lo) * K / E)
        cands = [(t, k) for t in range(lo, hi) for k in range(K)]
        for (t, k) in cands:
            e = idx[t, k]
            better = sum(1 for (u, j) in cands if idx[u, j] == e and
                         (prob[u, j] > prob[t, k] or (prob[u, j] == prob[t, k] and u < t)))
            keep[t, k] = 1 if better < cap else 0
    return keep


@pytest.mark.parametrize("T,E,K,S,cf,ties", [
    (48, 4, 2, 16, 1.0, False), (48, 4, 2, 16, 1.0, True), (50, 8, 2, 20, 1.0, False),
    (40, 4, 1, 40, 0.5, False), (64, 8, 4, 16, 1.25, True), (30, 4, 2, 7, 1.0, False)])
def test_capacity_brute_force(T, E, K, S, cf, ties):
    rng = np.random.default_rng(T + E + K)
    l = rng.standard_normal((T, E)).astype(np.float32)
    if ties:
        # repeated token rows -> equal probabilities across tokens, so the
        # token-index tie rule decides which of them survive
        l = np.tile(l[:5], (T // 5 + 1, 1))[:T]
    p = O.softmax_f32(l)
    idx, prob = O.topk(p, K)
    keep = O.capacity_keep(idx, prob, E, cf, S)
    assert np.array_equal(keep, _brute_keep(idx, prob, E, cf, S))


def test_capacity_short_last_subsequence_uses_its_own_length():
    """T = 37 in sub-sequences of 16 leaves a last one of 5 tokens, whose
    capacity is ceil(1.0 * 5 * 2 / 4) = 3 (the full blocks' is 8). Expert 0
    is every token's first choice, so it has 5 candidates there and keeps 3,
    the 3 highest-probability ones."""
    rng = np.random.default_rng(11)
    T, E, K, S = 37, 4, 2, 16
    l = rng.standard_normal((T, E)).astype(np.float32)
    l[:, 0] += np.float32(6.0)
    p = O.softmax_f32(l)
    idx, prob = O.topk(p, K)
    keep = O.capacity_keep(idx, prob, E, 1.0, S)
    assert np.array_equal(keep, _brute_keep(idx, prob, E, 1.0, S))
    last = slice(32, 37)
    assert np.all(idx[last, 0] == 0)
    kept = keep[last, 0]
    assert kept.sum() == 3
    assert prob[last, 0][kept == 1].min() > prob[last, 0][kept == 0].max()
    for lo in (0, 16):   # full blocks: 16 candidates, 8 kept
        assert keep[lo:lo + 16, 0].sum() == 8


def test_capacity_invariants():
    rng = np.random.default_rng(5)
    T, E, K, S = 1000, 8, 2, 256
    p = O.softmax_f32((rng.standard_normal((T, E)) * 2).astype(np.float32))
    idx, prob = O.topk(p, K)
    keep = O.capacity_keep(idx, prob, E, 1.0, S)
    for lo in range(0, T, S):
        hi = min(T, lo + S)
        cap = O.capacity(1.0, hi - lo, K, E)
        for e in range(E):
            m = idx[lo:hi] == e
            demand = int(m.sum())
            kept = int(keep[lo:hi][m].sum())
            assert kept == min(cap, demand)
            if kept < demand:   # every dropped key is below every kept key
                kp = prob[lo:hi][m & (keep[lo:hi] == 1)]
                dp = prob[lo:hi][m & (keep[lo:hi] == 0)]
                assert dp.max() <= kp.min()
    # a capacity factor so large that cap >= demand everywhere keeps everything
    assert O.capacity_keep(idx, prob, E, 1e6, S).all()
    assert O.capacity_keep(idx, prob, E, float(E) / K, S).all()   # cap = S
    # S = T is the full-sequence rule
    assert np.array_equal(O.capacity_keep(idx, prob, E, 1.0, 0),
                          O.capacity_keep(idx, prob, E, 1.0, T))


@pytest.mark.parametrize("drop", [False, True])
def test_map_invariants(drop):
    rng = np.random.default_rng(7)
    T, E, K = 777, 8, 3
    p = O.softmax_f32((rng.standard_normal((T, E)) * 2).astype(np.float32))
    idx, prob = O.topk(p, K)
    keep = O.capacity_keep(idx, prob, E, 0.8, 100) if drop else np.ones((T, K), np.uint8)
    counts, offsets, row_of, src_of, n_kept = O.build_map(idx, keep, E)
    assert counts.sum() == keep.sum() == n_kept
    if not drop:
        assert n_kept == T * K
    assert offsets[0] == 0 and np.all(np.diff(offsets) == counts)
    # row_of on kept slots is a bijection onto [0, n_kept), src_of its inverse
    kept_rows = row_of[keep == 1]
    assert np.array_equal(np.sort(kept_rows), np.arange(n_kept))
    assert np.all(row_of[keep == 0] == -1)
    t_of, k_of = src_of // K, src_of % K
    assert np.array_equal(row_of[t_of, k_of], np.arange(n_kept))
    # expert-major, token-ascending within an expert
    e_of = idx[t_of, k_of]
    for e in range(E):
        seg = slice(offsets[e], offsets[e + 1])
        assert np.all(e_of[seg] == e)
        assert np.all(np.diff(t_of[seg]) > 0)


def test_route_composes_the_pinned_steps():
    """route() wires the steps the way the readings say: Top-K on the fp32
    softmax of the logits; capacity ranks by the raw probability p (not the
    renormalised weight); the weights are prob / (sum of the K probs); a
    dropless layer keeps every slot."""
    from synthetic import MoEConfig
    rng = np.random.default_rng(21)
    for drop, renorm, K, cf in [(True, True, 2, 0.6), (True, False, 3, 0.5), (False, True, 2, 1.0)]:
        cfg = MoEConfig("r", T=48, d=8, E=6, K=K, F=8, dtype="f32", drop=drop, cf=cf, S=16,
                        renorm=renorm)
        logits = (rng.standard_normal((cfg.T, cfg.E)) * 2).astype(np.float32)
        r = O.route(cfg, None, logits=logits.astype(np.float64))
        p = O.softmax_f32(logits)
        assert np.array_equal(r["p"], p)
        for t in range(cfg.T):   # Top-K by the brute-force total order
            for k in range(K - 1):
                assert _beats(p[t], r["topk_idx"][t, k], r["topk_idx"][t, k + 1])
            rest = [e for e in range(cfg.E) if e not in r["topk_idx"][t]]
            assert all(_beats(p[t], r["topk_idx"][t, K - 1], e) for e in rest)
        prob = np.take_along_axis(p, r["topk_idx"].astype(np.int64), axis=1)
        assert np.array_equal(r["topk_prob"], prob)
        w_ref = prob / prob.sum(axis=1, keepdims=True, dtype=np.float32) if renorm else prob
        assert np.allclose(r["topk_w"], w_ref, rtol=2e-7, atol=0)
        if drop:
            keep = _brute_keep(r["topk_idx"], prob, cfg.E, cf, cfg.S)
            assert 0 < keep.sum() < cfg.T * K
        else:
            keep = np.ones((cfg.T, K), np.uint8)
        assert np.array_equal(r["keep"], keep)


# ---- GShard-style padded layout (f2) ----

def test_padded_map_is_the_compact_map_with_fixed_strides():
    """Expert e's rows of the padded map are its compact rows shifted from
    offsets[e] to e*C, in the same order; padding rows are empty; every kept
    expert count fits the capacity the drop rule implies."""
    rng = np.random.default_rng(3)
    for T, S, E, K, cf in [(60, 16, 4, 2, 1.0), (45, 45, 8, 3, 0.75), (33, 8, 5, 2, 4.0)]:
        logits = rng.standard_normal((T, E))
        p = O.softmax_f32(logits)
        idx, prob = O.topk(p, K)
        keep = O.capacity_keep(idx, prob, E, cf, S)
        C = O.padded_capacity(T, S, K, E, cf)
        counts, offsets, row_of, src_of, n = O.build_map(idx, keep, E)
        pc, po, prow, psrc = O.build_map_padded(idx, keep, E, C)
        assert np.array_equal(pc, counts) and counts.max() <= C
        assert np.array_equal(po, np.arange(E + 1) * C)
        for e in range(E):
            assert np.array_equal(psrc[e * C:e * C + counts[e]], src_of[offsets[e]:offsets[e + 1]])
            assert np.all(psrc[e * C + counts[e]:(e + 1) * C] == -1)
        kept = keep.astype(bool)
        e_of = idx.astype(np.int64)
        assert np.array_equal(prow[kept] - e_of[kept] * C, row_of[kept] - offsets[e_of[kept]])
        assert np.all(prow[~kept] == -1)
        x = rng.standard_normal((T, 6)).astype(np.float32)
        Xp = O.permute_padded(x, psrc, K)
        assert np.array_equal(Xp[psrc >= 0], x[psrc[psrc >= 0] // K])
        assert not Xp[psrc < 0].any()


def test_padded_capacity_formula():
    # two sub-sequences of 4096, cap = ceil(1.0 * 4096 * 2 / 8) = 1024 each
    assert O.padded_capacity(8192, 4096, 2, 8, 1.0) == 2048
    # full sequence: S = 0 means S = T
    assert O.padded_capacity(100, 0, 2, 4, 1.0) == 50
    # capacity above the sub-sequence length is clipped to it (one slot per token)
    assert O.padded_capacity(10, 4, 2, 2, 4.0) == 4 + 4 + 2
