"""Pins of the balanced expert-parallel plan oracle (oracle/ep_plan.py).

The K3 report review's MoonEP paragraph fixes the guarantee: with E experts on
R ranks and at most E/R redundant expert slots per rank, every rank can receive
exactly S x K routed tokens, and the bound is close to tight in the worst case.
The checker states that guarantee directly; the greedy is checked against it,
against hand traces, and against a brute-force transportation LP that finds
the smallest slot bound for tiny cases without any greedy."""
import numpy as np
import pytest

from oracle import ep_plan as ep


def _plan_from_segments(seg, R, E):
    """A plan dict from hand-written segments listed rank by rank."""
    rank_begin, rank_nseg = [0] * R, [0] * R
    for r in range(R):
        ids = [i for i, s in enumerate(seg) if s[1] == r]
        rank_begin[r], rank_nseg[r] = (ids[0], len(ids)) if ids else (len(seg), 0)
    exp_off, exp_seg = [0], []
    for e in range(E):
        exp_seg += sorted((i for i, s in enumerate(seg) if s[0] == e), key=lambda i: seg[i][2])
        exp_off.append(len(exp_seg))
    return dict(seg=seg, rank_begin=rank_begin, rank_nseg=rank_nseg, exp_off=exp_off, exp_seg=exp_seg)


# R = 3 ranks with one expert each (m = 1), C = 2 rows per rank, loads 3, 3, 0:
# rank 2 has nothing of its own and must borrow; a plan with one redundant
# expert per rank exists by routing expert 0 through rank 2 and expert 1
# through rank 0.
HAND_SEG = [(0, 0, 2, 1, 0), (1, 0, 0, 1, 1), (1, 1, 1, 2, 0), (0, 2, 0, 2, 0)]


def test_checker_accepts_a_hand_plan():
    p = _plan_from_segments(HAND_SEG, 3, 3)
    assert ep.check_plan(p, [3, 3, 0], 3, 2) == 1


# each plan breaks exactly one rule of the guarantee (loads 3, 3, 0 unless stated)
MISTAKES = {
    # rank 1 receives 3 rows (expert 1 given 4 tokens so that coverage still holds)
    "rows": ([(0, 0, 2, 1, 0), (1, 0, 0, 1, 1), (1, 1, 1, 3, 0), (0, 2, 0, 2, 0)], [3, 4, 0], "receives 3 rows"),
    # expert 0's token 1 is placed twice and token 0 never
    "overlap": ([(0, 0, 1, 1, 0), (1, 0, 0, 1, 1), (1, 1, 1, 2, 0), (0, 2, 1, 2, 0)], [3, 3, 0], "gap or overlap"),
    # rank 2 borrows experts 0 and 1: two redundant slots with m = 1
    "slots": ([(0, 0, 1, 2, 0), (1, 1, 1, 2, 0), (0, 2, 0, 1, 0), (1, 2, 0, 1, 1)], [3, 3, 0], "redundant slots"),
    # rank 2 holds expert 0 in two segments
    "twice": ([(0, 0, 2, 1, 0), (1, 0, 0, 1, 1), (1, 1, 1, 2, 0), (0, 2, 0, 1, 0), (0, 2, 1, 1, 1)], [3, 3, 0],
              "twice"),
    # rank 0's second segment starts at row 2
    "gap": ([(0, 0, 2, 1, 0), (1, 0, 0, 1, 2), (1, 1, 1, 2, 0), (0, 2, 0, 2, 0)], [3, 3, 0], "starts at row 2"),
    # expert 1 has 4 tokens, only 3 placed
    "missing": (HAND_SEG, [3, 4, 0], "3 of 4 tokens"),
}


@pytest.mark.parametrize("mistake", sorted(MISTAKES))
def test_checker_rejects_planted_mistakes(mistake):
    seg, counts, msg = MISTAKES[mistake]
    p = _plan_from_segments(seg, 3, 3)
    with pytest.raises(AssertionError, match=msg):
        ep.check_plan(p, counts, 3, 2)


def test_greedy_hand_trace():
    # H = (3, 3, 0): rank 2 first, takes 2 of the largest expert (0, the lower
    # index of the tie); then rank 0 (H = 1) keeps expert 0's last token and
    # takes 1 of expert 1; rank 1 keeps the rest.
    p = ep.plan([3, 3, 0], 3, 2)
    assert p["seg"] == [(0, 2, 0, 2, 0), (0, 0, 2, 1, 0), (1, 0, 0, 1, 1), (1, 1, 1, 2, 0)]
    assert ep.check_plan(p, [3, 3, 0], 3, 2) == 1


def test_balanced_load_stays_home():
    rng = np.random.default_rng(5)
    R, m, C = 4, 3, 60
    counts = []
    for _ in range(R):
        cut = np.sort(rng.integers(0, C + 1, m - 1))
        counts += list(np.diff(np.concatenate([[0], cut, [C]])))
    p = ep.plan(counts, R, C)
    assert ep.check_plan(p, counts, R, C) == 0
    assert all(s[1] == ep.home(s[0], R * m, R) for s in p["seg"])
    assert len(p["seg"]) == sum(1 for v in counts if v > 0)


def _loads(rng, kind, R, m, C):
    E = R * m
    total = R * C
    if kind == "uniform":
        return rng.multinomial(total, np.full(E, 1.0 / E))
    if kind == "zipf":
        w = 1.0 / np.arange(1, E + 1) ** 1.1
        return rng.multinomial(total, rng.permutation(w / w.sum()))
    if kind == "one":
        c = np.zeros(E, np.int64)
        c[rng.integers(E)] = total
        return c
    if kind == "idle_ranks":
        w = rng.random(E)
        w[: (R // 2) * m] = 0.0
        return rng.multinomial(total, w / w.sum())
    if kind == "sparse":
        w = (rng.random(E) < 0.2) * rng.random(E) + 1e-12
        return rng.multinomial(total, w / w.sum())
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["uniform", "zipf", "one", "idle_ranks", "sparse"])
@pytest.mark.parametrize("R,m", [(1, 4), (2, 1), (3, 2), (4, 7), (8, 3), (16, 2)])
def test_greedy_meets_the_guarantee(kind, R, m):
    rng = np.random.default_rng(100 * R + m)
    for C in (1, 7, 64):
        counts = _loads(rng, kind, R, m, C)
        p = ep.plan(counts, R, C)
        red = ep.check_plan(p, counts, R, C)
        assert red <= m and red == p["max_redundant"]


@pytest.mark.parametrize("R,m", [(2, 1), (2, 2), (3, 1), (3, 2)])
def test_slot_bound_holds_by_brute_force(R, m):
    """The guarantee itself, with no greedy: over every choice of redundant
    experts, m slots per rank always admit a balanced plan."""
    rng = np.random.default_rng(7 * R + m)
    for _ in range(6):
        C = int(rng.integers(1, 6))
        counts = _loads(rng, ["zipf", "idle_ranks", "one"][int(rng.integers(3))], R, m, C)
        s = ep.min_redundant(counts, R, C)
        assert s <= m
        assert ep.plan(counts, R, C)["max_redundant"] >= s


@pytest.mark.parametrize("R,m", [(2, 1), (2, 2), (3, 1), (3, 2)])
def test_lower_bound_family_by_brute_force(R, m):
    """One idle rank, all other experts equal: exactly ceil((R-1) m / R) slots
    are needed (brute force), which is m itself at R = 3, m = 2."""
    counts, C, bound = ep.lower_bound_counts(R, m)
    assert ep.min_redundant(counts, R, C) == bound
    assert ep.plan(counts, R, C)["max_redundant"] == bound


def test_lower_bound_family_approaches_the_bound():
    # 896 experts on 8 ranks: the idle rank needs ceil(7 * 112 / 8) = 98 of its 112 slots
    counts, C, bound = ep.lower_bound_counts(8, 112)
    assert bound == 98
    p = ep.plan(counts, 8, C)
    assert ep.check_plan(p, counts, 8, C) == 98


def test_dispatch_hand_trace():
    # 2 ranks, 2 experts, S = 2, K = 1.  Rank 0 routes both tokens to expert 0,
    # rank 1 its tokens to experts 0 and 1: loads (3, 1), C = 2.  The plan:
    # rank 1 (H = 1) keeps expert 1 and takes expert 0's first token; rank 0
    # keeps expert 0's tokens 1 and 2.  Expert 0's tokens in (rank, token)
    # order: rank 0 token 0 -> rank 1 row 1; rank 0 token 1 -> rank 0 row 0;
    # rank 1 token 0 -> rank 0 row 1; expert 1: rank 1 token 1 -> rank 1 row 0.
    idx = [np.array([[0], [0]]), np.array([[0], [1]])]
    p = ep.plan([3, 1], 2, 2)
    assert p["seg"] == [(1, 1, 0, 1, 0), (0, 1, 0, 1, 1), (0, 0, 1, 2, 0)]
    (r0, w0), (r1, w1) = ep.dispatch(idx, p, 2)
    assert r0.ravel().tolist() == [1, 0] and w0.ravel().tolist() == [1, 0]
    assert r1.ravel().tolist() == [0, 1] and w1.ravel().tolist() == [1, 0]


def _routing(rng, R, S, K, E, skew):
    w = 1.0 / np.arange(1, E + 1) ** skew
    w = rng.permutation(w / w.sum())
    return [np.stack([rng.choice(E, K, replace=False, p=w) for _ in range(S)]).astype(np.int32)
            for _ in range(R)]


@pytest.mark.parametrize("R,m,S,K,skew", [(2, 3, 10, 2, 0.0), (4, 4, 16, 4, 1.2), (8, 2, 6, 3, 2.0)])
def test_dispatch_fills_every_row_once(R, m, S, K, skew):
    rng = np.random.default_rng(R * 31 + S)
    E = R * m
    idx = _routing(rng, R, S, K, E, skew)
    cnt = ep.rank_counts(idx, E)
    p = ep.plan(cnt.sum(axis=0), R, S * K)
    ep.check_plan(p, cnt.sum(axis=0), R, S * K)
    # the expert held at each destination row, from the segments
    held = np.full((R, S * K), -1)
    for e, r, _, n, dst in p["seg"]:
        held[r, dst:dst + n] = e
    hit = np.zeros((R, S * K), np.int64)
    sends = np.zeros((R, R), np.int64)
    for q, (rank, row) in enumerate(ep.dispatch(idx, p, E)):
        for s in range(S):
            for k in range(K):
                hit[rank[s, k], row[s, k]] += 1
                assert held[rank[s, k], row[s, k]] == idx[q][s, k]
                sends[q, rank[s, k]] += 1
    assert (hit == 1).all()
    assert (sends == ep.send_counts(cnt, p)).all()
    assert (sends.sum(axis=0) == S * K).all()
