"""Oracle of the balanced expert-parallel dispatch plan (MoonEP).

TEST INFRASTRUCTURE ONLY (tests and the smoke check).

Source: the K3 report review, section "3T pre-training: turning irregular MoE
into a static execution plan" (the MoonEP paragraph).  From the router output
of the current micro-batch the planner copies hot experts to other ranks for
the step and sends every routed token straight to the expert copy that will
process it.  With E experts and R expert-parallel ranks, at most E/R redundant
expert slots per rank always suffice for a plan in which every rank receives
exactly S x K routed tokens (S tokens per rank, top-K routing); the pages add
that the bound is close to tight for the worst load distribution, and that the
fixed per-rank size removes the host read of token counts before the expert
kernels.  The pages give the guarantee, not an algorithm.

Readings (the pages print no algorithm or layout):
- rank r owns the m = E/R experts r*m .. r*m + m - 1 ("home" experts); an
  expert processed on another rank occupies one of that rank's m redundant
  slots;
- the plan is the greedy below.  Repeat R times: take the unplanned rank with
  the smallest remaining home load H (ties: lowest rank), give it every
  remaining token of its home experts, then fill the rest of its C = S*K rows
  from the largest remaining experts (ties: lowest expert index), whole
  experts first and a part of the last one.  Why at most m experts are taken:
  with n ranks left, their experts hold n*C tokens and the chosen rank holds
  H <= C of them; the other ranks' at most (n-1)*m experts hold n*C - H, so
  their m largest hold at least (n*C - H)/(n-1) >= C - H, the rows still to
  fill.  Each take removes an expert except the last, which ends the rank;
- the tokens of expert e are numbered globally in (source rank, token) order;
  successive takes of e get successive ranges of that numbering, the home
  rank's share last;
- a rank's receive buffer holds its segments in the order they were planned
  (home experts in index order, then the takes), each one a contiguous run of
  rows.

Verified independently of the greedy by check_plan (the guarantee itself),
by the transportation LP in min_redundant (which finds the smallest per-rank
slot bound for tiny cases by trying every choice of redundant experts), and
by the closed-form lower bound of lower_bound_counts.
"""
from __future__ import annotations

from itertools import combinations, product

import numpy as np


def home(e: int, E: int, R: int) -> int:
    """The rank that owns expert e: contiguous blocks of E/R experts."""
    return e // (E // R)


def plan(counts, R: int, C: int) -> dict:
    """The greedy plan for per-expert loads `counts` [E] (sum R*C).

    Returns a dict of
      seg: list of (expert, rank, src, count, dst) in planning order,
      rank_begin, rank_nseg: each rank's segments are seg[rank_begin[r] : +rank_nseg[r]],
      exp_off [E+1], exp_seg: expert e's segments, increasing src, are
          seg[exp_seg[i]] for i in exp_off[e] .. exp_off[e+1]-1,
      max_redundant: the largest number of non-home experts on one rank.
    """
    c = np.asarray(counts, dtype=np.int64)
    E = c.size
    if R <= 0 or E % R:
        raise ValueError("E must be a positive multiple of R")
    if int(c.sum()) != R * C or (c < 0).any():
        raise ValueError("loads must be non-negative and sum to R * C")
    m = E // R
    rem = [int(v) for v in c]
    taken = [0] * E
    H = [sum(rem[r * m:(r + 1) * m]) for r in range(R)]
    planned = [False] * R
    seg = []
    rank_begin, rank_nseg = [0] * R, [0] * R
    max_red = 0
    for _ in range(R):
        r = min((H[q], q) for q in range(R) if not planned[q])[1]
        need = C - H[r]
        assert need >= 0
        begin, dst = len(seg), 0
        for e in range(r * m, (r + 1) * m):
            if rem[e] > 0:
                seg.append((e, r, taken[e], rem[e], dst))
                dst += rem[e]
                taken[e] += rem[e]
                rem[e] = 0
        H[r] = 0
        nred = 0
        while need > 0:
            e = max(range(E), key=lambda j: (rem[j], -j))
            assert rem[e] > 0
            t = min(rem[e], need)
            seg.append((e, r, taken[e], t, dst))
            dst += t
            taken[e] += t
            rem[e] -= t
            H[home(e, E, R)] -= t
            need -= t
            nred += 1
        assert dst == C
        max_red = max(max_red, nred)
        planned[r] = True
        rank_begin[r], rank_nseg[r] = begin, len(seg) - begin
    per_e = [[] for _ in range(E)]
    for i, s in enumerate(seg):
        per_e[s[0]].append(i)
    exp_off = [0]
    exp_seg = []
    for e in range(E):
        exp_seg += sorted(per_e[e], key=lambda i: seg[i][2])
        exp_off.append(len(exp_seg))
    return dict(seg=seg, rank_begin=rank_begin, rank_nseg=rank_nseg, exp_off=exp_off, exp_seg=exp_seg,
                max_redundant=max_red)


def check_plan(p: dict, counts, R: int, C: int) -> int:
    """Assert that plan `p` meets the guarantee; return its max redundant count.

    Every rank receives exactly C rows as contiguous segments from row 0; every
    expert's tokens 0 .. counts[e]-1 are covered exactly once; a rank holds
    an expert at most once; and no rank holds more than E/R non-home experts.
    """
    c = [int(v) for v in np.asarray(counts, dtype=np.int64)]
    E = len(c)
    m = E // R
    seg = p["seg"]
    assert sorted(i for r in range(R) for i in range(p["rank_begin"][r], p["rank_begin"][r] + p["rank_nseg"][r])) \
        == list(range(len(seg))), "rank ranges do not partition the segments"
    worst = 0
    for r in range(R):
        rows, experts, red = 0, set(), 0
        for i in range(p["rank_begin"][r], p["rank_begin"][r] + p["rank_nseg"][r]):
            e, rk, src, n, dst = seg[i]
            assert rk == r and 0 <= e < E and n > 0, f"bad segment {seg[i]}"
            assert dst == rows, f"rank {r}: segment {i} starts at row {dst}, expected {rows}"
            assert e not in experts, f"rank {r} holds expert {e} twice"
            experts.add(e)
            rows += n
            red += home(e, E, R) != r
        assert rows == C, f"rank {r} receives {rows} rows, not {C}"
        assert red <= m, f"rank {r} uses {red} redundant slots > {m}"
        worst = max(worst, red)
    for e in range(E):
        ids = p["exp_seg"][p["exp_off"][e]:p["exp_off"][e + 1]]
        at = 0
        for i in ids:
            assert seg[i][0] == e
            assert seg[i][2] == at, f"expert {e}: gap or overlap at token {at}"
            at += seg[i][3]
        assert at == c[e], f"expert {e}: {at} of {c[e]} tokens placed"
    assert sum(p["exp_off"][e + 1] - p["exp_off"][e] for e in range(E)) == len(seg)
    return worst


def transport_feasible(counts, R: int, C: int, allowed) -> bool:
    """Is there x[e][r] >= 0 on the allowed (e, r) pairs with row sums counts[e]
    and column sums C?  A transportation LP; integer data give integer vertices,
    so a real solution implies an integer one."""
    from scipy.optimize import linprog

    c = np.asarray(counts, dtype=np.float64)
    E = c.size
    pairs = [(e, r) for e in range(E) for r in range(R) if allowed(e, r)]
    A = np.zeros((E + R, len(pairs)))
    for j, (e, r) in enumerate(pairs):
        A[e, j] = 1.0
        A[E + r, j] = 1.0
    b = np.concatenate([c, np.full(R, float(C))])
    res = linprog(np.zeros(len(pairs)), A_eq=A, b_eq=b, bounds=(0, None), method="highs")
    return res.status == 0


def min_redundant(counts, R: int, C: int) -> int:
    """The smallest s such that some choice of at most s redundant experts per
    rank admits a balanced plan (brute force over all choices; tiny cases)."""
    E = len(counts)
    m = E // R
    for s in range(0, E - m + 1):
        choices = [list(combinations([e for e in range(E) if home(e, E, R) != r], s)) for r in range(R)]
        for pick in product(*choices):
            sets = [set(x) for x in pick]
            if transport_feasible(counts, R, C, lambda e, r: home(e, E, R) == r or e in sets[r]):
                return s
    raise AssertionError("no balanced plan at all")


def lower_bound_counts(R: int, m: int, unit: int = 1):
    """A load where one rank's experts are idle and all others are equal.

    Every other expert holds R*unit tokens and C = (R-1)*m*unit, so the idle
    rank must fill C rows from experts of R*unit tokens: ceil((R-1)*m/R)
    redundant experts, which approaches m as R grows.  Returns (counts, C, bound).
    """
    E = R * m
    counts = [0 if home(e, E, R) == R - 1 else R * unit for e in range(E)]
    C = (R - 1) * m * unit
    return counts, C, -(-(R - 1) * m // R)


def rank_counts(idx_by_rank, E: int) -> np.ndarray:
    """cnt[q][e]: routed pairs of source rank q that select expert e."""
    cnt = np.zeros((len(idx_by_rank), E), dtype=np.int64)
    for q, idx in enumerate(idx_by_rank):
        for e in np.asarray(idx).reshape(-1):
            cnt[q, int(e)] += 1
    return cnt


def dispatch_rank(idx, q: int, cnt, p: dict):
    """Destinations of source rank q's pairs idx [S, K]: (rank, row) arrays.

    Expert e's tokens are numbered in (source rank, token) order, so rank q's
    tokens of e are numbers sum(cnt[:q, e]) onward in token order; number j
    lands in the segment of e whose source range holds j."""
    seg = p["seg"]
    idx = np.asarray(idx)
    S, K = idx.shape
    seen = np.asarray(cnt)[:q].sum(axis=0).astype(np.int64)
    rank = np.zeros((S, K), dtype=np.int32)
    row = np.zeros((S, K), dtype=np.int32)
    for s in range(S):
        for k in range(K):
            e = int(idx[s, k])
            j = int(seen[e])
            seen[e] += 1
            for i in p["exp_seg"][p["exp_off"][e]:p["exp_off"][e + 1]]:
                _, r, src, n, dst = seg[i]
                if src <= j < src + n:
                    rank[s, k], row[s, k] = r, dst + j - src
                    break
            else:
                raise AssertionError(f"token {j} of expert {e} has no segment")
    return rank, row


def dispatch(idx_by_rank, p: dict, E: int):
    """dispatch_rank for every source rank."""
    cnt = rank_counts(idx_by_rank, E)
    return [dispatch_rank(idx, q, cnt, p) for q, idx in enumerate(idx_by_rank)]


def send_counts(cnt, p: dict) -> np.ndarray:
    """sends[q][r]: pairs source rank q sends to rank r, from the overlap of
    q's number range of each expert with that expert's segments (no per-token
    walk).  Row sums are S*K, column sums C."""
    cnt = np.asarray(cnt, dtype=np.int64)
    R, E = cnt.shape
    base = np.concatenate([np.zeros((1, E), np.int64), np.cumsum(cnt, axis=0)])
    out = np.zeros((R, R), dtype=np.int64)
    for e in range(E):
        for i in p["exp_seg"][p["exp_off"][e]:p["exp_off"][e + 1]]:
            _, r, src, n, _ = p["seg"][i]
            for q in range(R):
                lo, hi = max(src, base[q, e]), min(src + n, base[q + 1, e])
                if hi > lo:
                    out[q, r] += hi - lo
    return out
