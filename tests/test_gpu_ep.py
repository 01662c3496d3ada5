"""GPU parity of the balanced expert-parallel plan and dispatch
(k3moe_ep_plan_compute, k3moe_ep_dispatch) against the oracle
(oracle/ep_plan.py): the plan bit-exact (the same greedy and tie-breaks) and
valid by the oracle's checker of the guarantee; every destination bit-exact,
and every receive row of every rank filled exactly once."""
import numpy as np
import pytest

from latent_moe_layer_gb300 import synth
from oracle import ep_plan as ep

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from latent_moe_layer_gb300 import k3moe  # noqa: E402

RANGE = -10


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


_LAYERS = {}


def _layer(E, K):
    """A loaded handle with E experts and top-K (tiny expert shapes: the plan
    uses only E, K and the status word)."""
    if (E, K) not in _LAYERS:
        cfg = synth.LayerConfig(f"ep_E{E}_K{K}", seed=5, wseed=5, T=8, H=256, L=128, E=E, K=K, I=96,
                                exp_lo=120, exp_hi=124, router_dtype="bf16")
        layer = k3moe.Layer(cfg)
        layer.load(k3moe.DeviceWeights(cfg))
        _LAYERS[(E, K)] = layer
    return _LAYERS[(E, K)]


def _routing(rng, R, S, K, E, skew):
    """Per-rank top-K expert ids (distinct per token) from a seeded Zipf-like law."""
    w = 1.0 / np.arange(1, E + 1) ** skew
    p = rng.permutation(w / w.sum())
    out = []
    for _ in range(R):
        # Gumbel top-K: K distinct experts per token, drawn with weights p
        g = np.log(p)[None, :] - np.log(-np.log(rng.random((S, E)) + 1e-300))
        out.append(np.ascontiguousarray(np.argpartition(-g, K - 1, axis=1)[:, :K]).astype(np.int32))
    return out


def _gpu_plan(layer, cnt, S):
    plan = layer.ep_plan(torch.from_numpy(np.ascontiguousarray(cnt, dtype=np.int32)).cuda(), S)
    torch.cuda.synchronize()
    return plan


def _as_dict(plan, R, E):
    n = int(plan["info"][0])
    seg = [tuple(int(v) for v in row) for row in plan["seg"][:n].cpu().numpy()]
    rs = plan["rank_seg"].cpu().numpy()
    return dict(seg=seg, rank_begin=[int(v) for v in rs[:, 0]], rank_nseg=[int(v) for v in rs[:, 1]],
                exp_off=[int(v) for v in plan["exp_off"].cpu().numpy()],
                exp_seg=[int(v) for v in plan["exp_seg"][:n].cpu().numpy()],
                max_redundant=int(plan["info"][1]))


def _assert_plan(layer, cnt, R, S, K):
    E = cnt.shape[1]
    tot = cnt.sum(axis=0)
    got = _as_dict(_gpu_plan(layer, cnt, S), R, E)
    assert layer.status() == 0
    want = ep.plan(tot, R, S * K)
    assert got["seg"] == want["seg"]
    for k in ("rank_begin", "rank_nseg", "exp_off", "exp_seg", "max_redundant"):
        assert got[k] == want[k], k
    assert ep.check_plan(got, tot, R, S * K) == got["max_redundant"] <= E // R
    return got


PLAN_CASES = [  # E, K, R, S, skew
    (896, 16, 8, 64, 1.2), (896, 16, 64, 16, 0.0), (896, 16, 2, 512, 2.5), (896, 16, 1, 16, 0.0),
    (896, 16, 896, 2, 1.0), (24, 4, 3, 40, 1.5), (24, 4, 24, 7, 1.0), (1024, 8, 1024, 4, 1.1),
    (1024, 8, 16, 300, 3.0),
]


@pytest.mark.parametrize("E,K,R,S,skew", PLAN_CASES)
def test_plan_matches_oracle(E, K, R, S, skew):
    rng = np.random.default_rng(E + K + R + S)
    cnt = np.stack([np.bincount(i.ravel(), minlength=E) for i in _routing(rng, R, S, K, E, skew)])
    _assert_plan(_layer(E, K), cnt, R, S, K)


@pytest.mark.parametrize("R,m", [(8, 112), (4, 224), (56, 16)])
def test_plan_on_the_lower_bound_family(R, m):
    """One rank idle, all other experts equal: the idle rank takes exactly
    ceil((R-1) m / R) experts."""
    K = 16
    E = R * m
    counts, C, bound = ep.lower_bound_counts(R, m, unit=K)
    S = C // K
    cnt = np.zeros((R, E), np.int64)
    cnt[0] = counts                      # any split over source ranks: the plan sees the totals
    got = _assert_plan(_layer(E, K), cnt, R, S, K)
    assert got["max_redundant"] == bound


def test_plan_all_load_on_one_expert():
    E, K, R, S = 896, 16, 8, 32
    cnt = np.zeros((R, E), np.int64)
    cnt[3, 5] = R * S * K
    got = _assert_plan(_layer(E, K), cnt, R, S, K)
    assert sum(1 for s in got["seg"] if s[0] == 5) == R


DISPATCH_CASES = [  # E, K, R, S, skew
    (896, 16, 8, 128, 1.2), (896, 16, 4, 1000, 0.0), (896, 16, 2, 40, 2.0), (24, 4, 3, 33, 1.5),
    (24, 4, 1, 70, 0.0), (1024, 8, 16, 64, 1.1),
]


def _dispatch_all(layer, idx, cnt, plan):
    cnt_t = torch.from_numpy(np.ascontiguousarray(cnt, dtype=np.int32)).cuda()
    out = []
    for q, i in enumerate(idx):
        rank, row = layer.ep_dispatch(torch.from_numpy(i).cuda(), q, cnt_t, plan)
        out.append((rank.cpu().numpy(), row.cpu().numpy()))
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("E,K,R,S,skew", DISPATCH_CASES)
def test_dispatch_matches_oracle(E, K, R, S, skew):
    rng = np.random.default_rng(7 * E + R + S)
    layer = _layer(E, K)
    idx = _routing(rng, R, S, K, E, skew)
    cnt = ep.rank_counts(idx, E)
    plan = _gpu_plan(layer, cnt, S)
    got = _dispatch_all(layer, idx, cnt, plan)
    assert layer.status() == 0
    p = _as_dict(plan, R, E)
    want = ep.dispatch(idx, p, E)
    for (gr, gw), (wr, ww) in zip(got, want):
        assert np.array_equal(gr, wr) and np.array_equal(gw, ww)
    # every receive row of every rank exactly once, holding the planned expert
    held = np.full((R, S * K), -1)
    for e, r, _, n, dst in p["seg"]:
        held[r, dst:dst + n] = e
    hits = np.zeros((R, S * K), np.int64)
    for q, (rk, rw) in enumerate(got):
        np.add.at(hits, (rk.ravel(), rw.ravel()), 1)
        assert np.array_equal(held[rk.ravel(), rw.ravel()], idx[q].ravel())
    assert (hits == 1).all()


def test_dispatch_full_size_by_properties():
    """8 ranks of 8192 tokens, top-16 of 896 experts (1M routed pairs): the
    destinations fill every rank's 131072 rows exactly once with the planned
    experts, and the per-destination sizes equal the plan's send counts."""
    E, K, R, S = 896, 16, 8, 8192
    rng = np.random.default_rng(11)
    layer = _layer(E, K)
    idx = _routing(rng, R, S, K, E, 1.0)
    cnt = np.stack([np.bincount(i.ravel(), minlength=E) for i in idx])
    plan = _gpu_plan(layer, cnt, S)
    got = _dispatch_all(layer, idx, cnt, plan)
    assert layer.status() == 0
    p = _as_dict(plan, R, E)
    assert ep.check_plan(p, cnt.sum(axis=0), R, S * K) <= E // R
    held = np.full((R, S * K), -1)
    for e, r, _, n, dst in p["seg"]:
        held[r, dst:dst + n] = e
    hits = np.zeros((R, S * K), np.int64)
    sends = np.zeros((R, R), np.int64)
    for q, (rk, rw) in enumerate(got):
        np.add.at(hits, (rk.ravel(), rw.ravel()), 1)
        assert np.array_equal(held[rk.ravel(), rw.ravel()], idx[q].ravel())
        sends[q] = np.bincount(rk.ravel(), minlength=R)
    assert (hits == 1).all()
    assert np.array_equal(sends, ep.send_counts(cnt, p))
    # sampled pairs against the oracle's numbering: rank 5's pairs in token order
    q = 5
    seen = cnt[:q].sum(axis=0)
    for s in range(0, S, 997):
        for k in range(K):
            e = int(idx[q][s, k])
            j = int(seen[e] + np.count_nonzero(idx[q][:s] == e))
            for i in p["exp_seg"][p["exp_off"][e]:p["exp_off"][e + 1]]:
                _, r, src, n, dst = p["seg"][i]
                if src <= j < src + n:
                    assert (got[q][0][s, k], got[q][1][s, k]) == (r, dst + j - src)
                    break
            else:
                raise AssertionError("no segment")


def test_device_errors_are_reported():
    E, K, R, S = 24, 4, 3, 10
    layer = _layer(E, K)
    rng = np.random.default_rng(3)
    idx = _routing(rng, R, S, K, E, 1.0)
    cnt = ep.rank_counts(idx, E)
    bad = cnt.copy()
    bad[1, 2] += 1                            # one pair too many: the sum is not R*S*K
    plan = _gpu_plan(layer, bad, S)
    assert layer.status() == RANGE
    assert plan["info"].cpu().tolist() == [0, -1]
    assert layer.status() == 0                # read and cleared
    # a dispatch under the failed plan reads none of its other buffers: every pair -1
    rank, row = layer.ep_dispatch(torch.from_numpy(idx[0]).cuda(), 0, torch.from_numpy(bad.astype(np.int32)).cuda(),
                                  plan)
    assert layer.status() == RANGE
    assert (rank.cpu().numpy() == -1).all() and (row.cpu().numpy() == -1).all()
    plan = _gpu_plan(layer, cnt, S)
    assert layer.status() == 0
    wrong = [i.copy() for i in idx]
    wrong[0][4, 1] = E                       # an expert id outside [0, E)
    rank, row = layer.ep_dispatch(torch.from_numpy(wrong[0]).cuda(), 0,
                                  torch.from_numpy(cnt.astype(np.int32)).cuda(), plan)
    assert layer.status() == RANGE
    assert int(rank[4, 1]) == -1 and int(row[4, 1]) == -1
