"""GPU parity of the Quantile-Balancing bias update (k3moe_qb_bias) against the
fp64 oracle (oracle/qb.py), on seeded synthetic router logits."""
import numpy as np
import pytest

from latent_moe_layer_gb300 import synth
from oracle import qb

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from latent_moe_layer_gb300 import k3moe  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _layer(E, K):
    d = dict(synth.SMALL_ALIGNED.__dict__)
    d.update(E=E, K=K, name=f"qb_E{E}_K{K}")
    return k3moe.Layer(synth.LayerConfig(**d))


def _inputs(T, E, seed, skew=0.0):
    rng = np.random.default_rng(seed)
    l = rng.standard_normal((T, E)) * 1.5 + skew * np.linspace(-1, 1, E)[None, :]
    b = rng.standard_normal(E) * 0.02
    return l.astype(np.float32), b.astype(np.float32)


def _gpu(layer, l, b, nbins):
    out = layer.qb_bias(torch.from_numpy(l).cuda(), None if b is None else torch.from_numpy(b).cuda(), nbins)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("T,E,K", [(2048, 96, 8), (8192, 896, 16), (300, 16, 4), (32768, 896, 16)])
def test_within_one_bin_of_the_exact_quantile(T, E, K):
    l, b = _inputs(T, E, seed=T + E)
    got = _gpu(_layer(E, K), l, b, 1000)
    l64, b64 = l.astype(np.float64), b.astype(np.float64)
    exact_r = qb.rth_margin(l64, b64, K)
    mg = qb.margins(qb.scores(l64), b64, K)
    w = (mg.max() - mg.min()) / 1000
    d = got - exact_r
    # the estimate is the upper edge of the bin holding the r-th margin; fp32
    # margins move the order statistic by ~1e-7 at most
    assert np.all(d >= -1e-5) and np.all(d <= w + 1e-5), (d.min(), d.max(), w)


def test_repeatable_and_in_place():
    l, b = _inputs(4096, 128, seed=3)
    layer = _layer(128, 8)
    lt, bt = torch.from_numpy(l).cuda(), torch.from_numpy(b).cuda()
    a1 = layer.qb_bias(lt, bt).cpu().numpy()
    a2 = layer.qb_bias(lt, bt).cpu().numpy()
    assert a1.tobytes() == a2.tobytes()
    # bias_out may be bias_in
    L = k3moe.lib()
    n = L.k3moe_qb_workspace_bytes(layer.h, 4096, 1000)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    inout = bt.clone()
    s = torch.cuda.current_stream().cuda_stream
    assert L.k3moe_qb_bias(layer.h, lt.data_ptr(), 4096, inout.data_ptr(), inout.data_ptr(), 1000,
                           ws.data_ptr(), n, s) == 0
    assert inout.cpu().numpy().tobytes() == a1.tobytes()


def test_balances_a_skewed_router():
    T, E, K = 8192, 64, 4
    l, _ = _inputs(T, E, seed=11, skew=3.0)
    zero = np.zeros(E, np.float32)
    got = _gpu(_layer(E, K), l, zero, 1000)
    s = qb.scores(l.astype(np.float64))

    def load(bias):
        alpha = qb.thresholds(s, bias, K)
        return (s + bias[None, :] > alpha[:, None]).sum(axis=0)

    q = T * K / E
    before, after = np.abs(load(np.zeros(E)) - q).max(), np.abs(load(got) - q).max()
    assert after < 0.1 * before, (before, after)


def test_degenerate_cases():
    # one bin: every expert gets the largest margin of the batch
    l, b = _inputs(500, 32, seed=5)
    got = _gpu(_layer(32, 4), l, b, 1)
    mg = qb.margins(qb.scores(l.astype(np.float64)), b.astype(np.float64), 4)
    assert np.allclose(got, mg.max(), atol=1e-5)
    # top_k + 1 = n_experts: the threshold is each token's smallest key; no bias given
    l, _ = _inputs(256, 16, seed=6)
    got = _gpu(_layer(16, 15), l, None, 1000)
    exact_r = qb.rth_margin(l.astype(np.float64), np.zeros(16), 15)
    mg = qb.margins(qb.scores(l.astype(np.float64)), np.zeros(16), 15)
    w = (mg.max() - mg.min()) / 1000
    assert np.all(got - exact_r >= -1e-5) and np.all(got - exact_r <= w + 1e-5)
    # two tokens (r = 1)
    l, b = _inputs(2, 16, seed=7)
    got = _gpu(_layer(16, 2), l, b, 1000)
    exact_r = qb.rth_margin(l.astype(np.float64), b.astype(np.float64), 2)
    mg = qb.margins(qb.scores(l.astype(np.float64)), b.astype(np.float64), 2)
    w = (mg.max() - mg.min()) / 1000
    assert np.all(got - exact_r >= -1e-5) and np.all(got - exact_r <= w + 1e-5)


def test_errors():
    layer = _layer(16, 4)
    L = k3moe.lib()
    l = torch.zeros((8, 16), dtype=torch.float32, device="cuda")
    out = torch.empty(16, dtype=torch.float32, device="cuda")
    n = L.k3moe_qb_workspace_bytes(layer.h, 8, 1000)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    E = k3moe.ERR_CODE
    assert L.k3moe_qb_bias(layer.h, l.data_ptr(), 1, None, out.data_ptr(), 1000, ws.data_ptr(), n, s) == E["ARG"]
    assert L.k3moe_qb_bias(layer.h, l.data_ptr(), 8, None, out.data_ptr(), 0, ws.data_ptr(), n, s) == E["ARG"]
    assert L.k3moe_qb_bias(layer.h, l.data_ptr(), 8, None, out.data_ptr(), 9000, ws.data_ptr(), n, s) == E["ARG"]
    assert L.k3moe_qb_bias(layer.h, l.data_ptr(), 8, None, out.data_ptr(), 1000, ws.data_ptr(), 64, s) == E["WORKSPACE"]
    assert L.k3moe_qb_bias(layer.h, None, 8, None, out.data_ptr(), 1000, ws.data_ptr(), n, s) == E["ARG"]
    full = _layer(16, 16)
    assert L.k3moe_qb_bias(full.h, l.data_ptr(), 8, None, out.data_ptr(), 1000, ws.data_ptr(), n, s) == E["UNSUPPORTED"]
    assert L.k3moe_qb_workspace_bytes(layer.h, 1, 1000) == 0
