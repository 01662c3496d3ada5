"""The allocation-free routing entry point (k3moe_route_static).

It serves callers that cannot allocate device memory (plugin hosts that give
an operator only its input and output buffers): its logits scratch is a static
device array inside the library.  Checked through the C ABI, on two calls in a
row with different inputs (a stale scratch from the first call would show in
the second), against the routing that k3moe_forward returns and against the
fp64 oracle under the parity rule (index sets and order where the key gaps are
>= 1e-4, weights within 1e-5); and the device memory in use must not change
across calls after the first.  This file is collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest

from latent_moe_layer_gb300 import synth
from oracle import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from latent_moe_layer_gb300 import k3moe  # noqa: E402
from parity_util import GAP, index_check, selection_gaps  # noqa: E402

W_TOL = 1e-5          # the mixture-weight tolerance of the parity tests
MAX_LOGITS = 256 * 1024

# K3 router dimensions (7168 hidden, 896 experts, top-16, fp32 router) with small
# experts, so the weights are cheap to draw; and the tiny case with a BF16
# router plus a selection bias.
K3_ROUTER = synth.LayerConfig("k3_router_small_experts", seed=21, wseed=21, T=48, H=7168, L=32,
                              E=896, K=16, I=32)
TINY_BIAS = synth.LayerConfig("tiny_bias", seed=22, wseed=22, T=40, H=256, L=128, E=16, K=4, I=96,
                              exp_lo=120, exp_hi=124, router_dtype="bf16", select_bias=True)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _route_static(layer, x, T, idx, w):
    L = k3moe.lib()
    L.k3moe_route_static.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_void_p, C.c_void_p,
                                     C.c_void_p]
    L.k3moe_route_static.restype = C.c_int
    return L.k3moe_route_static(layer.h, x.data_ptr() if x is not None else None, T,
                                idx.data_ptr(), w.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _inputs(cfg, T, seed):
    x = synth.gen_x(synth.LayerConfig(**{**cfg.__dict__, "seed": seed, "T": T}))
    return torch.from_numpy(x.view(np.int16)).cuda()


@pytest.mark.parametrize("cfg", [K3_ROUTER, TINY_BIAS], ids=["k3_router", "tiny_bias"])
def test_route_static_matches_forward_two_calls(cfg):
    dense = synth.gen_dense(cfg)
    if cfg.select_bias:
        dense.select_bias = np.random.default_rng(3).uniform(-0.3, 0.3, cfg.E).astype(np.float32)
    dw = k3moe.DeviceWeights(cfg, dense=dense)
    layer = k3moe.Layer(cfg)
    layer.load(dw)
    calls = [(cfg.T, 100), (16, 200)]          # two calls in a row, different sizes and tokens
    refs = []
    for T, seed in calls:
        x = _inputs(cfg, T, seed)
        idx = torch.empty((T, cfg.K), dtype=torch.int32, device="cuda")
        w = torch.empty((T, cfg.K), dtype=torch.float32, device="cuda")
        layer.forward(x, idx_out=idx, w_out=w)
        refs.append((x, idx.cpu().numpy(), w.cpu().numpy()))
    outs = [(torch.empty((T, cfg.K), dtype=torch.int32, device="cuda"),
             torch.empty((T, cfg.K), dtype=torch.float32, device="cuda")) for T, _ in calls]
    # a first call on this device resolves the static array's address; from
    # then on the calls must leave the device's memory use unchanged
    for (T, _), (x, _, _), (idx, w) in zip(calls, refs, outs):
        assert _route_static(layer, x, T, idx, w) == 0
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for (T, _), (x, ridx, rw), (idx, w) in zip(calls, refs, outs):
        idx.fill_(-1)
        w.fill_(-1.0)
        assert _route_static(layer, x, T, idx, w) == 0
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0 and torch.cuda.memory_allocated() == alloc0
        g_idx, g_w = idx.cpu().numpy(), w.cpu().numpy()
        # against the oracle: the parity rule on index sets, order and weights
        x_np = x.cpu().numpy().view(np.uint16)
        o_idx, o_w, gap, lg = oracle.route(cfg, dense, x_np, want_logits=True)
        set_bad, order_bad, _, _ = index_check(g_idx, o_idx, gap, selection_gaps(cfg, dense, o_idx, lg))
        assert not set_bad and not order_bad, (set_bad, order_bad)
        for t in np.nonzero(gap >= GAP)[0]:
            pos = {int(e): k for k, e in enumerate(o_idx[t])}
            assert max(abs(g_w[t, k] - o_w[t, pos[int(e)]]) for k, e in enumerate(g_idx[t])) <= W_TOL
        # and the forward's routing on the same tokens (same rule: the two logit
        # paths differ by about 1e-6, so only near-ties may differ)
        f_bad, f_order, _, _ = index_check(g_idx, ridx, gap, selection_gaps(cfg, dense, o_idx, lg))
        assert not f_bad and not f_order
        keep = gap >= GAP
        assert np.abs(g_w[keep] - rw[keep]).max() <= W_TOL
    assert layer.status() == 0


def test_route_static_rejects_sizes_beyond_its_scratch():
    cfg = K3_ROUTER
    dw = k3moe.DeviceWeights(cfg)
    layer = k3moe.Layer(cfg)
    layer.load(dw)
    T = MAX_LOGITS // cfg.E + 1                 # one token past the static capacity
    x = _inputs(cfg, T, 300)
    idx = torch.empty((T, cfg.K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, cfg.K), dtype=torch.float32, device="cuda")
    assert _route_static(layer, x, T, idx, w) == k3moe.ERR_CODE["WORKSPACE"]
    T_ok = MAX_LOGITS // cfg.E                  # exactly at capacity is accepted
    assert _route_static(layer, x, T_ok, idx, w) == 0
    torch.cuda.synchronize()
    assert layer.status() == 0
