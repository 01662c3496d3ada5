"""Pins of the fp64 oracle against what the sources and mathematics fix.

None of these recomputes the oracle's own loops: each check is a printed
number from the pages, a published table, a closed form, an independent
algorithm (brute force), or an invariant that a dropped term, a wrong sign or
index, or a swapped operand would break.
"""
import itertools
import math
import os

import numpy as np
import pytest

from latent_moe_layer_gb300 import synth
from oracle import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ocp_table():
    vals = {}
    with open(os.path.join(GOLDEN, "e2m1_ocp_mx_v1.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            c, v = line.split()
            vals[int(c)] = float(v)
    return vals


OCP = _ocp_table()


# ------------------------------------------------------------------ formats
def test_e2m1_matches_ocp_table():
    for code, v in OCP.items():
        got = oracle.e2m1(code)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), code


def test_e8m0_is_exact_power_of_two_full_range():
    # "Kimi K3, as released", Gate 3 section: value exactly 2^(e-127)
    for e in range(255):
        assert oracle.e8m0(e) == math.ldexp(1.0, e - 127)


def test_nibble_order_low_first():
    # byte 0x7A: low nibble 0xA (-1.0) is element 0, high nibble 0x7 (6.0) is element 1
    packed = np.zeros((1, 16), np.uint8)
    packed[0, 0] = 0x7A
    scale = np.full((1, 1), 127, np.uint8)
    d = oracle.dequant(packed, scale)
    assert d[0, 0] == -1.0 and d[0, 1] == 6.0
    assert np.all(d[0, 2:] == 0.0)


def test_dequant_every_code_and_exponent():
    # every (code pair) byte x a spread of exponents, against the OCP table x ldexp
    rng = np.random.default_rng(123)
    for e in [0, 1, 100, 118, 120, 122, 124, 127, 200, 254]:
        packed = np.arange(256, dtype=np.uint8).reshape(1, 256)   # 512 values, 16 blocks
        scale = np.full((1, 16), e, np.uint8)
        scale[0, rng.integers(0, 16)] = 127                          # one block at unit scale
        d = oracle.dequant(packed, scale)
        for k in range(512):
            byte = k // 2
            code = byte & 0xF if k % 2 == 0 else byte >> 4
            assert d[0, k] == OCP[code] * math.ldexp(1.0, int(scale[0, k // 32]) - 127)


def test_bf16_widening_is_exact():
    for bits, val in [(0x3F80, 1.0), (0xBF80, -1.0), (0x4049, 3.140625), (0x0001, 2.0 ** -133),
                      (0x7F7F, 3.3895313892515355e38)]:
        assert oracle.bf16(bits) == val


# ------------------------------------------------------------------ shape arithmetic
def test_shard_header_arithmetic():
    # "Kimi K3, as released": w1 U8 [3072,1792] scale [3072,112]; w2 U8 [3584,1536] scale [3584,96]
    cfg = synth.CONFIGS[1]
    (r1, c1), (r3, c3), (r2, c2) = synth.expert_dims(cfg)
    assert synth.packed_shape(r1, c1) == ((3072, 1792), (3072, 112))
    assert synth.packed_shape(r3, c3) == ((3072, 1792), (3072, 112))
    assert synth.packed_shape(r2, c2) == ((3584, 1536), (3584, 96))
    # 1792 bytes at 4 bits = 3584 values; 112 scales x 32 = 3584
    assert 1792 * 2 == 3584 and 112 * 32 == 3584 and 1536 * 2 == 3072 and 96 * 32 == 3072
    per_expert = 2 * (3072 * 1792 + 3072 * 112) + (3584 * 1536 + 3584 * 96)
    assert per_expert == 17_547_264
    assert round(per_expert / 1e6, 1) == 17.5                  # "17.5 MB per expert on disk"
    assert round(per_expert / 2 ** 20, 1) == 16.7              # "16.7 MB" at 4.25 b/w (MiB)
    params = 3 * 3072 * 3584
    assert params == 33_030_144                                # "33.0 M params per expert"
    assert round(per_expert * 8 / params, 2) == 4.25           # 4.25 bits/weight
    assert round(params * 896 / 1e9, 3) == 29.595              # 29.595 B per layer
    assert round(92 * 896 * params / 1e12, 2) == 2.72          # "2.72 T routed"
    assert round(82_432 * per_expert / 1e12, 2) == 1.45        # "1.44 TB over 82,432 experts"
    assert 92 * 896 == 82_432
    assert round(3 * 3072 * 7168 / 1e6, 2) == 66.06           # non-latent expert: 66.06 M
    assert round(16 * 92 * per_expert / 2 ** 30, 1) == 24.1    # "24.1 GB read/token (cold)"


def test_dequant_consumes_full_row():
    packed = np.full((1, 1792), 0x22, np.uint8)                # every code 2 (1.0)
    scale = np.full((1, 112), 127, np.uint8)
    d = oracle.dequant(packed, scale)
    assert d.shape == (1, 3584) and np.all(d == 1.0)


# ------------------------------------------------------------------ router
# Every router pin runs on both weight types: the tiny case's BF16 router and
# the fp32 router of the K3 checkpoint (the K3 workloads' branch).
ROUTERS = ["bf16", "f32"]


def _tiny(router_dtype="bf16"):
    cfg = synth.CONFIGS[0]
    if router_dtype != cfg.router_dtype:
        cfg = synth.LayerConfig(**{**cfg.__dict__, "router_dtype": router_dtype,
                                   "name": f"tiny_router_{router_dtype}"})
    dense = synth.gen_dense(cfg)
    x = synth.gen_x(cfg)
    return cfg, dense, x


def _router_f64(dense, router_dtype):
    """W_router widened to fp64 by numpy, independently of the oracle's reader."""
    if router_dtype == "bf16":
        assert dense.w_router.dtype == np.uint16
        return synth.bf16_bits_to_f32(dense.w_router).astype(np.float64)
    assert dense.w_router.dtype == np.float32
    return dense.w_router.astype(np.float64)


@pytest.mark.parametrize("router_dtype", ROUTERS)
def test_router_logits_against_matmul(router_dtype):
    cfg, dense, x = _tiny(router_dtype)
    _, _, _, lg = oracle.route(cfg, dense, x, want_logits=True)
    ref = synth.bf16_bits_to_f32(x).astype(np.float64) @ _router_f64(dense, router_dtype).T
    np.testing.assert_allclose(lg, ref, rtol=0, atol=1e-12)


def test_fp32_router_logits_at_k3_dimensions():
    # The K3 router: fp32 W [896, 7168].  The logits equal the fp64 product of the
    # fp32 weights, and that product is far (> 1e-4) from the product of the same
    # weights rounded to BF16, so reading the fp32 router at BF16 precision (or its
    # bytes as BF16 halves) fails this pin.
    cfg = synth.CONFIGS[1]
    dense = synth.DenseWeights(synth.gen_router(cfg), None, None, None, None, None)
    x = synth.gen_x(cfg)[:4]
    _, _, _, lg = oracle.route(cfg, dense, x, want_logits=True)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    ref = xf @ dense.w_router.astype(np.float64).T
    np.testing.assert_allclose(lg, ref, rtol=0, atol=1e-12)
    rounded = xf @ synth.bf16_bits_to_f32(synth.f64_to_bf16_bits(dense.w_router)).astype(np.float64).T
    assert np.abs(rounded - ref).max() > 1e-4


@pytest.mark.parametrize("router_dtype", ROUTERS)
def test_topk_against_brute_force_subsets(router_dtype):
    # all C(16,4) = 1820 subsets; the selection is the max key-sum subset, and
    # among equal sums the lexicographically lowest (lower index wins ties)
    cfg, dense, x = _tiny(router_dtype)
    rng = np.random.default_rng(7)
    xs = np.concatenate([x, synth.f64_to_bf16_bits(rng.standard_normal((56, cfg.H)))])
    idx, w, gap, lg = oracle.route(cfg, dense, xs, want_logits=True)
    subsets = list(itertools.combinations(range(cfg.E), cfg.K))
    assert len(subsets) == 1820
    for t in range(xs.shape[0]):
        best = max(subsets, key=lambda s: (sum(lg[t, j] for j in s), [-j for j in s]))
        assert sorted(idx[t]) == list(best)
        rest = sorted((lg[t, j] for j in range(cfg.E) if j not in best), reverse=True)
        assert gap[t] == pytest.approx(min(lg[t, j] for j in best) - rest[0], abs=1e-15)
        # selection order is key-descending
        assert all(lg[t, idx[t, i]] >= lg[t, idx[t, i + 1]] for i in range(cfg.K - 1))


@pytest.mark.parametrize("router_dtype", ROUTERS)
def test_ties_go_to_lowest_index(router_dtype):
    cfg, dense, x = _tiny(router_dtype)
    d = synth.DenseWeights(**dense.__dict__)
    d.w_router = np.tile(dense.w_router[:1], (cfg.E, 1))        # all logits equal
    idx, w, gap, _ = oracle.route(cfg, d, x)
    assert np.all(idx == np.arange(cfg.K)) and np.all(gap == 0.0)
    np.testing.assert_allclose(w, 1.0 / cfg.K, rtol=0, atol=1e-15)
    # one tie at the boundary: rows 9 and 3 equal and top; the lower (3) is taken first
    wr = np.zeros_like(dense.w_router)
    wr[9] = wr[3] = dense.w_router[0]
    xs = np.abs(synth.bf16_bits_to_f32(x)).astype(np.float64)
    xpos = synth.f64_to_bf16_bits(xs)
    dpos = synth.DenseWeights(**d.__dict__)
    if router_dtype == "bf16":
        dpos.w_router = synth.f64_to_bf16_bits(np.abs(synth.bf16_bits_to_f32(wr)))
    else:
        dpos.w_router = np.abs(wr)
    idx, _, _, _ = oracle.route(cfg, dpos, xpos)
    assert np.all(idx[:, 0] == 3) and np.all(idx[:, 1] == 9)
    # rest are zero logits: lowest remaining indices
    assert np.all(idx[:, 2] == 0) and np.all(idx[:, 3] == 1)


@pytest.mark.parametrize("router_dtype", ROUTERS)
def test_weights_sum_to_one_and_match_sigmoid(router_dtype):
    cfg, dense, x = _tiny(router_dtype)
    idx, w, gap, lg = oracle.route(cfg, dense, x, want_logits=True)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-12)
    s = 1 / (1 + np.exp(-np.take_along_axis(lg, idx, 1)))
    np.testing.assert_allclose(w, s / s.sum(1, keepdims=True), rtol=1e-14)


@pytest.mark.parametrize("router_dtype", ROUTERS)
def test_bias_selects_but_never_weights(router_dtype):
    cfg, dense, x = _tiny(router_dtype)
    cfgb = synth.LayerConfig(**{**cfg.__dict__, "select_bias": True})
    rng = np.random.default_rng(5)
    b = rng.standard_normal(cfg.E).astype(np.float32)
    db = synth.DenseWeights(**{**dense.__dict__, "select_bias": b})
    idx, w, gap, lg = oracle.route(cfgb, db, x, want_logits=True)
    np.testing.assert_allclose(lg, synth.bf16_bits_to_f32(x).astype(np.float64) @
                               _router_f64(dense, router_dtype).T, rtol=0, atol=1e-12)
    s = 1 / (1 + np.exp(-lg))
    key = s + b.astype(np.float64)
    for t in range(x.shape[0]):
        assert set(idx[t]) == set(np.argsort(-key[t], kind="stable")[:cfg.K])
    sel = np.take_along_axis(s, idx, 1)
    np.testing.assert_allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-14)
    # a constant shift of the bias changes neither the selection nor the weights
    db2 = synth.DenseWeights(**{**db.__dict__, "select_bias": b + np.float32(0.5)})
    idx2, w2, _, _ = oracle.route(cfgb, db2, x)
    assert np.array_equal(idx, idx2)
    np.testing.assert_allclose(w, w2, rtol=1e-14)


def test_all_experts_selected():
    cfg = synth.LayerConfig(**{**synth.CONFIGS[0].__dict__, "K": 16})
    dense = synth.gen_dense(cfg)
    x = synth.gen_x(cfg)
    idx, w, gap, lg = oracle.route(cfg, dense, x, want_logits=True)
    assert np.all(np.sort(idx, 1) == np.arange(16)) and np.all(np.isinf(gap))
    s = 1 / (1 + np.exp(-lg))
    np.testing.assert_allclose(np.take_along_axis(w, np.argsort(idx, 1), 1),
                               s / s.sum(1, keepdims=True), rtol=1e-14)


# ------------------------------------------------------------------ layer
def _tiny_experts(cfg):
    return {e: synth.gen_expert(cfg, e) for e in range(cfg.E)}


def _ocp_dequant(p, s):
    # independent numpy dequantiser built from the OCP table (not the oracle's code)
    lut = np.array([OCP[c] for c in range(16)])
    codes = np.stack([p & 0xF, p >> 4], axis=-1).reshape(p.shape[0], -1)
    scale = np.ldexp(1.0, s.astype(np.int64) - 127)
    return lut[codes] * np.repeat(scale, 32, axis=1)


def _f(b):
    return synth.bf16_bits_to_f32(b).astype(np.float64)


def test_single_expert_reduces_to_dense_glu_sandwich():
    # E = K = 1: out = W_up rmsnorm(W2 (silu(W1 h) * W3 h)), h = W_down x, weight 1
    base = synth.CONFIGS[0]
    cfg = synth.LayerConfig(**{**base.__dict__, "E": 1, "K": 1})
    dense = synth.gen_dense(cfg)
    x = synth.gen_x(cfg)
    ex = _tiny_experts(cfg)
    res = oracle.forward(cfg, dense, ex, x, want_latent=True)
    h = _f(x) @ _f(dense.w_down).T
    (p1, s1), (p3, s3), (p2, s2) = ex[0]
    W1, W3, W2 = _ocp_dequant(p1, s1), _ocp_dequant(p3, s3), _ocp_dequant(p2, s2)
    g, u = h @ W1.T, h @ W3.T
    a = g / (1 + np.exp(-g)) * u
    z = a @ W2.T
    n = z / np.sqrt((z * z).mean(1, keepdims=True) + cfg.rms_eps)
    o = n @ _f(dense.w_up).T
    assert np.all(res["idx"] == 0) and np.all(res["w"] == 1.0)
    np.testing.assert_allclose(res["h"], h, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res["z"], z, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res["out"], o, rtol=1e-11, atol=1e-11)


def _worked(gate_code, up_code, down_code, flip_router=False, wu_perm=None):
    """Layer with H=L=I=32, E=2, K=1 whose output has a closed form."""
    cfg = synth.LayerConfig("worked", seed=0, wseed=0, T=1, H=32, L=32, E=2, K=1, I=32,
                            router_dtype="bf16")
    x = np.zeros((1, 32), np.uint16)
    x[0, 0] = 0x3F80                                   # x = e_0
    wr = np.zeros((2, 32), np.uint16)
    wr[0 if flip_router else 1, 0] = 0x3F80            # logit 1 for the chosen expert, 0 else
    wd = np.zeros((32, 32), np.uint16)
    np.fill_diagonal(wd, 0x3F80)                       # h = x
    wu = np.zeros((32, 32), np.uint16)
    perm = np.arange(32) if wu_perm is None else wu_perm
    wu[np.arange(32), perm] = 0x3F80                   # out[r] = n[perm[r]]
    gamma = np.full(32, 0x3F80, np.uint16)
    dense = synth.DenseWeights(wr, None, wd, wu, gamma, None)

    def mat(code):
        return (np.full((32, 16), code | (code << 4), np.uint8), np.full((32, 1), 127, np.uint8))

    e = 0 if flip_router else 1
    experts = {e: [mat(gate_code), mat(up_code), mat(down_code)]}
    return cfg, dense, experts, x


def _sig(v):
    return 1 / (1 + math.exp(-v))


@pytest.mark.parametrize("gate,up,down,flip", [(2, 4, 2, False), (4, 2, 2, True),
                                               (2, 4, 10, False), (9, 7, 3, False)])
def test_worked_example_closed_form(gate, up, down, flip):
    # h = e_0; g_r = E2M1(gate) (row sum against e_0 picks column 0), u_r = E2M1(up),
    # a = silu(g) u for all 32 rows; y_r = 32 * E2M1(down) * a; z = y (weight 1);
    # rmsnorm of a constant vector c: c / sqrt(c^2 + eps); W_up = identity.
    cfg, dense, experts, x = _worked(gate, up, down, flip)
    res = oracle.forward(cfg, dense, experts, x)
    g, u, dn = OCP[gate], OCP[up], OCP[down]
    a = g * _sig(g) * u
    c = 32 * dn * a
    want = c / math.sqrt(c * c + 1e-6)
    assert res["idx"][0, 0] == (0 if flip else 1) and res["w"][0, 0] == 1.0
    np.testing.assert_allclose(res["out"][0], want, rtol=1e-14)


def test_worked_example_gate_up_roles_differ():
    # swapping which matrix is the gate changes the result: silu(1)*2 vs silu(2)*1
    o1 = oracle.forward(*_worked(2, 4, 2)[:3], _worked(2, 4, 2)[3])["out"][0, 0]
    o2 = oracle.forward(*_worked(4, 2, 2)[:3], _worked(4, 2, 2)[3])["out"][0, 0]
    assert o1 == pytest.approx(1.0, abs=1e-6) and o2 == pytest.approx(1.0, abs=1e-6)
    cfg, dense, ex, x = _worked(2, 4, 2)
    cfg2, dense2, ex2, x2 = _worked(4, 2, 2)
    # before the norm the two differ by silu(1)*2 / (silu(2)*1)
    r1 = oracle.forward(cfg, dense, ex, x, want_latent=True)["z"][0, 0]
    r2 = oracle.forward(cfg2, dense2, ex2, x2, want_latent=True)["z"][0, 0]
    assert r1 / r2 == pytest.approx((1 * _sig(1) * 2) / (2 * _sig(2) * 1), rel=1e-14)


def test_up_projection_orientation():
    perm = np.roll(np.arange(32), 5)
    cfg, dense, ex, x = _worked(9, 7, 3, wu_perm=perm)     # negative gate code -> varied signs
    res = oracle.forward(cfg, dense, ex, x, want_latent=True)
    z = res["z"][0]
    n = z / math.sqrt((z * z).mean() + 1e-6)
    np.testing.assert_allclose(res["out"][0], n[perm], rtol=1e-14)


def test_norm_sits_between_combine_and_up_projection():
    # scaling every w2 scale by 2 doubles z; RMSNorm removes it (up to eps)
    cfg, dense, x = _tiny()
    ex = _tiny_experts(cfg)
    ex2 = {e: [m[0], m[1], (m[2][0], m[2][1] + 1)] for e, m in ex.items()}
    r1 = oracle.forward(cfg, dense, ex, x, want_latent=True)
    r2 = oracle.forward(cfg, dense, ex2, x, want_latent=True)
    np.testing.assert_allclose(r2["z"], 2 * r1["z"], rtol=1e-14)
    np.testing.assert_allclose(r2["out"], r1["out"], rtol=1e-5, atol=1e-6)
    assert not np.allclose(r2["out"], r1["out"], rtol=0, atol=0)
    # unit RMS of the normalised latent: recover n from out through W_up's pseudo-inverse
    z = r1["z"]
    rms = np.sqrt((z * z).mean(1))
    n = z / np.sqrt(rms[:, None] ** 2 + cfg.rms_eps)
    np.testing.assert_allclose(np.sqrt((n * n).mean(1)), rms / np.sqrt(rms ** 2 + cfg.rms_eps))
    np.testing.assert_allclose(r1["out"], n @ _f(dense.w_up).T, rtol=1e-11, atol=1e-11)


def test_combine_is_weighted_sum_of_expert_outputs():
    # z_t = sum_k w_tk y_{e_tk}(h_t), each y from an independent numpy dequant of the expert
    cfg, dense, x = _tiny()
    ex = _tiny_experts(cfg)
    res = oracle.forward(cfg, dense, ex, x, want_latent=True)
    assert cfg.K == 4 and not np.allclose(res["w"], res["w"][:, :1])
    for t in range(cfg.T):
        h = res["h"][t]
        z = np.zeros(cfg.L)
        for k in range(cfg.K):
            (p1, s1), (p3, s3), (p2, s2) = ex[int(res["idx"][t, k])]
            g, u = _ocp_dequant(p1, s1) @ h, _ocp_dequant(p3, s3) @ h
            z += res["w"][t, k] * (_ocp_dequant(p2, s2) @ (g / (1 + np.exp(-g)) * u))
        np.testing.assert_allclose(res["z"][t], z, rtol=1e-12, atol=1e-12)


def test_norm_gain_multiplies_the_normalised_latent():
    # routed_expert_norm's gain gamma scales n elementwise before the up-projection
    cfg, dense, x = _tiny()
    ex = _tiny_experts(cfg)
    gam = synth.f64_to_bf16_bits(np.random.default_rng(2).uniform(0.5, 2.0, cfg.L))
    d2 = synth.DenseWeights(**{**dense.__dict__, "gamma": gam})
    r = oracle.forward(cfg, d2, ex, x, want_latent=True)
    z = r["z"]
    n = z / np.sqrt((z * z).mean(1, keepdims=True) + cfg.rms_eps) * _f(gam)
    np.testing.assert_allclose(r["out"], n @ _f(dense.w_up).T, rtol=1e-11, atol=1e-11)


def test_token_permutation_and_batch_invariance():
    cfg, dense, x = _tiny()
    ex = _tiny_experts(cfg)
    r = oracle.forward(cfg, dense, ex, x)
    perm = np.random.default_rng(3).permutation(cfg.T)
    rp = oracle.forward(cfg, dense, ex, x[perm])
    np.testing.assert_allclose(rp["out"], r["out"][perm], rtol=1e-13, atol=1e-13)
    r1 = oracle.forward(cfg, dense, ex, x[5:6])
    np.testing.assert_allclose(r1["out"][0], r["out"][5], rtol=1e-13, atol=1e-13)


def test_expert_relabelling_invariance():
    cfg, dense, x = _tiny()
    ex = _tiny_experts(cfg)
    r = oracle.forward(cfg, dense, ex, x)
    perm = np.random.default_rng(11).permutation(cfg.E)      # new label j holds old expert perm[j]
    d2 = synth.DenseWeights(**{**dense.__dict__, "w_router": dense.w_router[perm]})
    ex2 = {j: ex[int(perm[j])] for j in range(cfg.E)}
    r2 = oracle.forward(cfg, d2, ex2, x)
    np.testing.assert_allclose(r2["out"], r["out"], rtol=1e-13, atol=1e-13)
    assert np.array_equal(np.sort(perm[r2["idx"]], 1), np.sort(r["idx"], 1))


def test_shared_experts_add_a_full_width_glu():
    # with shared experts the output gains W2s (silu(W1s x) * W3s x), independent of routing
    cfg0 = synth.CONFIGS[0]
    cfg = cfg0.with_shared(64)
    dense = synth.gen_dense(cfg)
    x = synth.gen_x(cfg)
    ex = _tiny_experts(cfg)
    r_sh = oracle.forward(cfg, dense, ex, x)
    r_no = oracle.forward(cfg0, dense, ex, x)
    (p1, s1), (p3, s3), (p2, s2) = dense.shared
    xf = _f(x)
    g, u = xf @ _ocp_dequant(p1, s1).T, xf @ _ocp_dequant(p3, s3).T
    ys = (g / (1 + np.exp(-g)) * u) @ _ocp_dequant(p2, s2).T
    np.testing.assert_allclose(r_sh["out"] - r_no["out"], ys, rtol=1e-11, atol=1e-10)


def test_missing_expert_is_reported():
    cfg, dense, x = _tiny()
    with pytest.raises(KeyError):
        oracle.forward(cfg, dense, {}, x)
