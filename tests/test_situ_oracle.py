"""Pins of the oracle's SiTU-GLU reading (oracle/k3moe_oracle.c, step 5).

The pages print no SiTU formula.  "Kimi K3, as released" (section "What is new
since Kimi-Linear", item 3) gives the name (Sigmoid Tanh Unit) and its two
constants (activation_situ_beta 4, activation_situ_linear_beta 25); the K3
report review (section "SiTU-GLU is a soft fuse") states that sigmoid and tanh
soft-limit the two GLU branches, that every output coordinate is bounded by
100, and that beta tanh(z / beta) = z + O(z^3 / beta^2) makes the unit locally
SwiGLU.  These tests check exactly those statements -- the bound, the
small-argument expansion against SwiGLU (which also fixes which branch takes
which beta) and the saturation limits -- so the reading is pinned only as far
as the pages go ("parity unpinned" beyond them).
"""
import numpy as np

from latent_moe_layer_gb300 import synth
from oracle import oracle

B1, B2 = 4.0, 25.0


def _sig(x):
    return 1.0 / (1.0 + np.exp(-x))


def test_every_coordinate_is_bounded_by_100():
    rng = np.random.default_rng(1)
    g = np.concatenate([rng.standard_normal(2000) * 10 ** rng.uniform(-3, 6, 2000),
                        [1e300, -1e300, 1e6, -1e6, 0.0]])
    u = np.concatenate([rng.standard_normal(2000) * 10 ** rng.uniform(-3, 6, 2000),
                        [1e300, 1e300, -1e6, 1e6, 1e9]])
    a = oracle.act("situ", g, u)
    assert np.all(np.isfinite(a)) and np.all(np.abs(a) <= B1 * B2)
    # SwiGLU itself is unbounded on the same inputs
    assert np.abs(oracle.act("silu", g[:2000], u[:2000])).max() > 1e6


def test_locally_swiglu_with_the_stated_error_order():
    # beta tanh(z / beta) = z - z^3 / (3 beta^2) + O(z^5): the SiTU-GLU minus SwiGLU
    # difference has the leading term -sigmoid(g) g u (g^2 / (3 B1^2) + u^2 / (3 B2^2))
    for g, u in [(0.02, 0.01), (-0.015, 0.03), (0.01, -0.04), (0.005, 0.005)]:
        d = oracle.act("situ", g, u) - oracle.act("silu", g, u)
        lead = -_sig(g) * g * u * (g * g / (3 * B1 * B1) + u * u / (3 * B2 * B2))
        assert abs(d / lead - 1.0) < 2e-3, (g, u, d, lead)
    # relative gap to SwiGLU shrinks as z^2 / beta^2
    r = [abs(oracle.act("situ", z, z) / oracle.act("silu", z, z) - 1.0) for z in (0.4, 0.2, 0.1)]
    assert 3.5 < r[0] / r[1] < 4.5 and 3.5 < r[1] / r[2] < 4.5


def test_saturation_limits_of_each_branch():
    # gate branch -> beta (g -> +inf) or 0 (g -> -inf); up branch -> +-linear beta
    assert abs(oracle.act("situ", 60.0, 1e6) - B1 * B2) < 1e-9
    assert abs(oracle.act("situ", 60.0, -1e6) + B1 * B2) < 1e-9
    assert abs(oracle.act("situ", -60.0, 1e6)) < 1e-20
    for g in (-2.0, 0.5, 3.0):
        assert abs(oracle.act("situ", g, 1e6) - B2 * _sig(g) * B1 * np.tanh(g / B1)) < 1e-12
    for u in (-7.0, 0.3, 40.0):
        assert abs(oracle.act("situ", 60.0, u) - B1 * B2 * np.tanh(u / B2)) < 1e-9
    assert oracle.act("situ", 0.0, 5.0) == 0.0 and oracle.act("situ", 1.0, 0.0) == 0.0


def test_layer_option_reaches_the_glu():
    cfg = synth.CONFIGS[0]
    dense = synth.gen_dense(cfg)
    x = synth.gen_x(cfg)
    idx, _, _, _ = oracle.route(cfg, dense, x)
    experts = {int(e): synth.gen_expert(cfg, int(e)) for e in np.unique(idx)}
    o_silu = oracle.forward(cfg, dense, experts, x)["out"]
    o_situ = oracle.forward(cfg.with_act("situ"), dense, experts, x)["out"]
    assert np.all(np.isfinite(o_situ)) and not np.allclose(o_silu, o_situ)
