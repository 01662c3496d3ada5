"""The A8 option: pins of the oracle's MXFP8 step, and its cost against the exact layer.

The K3 report review (sections on deployment-aware post-training and on the
open weights) says the routed experts were trained and are shipped with MXFP4
weights and MXFP8 input activations.  The layer's definition, which the parity
bar is stated against, has no activation rounding.  This module measures what
rounding the expert GEMMs' two activation inputs (the latent h, and the GLU
output a) to MXFP8 would cost against that definition, using the fp64 oracle
for everything else.

MXFP8 follows the OCP Microscaling v1.0 definition: E4M3 elements (bias 7, 3
mantissa bits, subnormal spacing 2^-9, largest finite 448, conversion
saturating), one E8M0 scale per 32 elements, scale = 2^(floor(log2 amax) - 8)
(8 = E4M3's largest exponent).
"""
import numpy as np
import pytest

from latent_moe_layer_gb300 import synth
from oracle import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ------------------------------------------------------------------ MXFP8 (test-local)
def e4m3_round(v):
    """Round to the nearest E4M3 value (ties to even), saturating at +-448."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    _, e = np.frexp(np.where(a > 0, a, 1.0))    # a = m 2^e, 0.5 <= m < 1: floor(log2 a) = e - 1
    e = np.clip(e - 1, -6, 8)                      # below 2^-6 the spacing stays 2^-9 (subnormals)
    step = np.exp2(e - 3)
    q = np.rint(a / step) * step               # numpy rint: ties to even
    q = np.minimum(q, 448.0)
    return np.sign(v) * q


def e4m3_grid():
    """All finite non-negative E4M3 values, from the bit layout (s eeee mmm)."""
    vals = []
    for code in range(0x7F):                   # 0x7F is NaN
        e, m = code >> 3, code & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals)


def mxfp8(x, no_clip=False):
    """Quantise the last axis in blocks of 32 to E4M3 x 2^X (X shared per block).

    X = floor(log2 amax) - 8 (the OCP rule; the block maximum may saturate), or
    with ``no_clip`` the smallest X with amax / 2^X <= 448."""
    x = np.asarray(x, np.float64)
    b = x.reshape(*x.shape[:-1], -1, 32)
    amax = np.abs(b).max(axis=-1, keepdims=True)
    safe = np.where(amax > 0, amax, 1.0)
    X = np.ceil(np.log2(safe / 448.0)) if no_clip else np.frexp(safe)[1] - 1 - 8
    X = np.clip(X, -127, 127)
    s = np.exp2(X)
    return (e4m3_round(b / s) * s).reshape(x.shape)


def test_e4m3_rounding_pins():
    g = e4m3_grid()
    assert g.max() == 448.0 and g[1] == 2.0 ** -9 and g[8] == 2.0 ** -6
    assert np.array_equal(e4m3_round(g), g) and np.array_equal(e4m3_round(-g), -g)
    assert e4m3_round(500.0) == 448.0                     # saturating conversion
    assert e4m3_round(1 + 2 ** -4) == 1.0                 # tie -> even mantissa
    assert e4m3_round(1 + 3 * 2 ** -4) == 1.25            # tie -> even mantissa (up)
    assert e4m3_round(2.0 ** -10) == 0.0                  # half the smallest subnormal -> 0
    r = np.random.default_rng(0).standard_normal(4096) * 10
    q = e4m3_round(r)
    assert np.all(np.isin(np.abs(q), g))
    # nearest: no grid point strictly closer than the chosen one
    d = np.abs(np.abs(r)[:, None] - g[None, :]).min(axis=1)
    assert np.allclose(np.abs(np.abs(r) - np.abs(q)), d)


def test_mxfp8_block_scale():
    x = np.zeros(64)
    x[3], x[40], x[41], x[42] = 3.0, -1000.0, 0.3, 0.01
    q = mxfp8(x)
    assert q[3] == 3.0                  # block amax 3: X = 2^(1 - 8), 3 = 384 x 2^-7 exactly
    assert q[40] == -896.0              # block amax 1000: X = 2^(9 - 8), 500 saturates to 448
    assert q[41] == 0.3125              # 0.15 -> 10 x 2^-6 (normal, spacing 2^-6), x 2
    assert q[42] == 3 * 2.0 ** -9 * 2   # 0.005 -> 3 x 2^-9 (subnormal), x 2
    assert np.all(q[np.r_[0:3, 4:32]] == 0)


def test_mxfp8_scale_one_ulp_below_a_power_of_two():
    # amax = 2 - 2^-52: floor(log2 amax) = 0, so X = -8 and amax / 2^X = 512 - 2^-44
    # saturates to 448, giving 1.75.  An exponent taken from a log2 that rounded up
    # to 1.0 would give X = -7 and 2.0 instead.
    below = np.nextafter(2.0, 0.0)
    x = np.zeros(32)
    x[0], x[1] = below, 0.5
    for q in (mxfp8(x), oracle.mxfp8(x)):
        assert q[0] == 1.75 and q[1] == 0.5
    # the same one ulp below 2^-6 and 2^7: X = -14 and X = -2
    for amax, want in [(np.nextafter(2.0 ** -6, 0.0), 1.75 * 2.0 ** -7), (np.nextafter(128.0, 0.0), 112.0)]:
        x[0], x[1] = amax, 0.0
        for q in (mxfp8(x), oracle.mxfp8(x)):
            assert q[0] == want, (amax, q[0], want)
    assert oracle.e4m3(below) == 2.0 and e4m3_round(below) == 2.0


# ------------------------------------------------------------------ the layer, re-stated with hooks
def _bf16(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def _layer_from_latent(cfg, dense, experts, h, idx, w, quant, quant_h=None):
    """Experts, combine, RMSNorm and up-projection in fp64 from the oracle's latent
    h, indices and weights; ``quant`` is applied to each expert GEMM's input
    (``quant_h``, when given, to h instead)."""
    up, gamma = _bf16(dense.w_up), _bf16(dense.gamma)
    deq = {e: [oracle.dequant(p, s) for p, s in mats] for e, mats in experts.items()}
    out = np.zeros((h.shape[0], cfg.H))
    for t in range(h.shape[0]):
        z = np.zeros(cfg.L)
        hq = (quant_h or quant)(h[t])
        for k in range(cfg.K):
            w1, w3, w2 = deq[int(idx[t, k])]
            g, u = w1 @ hq, w3 @ hq
            a = g / (1.0 + np.exp(-g)) * u
            z += w[t, k] * (w2 @ quant(a))
        n = z / np.sqrt(np.mean(z * z) + cfg.rms_eps) * gamma
        out[t] = up @ n
    return out


def _rel_l2(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_mxfp8_activations_exceed_the_parity_bar():
    cfg = synth.SMALL_ALIGNED.with_tokens(16)
    dense = synth.gen_dense(cfg)
    x = synth.gen_x(cfg)
    idx, _, _, _ = oracle.route(cfg, dense, x)
    experts = {int(e): synth.gen_expert(cfg, int(e)) for e in np.unique(idx)}
    ref = oracle.forward(cfg, dense, experts, x, want_latent=True)
    exact = _layer_from_latent(cfg, dense, experts, ref["h"], ref["idx"], ref["w"], lambda v: v)
    # the re-statement reproduces the oracle (a second, independent reading of the steps)
    assert _rel_l2(exact, ref["out"]) < 1e-12
    # MXFP8 rounding of the two activation inputs alone costs several percent,
    # above the 2e-2 rel-L2 bar, under either block-scale rule; the
    # implementation therefore runs A16
    for no_clip in (False, True):
        q = lambda v: mxfp8(v, no_clip)
        a8 = _layer_from_latent(cfg, dense, experts, ref["h"], ref["idx"], ref["w"], q)
        err = _rel_l2(a8, ref["out"])
        assert 2e-2 < err < 1e-1, (no_clip, err)
        print(f"MXFP8 activations ({'no-clip' if no_clip else 'OCP'} scale): rel-L2 {err:.4f}")


# ------------------------------------------------------------------ the oracle's A8 step
def _bf16_round(v):
    """Nearest BF16 (ties to even) via float32 bit arithmetic (v exactly representable in fp32)."""
    f = np.asarray(v, np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16 << 16
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def test_oracle_rounding_steps_match_their_definitions():
    g = e4m3_grid()
    assert np.array_equal(oracle.e4m3(g), g) and np.array_equal(oracle.e4m3(-g), -g)
    r = np.random.default_rng(3).standard_normal(3000) * 10.0 ** np.random.default_rng(4).uniform(-4, 3, 3000)
    assert np.array_equal(oracle.e4m3(r), e4m3_round(r))
    assert oracle.e4m3(500.0) == 448.0 and oracle.e4m3(1 + 2 ** -4) == 1.0 and oracle.e4m3(2.0 ** -10) == 0.0
    x = r[:2048].reshape(4, 512)
    assert np.array_equal(oracle.mxfp8(x), mxfp8(x))
    f = r.astype(np.float32).astype(np.float64)
    assert np.array_equal(oracle.round_bf16(f), _bf16_round(f))
    assert oracle.round_bf16(1 + 2 ** -8) == 1.0 and oracle.round_bf16(1 + 3 * 2 ** -8) == 1 + 2 ** -6


def test_oracle_a8_mode_is_the_restated_layer():
    # the oracle's A8 option = MXFP8(BF16(h)) into gate/up and MXFP8(a) into down,
    # re-stated here from the test-local (grid-pinned) rounding
    cfg = synth.SMALL_ALIGNED.with_tokens(8)
    dense = synth.gen_dense(cfg)
    x = synth.gen_x(cfg)
    idx, _, _, _ = oracle.route(cfg, dense, x)
    experts = {int(e): synth.gen_expert(cfg, int(e)) for e in np.unique(idx)}
    exact = oracle.forward(cfg, dense, experts, x, want_latent=True)
    a8 = oracle.forward(cfg.with_a8(), dense, experts, x)
    re = _layer_from_latent(cfg, dense, experts, exact["h"], exact["idx"], exact["w"], mxfp8,
                            quant_h=lambda v: mxfp8(_bf16_round(v)))
    assert _rel_l2(a8["out"], re) < 1e-12
    assert 2e-2 < _rel_l2(a8["out"], exact["out"]) < 1e-1


def test_a8_output_moves_with_one_bf16_ulp_of_h():
    # Reading 16 quantises h from its BF16 value.  A BF16 h value that lies on an
    # E4M3 rounding tie (1 in 16 of them) changes its E4M3 code by a full step when
    # h moves by one BF16 ulp, and the GLU output's own MXFP8 rounding turns the
    # resulting ~0.1-0.5% shift of the gate/up sums into a percent-level change of
    # the token's output.  An implementation whose BF16 h differs from the exactly
    # rounded one in a few elements per token (fp32 instead of fp64 accumulation)
    # therefore lands percent-level away on some tokens: the A8 parity bar allows
    # those outputs past max-abs (at most 1e-3 of them, none past 0.25) while
    # rel-L2 keeps the full bar.  The A16 layer moves by orders of magnitude less.
    cfg = synth.SMALL_ALIGNED.with_tokens(4)
    dense = synth.gen_dense(cfg)
    x = synth.gen_x(cfg)
    idx, _, _, _ = oracle.route(cfg, dense, x)
    experts = {int(e): synth.gen_expert(cfg, int(e)) for e in np.unique(idx)}
    ref = oracle.forward(cfg, dense, experts, x, want_latent=True)
    hb = _bf16_round(ref["h"])
    t = 0
    # an element of token 0 on an E4M3 tie, not its block's maximum
    q = mxfp8(hb[t:t + 1])[0]
    tie = None
    for j in range(cfg.L):
        blk = slice(32 * (j // 32), 32 * (j // 32) + 32)
        if abs(hb[t, j]) >= np.abs(hb[t, blk]).max():
            continue
        up = hb[t, j] + 2.0 ** (np.frexp(abs(hb[t, j]))[1] - 8)     # the next BF16 value up
        h2 = hb[t].copy()
        h2[j] = up
        if mxfp8(h2[None])[0][j] != q[j] and abs(hb[t, j]) > 0.5:
            tie = (j, up)
            break
    assert tie is not None
    j, up = tie
    h_pert = hb.copy()
    h_pert[t, j] = up
    a8_base = _layer_from_latent(cfg, dense, experts, hb, ref["idx"], ref["w"], mxfp8)
    a8_pert = _layer_from_latent(cfg, dense, experts, h_pert, ref["idx"], ref["w"], mxfp8)
    a16_base = _layer_from_latent(cfg, dense, experts, hb, ref["idx"], ref["w"], lambda v: v)
    a16_pert = _layer_from_latent(cfg, dense, experts, h_pert, ref["idx"], ref["w"], lambda v: v)
    d8 = np.linalg.norm(a8_pert[t] - a8_base[t]) / np.linalg.norm(a8_base[t])
    d16 = np.linalg.norm(a16_pert[t] - a16_base[t]) / np.linalg.norm(a16_base[t])
    assert d8 > 1e-3 and d8 > 20 * d16, (d8, d16)
