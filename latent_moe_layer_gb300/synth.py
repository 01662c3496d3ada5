"""Seeded synthetic inputs for the latent routed-MoE layer.

This module only draws numbers: it holds none of the layer's arithmetic, so
both the CUDA path (through the binding) and the fp64 oracle consume exactly
the same bytes.  Every tensor has its own numpy stream, keyed by
``(seed, tensor id, ...)``, so any one expert or any block of tokens can be
regenerated on its own (random access), which is what lets the oracle rebuild
only the experts its sampled tokens touch.

Shapes follow the shard header of the released Kimi K3 checkpoint
("Kimi K3, as released", section "The headline correction"):
``experts.E.w1.weight_packed U8 [3072, 1792]``, ``weight_scale U8 [3072, 112]``,
``w2.weight_packed U8 [3584, 1536]``, ``weight_scale U8 [3584, 96]``;
rows are output features, two E2M1 codes per byte (low nibble first) and one
E8M0 exponent per 32 values along the row.

Recipe (all configurations):
  * x            ~ N(0, 1) drawn in fp64, rounded to fp32 then to BF16 (RNE);
                   drawn in blocks of 1024 tokens, stream (seed, 1, block).
  * W_router     ~ N(0, 1/H) -> fp32 (BF16 for the tiny case), stream (wseed, 2).
  * W_down [L,H] ~ N(0, 1/H) -> BF16, stream (wseed, 3).
  * W_up   [H,L] ~ N(0, 1/L) -> BF16, stream (wseed, 4).
  * gamma  [L]   = 1 (BF16), no draw.
  * expert e, matrix m (0 = w1 gate, 1 = w3 up, 2 = w2 down), stream
    (wseed, 5, e, m): packed bytes uniform over 0..255 (so both nibbles are
    i.i.d. uniform over the 16 E2M1 codes), then E8M0 exponents uniform over
    [exp_lo, exp_hi], one per 32 values.
  * shared GLU matrix m, stream (wseed, 6, m): same distributions.
  * selection bias (skewed case), stream (wseed, 7): R_j ~ Zipf(1.1) via
    ``Generator.zipf``, b_j = 2 ln R_j in fp64, stored fp32.
  * moderate-skew selection bias (bias "rank"), stream (wseed, 7, 1): a seeded
    permutation gives every expert a rank r_j in 1..E, b_j = -0.25 ln r_j
    (fp64, stored fp32).  The layer adds its bias to the sigmoid score, so
    this is the score-space form of a rank-based skew: about a hundred experts
    receive tokens and the top 16 about two thirds of them.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

# tensor ids of the per-tensor streams
_X, _WR, _WD, _WU, _EXPERT, _SHARED, _BIAS = 1, 2, 3, 4, 5, 6, 7
X_BLOCK = 1024


@dataclass(frozen=True)
class LayerConfig:
    """One synthetic workload of the layer (sizes, distributions, seeds)."""

    name: str
    seed: int          # drives x
    wseed: int         # drives every weight tensor
    T: int             # tokens
    H: int             # hidden
    L: int             # latent (expert input/output width)
    E: int             # routed experts
    K: int             # top-k
    I: int             # expert intermediate width
    S: int = 0         # shared-expert intermediate width (0 = no shared experts)
    exp_lo: int = 118
    exp_hi: int = 122
    router_dtype: str = "f32"   # "f32" or "bf16"
    select_bias: bool = False
    rms_eps: float = 1e-6
    routed_scaling: float = 1.0
    act: str = "silu"             # "silu" or "situ" (the GLU activation)
    situ_beta: float = 4.0
    situ_linear_beta: float = 25.0
    a8: bool = False              # MXFP8 activations into the routed experts (the A8 option)
    bias: str = "zipf"            # selection bias recipe when select_bias: "zipf" or "rank"
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    def with_tokens(self, T: int) -> "LayerConfig":
        d = dict(self.__dict__)
        d["T"] = T
        return LayerConfig(**d)

    def with_shared(self, S: int) -> "LayerConfig":
        d = dict(self.__dict__)
        d["S"] = S
        return LayerConfig(**d)

    def with_a8(self, a8: bool = True) -> "LayerConfig":
        d = dict(self.__dict__)
        d["a8"] = a8
        return LayerConfig(**d)

    def with_act(self, act: str) -> "LayerConfig":
        d = dict(self.__dict__)
        d["act"] = act
        return LayerConfig(**d)


K3 = dict(H=7168, L=3584, E=896, K=16, I=3072)

CONFIGS = {
    0: LayerConfig("tiny_t8", seed=0, wseed=0, T=8, H=256, L=128, E=16, K=4, I=96,
                   exp_lo=120, exp_hi=124, router_dtype="bf16"),
    1: LayerConfig("k3_decode_t16", seed=1, wseed=1, T=16, **K3),
    # same weights as the T=16 decode case, own tokens
    2: LayerConfig("k3_decode_t256", seed=2, wseed=1, T=256, **K3),
    3: LayerConfig("k3_prefill_t8192", seed=3, wseed=3, T=8192, **K3),
    4: LayerConfig("k3_prefill_t32768_skew_shared", seed=4, wseed=4, T=32768, S=6144,
                   select_bias=True, **K3),
}

# The secondary prefill workload: config 4 (same tokens, weights and shared
# experts) with the moderate rank-based selection bias instead of the Zipf one.
MODERATE_SKEW = LayerConfig("k3_prefill_t32768_moderate_skew_shared", seed=4, wseed=4, T=32768, S=6144,
                            select_bias=True, bias="rank", **K3)

# A small shape whose packed/scale rows are 16-byte aligned (the tensor-core
# path's requirement) and that spans several 128-row tiles with a ragged tail.
SMALL_ALIGNED = LayerConfig("small_aligned_t40", seed=10, wseed=10, T=40, H=1024, L=512, E=24,
                            K=4, I=512, exp_lo=118, exp_hi=122)
# The same with shared experts (merged intermediate 512).
SMALL_SHARED = LayerConfig("small_shared_t40", seed=11, wseed=11, T=40, H=1024, L=512, E=24, K=4,
                           I=512, S=512, exp_lo=118, exp_hi=122)


# ---------------------------------------------------------------- helpers
def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(list(key))


def f64_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp64 -> fp32 (RNE) -> BF16 (RNE); returns uint16 bit patterns."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def packed_shape(rows: int, cols: int):
    """(packed bytes shape, scale shape) of one MXFP4 matrix [rows, cols]."""
    assert cols % 32 == 0
    return (rows, cols // 2), (rows, cols // 32)


# ---------------------------------------------------------------- tensors
def gen_x(cfg: LayerConfig, rows: np.ndarray | None = None) -> np.ndarray:
    """x [T, H] as BF16 bits.  With ``rows`` only those tokens are returned."""
    nblk = (cfg.T + X_BLOCK - 1) // X_BLOCK

    def block(b):
        n = min(X_BLOCK, cfg.T - b * X_BLOCK)
        return f64_to_bf16_bits(_rng(cfg.seed, _X, b).standard_normal((n, cfg.H)))

    if rows is None:
        with ThreadPoolExecutor(8) as ex:
            parts = list(ex.map(block, range(nblk)))
        return np.concatenate(parts, axis=0)
    rows = np.asarray(rows)
    out = np.empty((len(rows), cfg.H), np.uint16)
    for b in np.unique(rows // X_BLOCK):
        blk = block(int(b))
        sel = np.nonzero(rows // X_BLOCK == b)[0]
        out[sel] = blk[rows[sel] - b * X_BLOCK]
    return out


def gen_router(cfg: LayerConfig) -> np.ndarray:
    """W_router [E, H]: fp32 array, or BF16 bits (uint16) for router_dtype bf16."""
    w = _rng(cfg.wseed, _WR).standard_normal((cfg.E, cfg.H)) * math.sqrt(1.0 / cfg.H)
    if cfg.router_dtype == "bf16":
        return f64_to_bf16_bits(w)
    return w.astype(np.float32)


def gen_down(cfg: LayerConfig) -> np.ndarray:
    w = _rng(cfg.wseed, _WD).standard_normal((cfg.L, cfg.H)) * math.sqrt(1.0 / cfg.H)
    return f64_to_bf16_bits(w)


def gen_up(cfg: LayerConfig) -> np.ndarray:
    w = _rng(cfg.wseed, _WU).standard_normal((cfg.H, cfg.L)) * math.sqrt(1.0 / cfg.L)
    return f64_to_bf16_bits(w)


def gen_gamma(cfg: LayerConfig) -> np.ndarray:
    return np.full(cfg.L, 0x3F80, np.uint16)  # BF16 1.0


RANK_BIAS_BETA = 0.25


def gen_bias(cfg: LayerConfig) -> np.ndarray | None:
    if not cfg.select_bias:
        return None
    if cfg.bias == "rank":
        rank = np.empty(cfg.E, np.float64)
        rank[_rng(cfg.wseed, _BIAS, 1).permutation(cfg.E)] = np.arange(1, cfg.E + 1)
        return (-RANK_BIAS_BETA * np.log(rank)).astype(np.float32)
    r = _rng(cfg.wseed, _BIAS).zipf(1.1, cfg.E).astype(np.float64)
    return (2.0 * np.log(r)).astype(np.float32)


def _mx_matrix(rng: np.random.Generator, rows: int, cols: int, lo: int, hi: int):
    ps, ss = packed_shape(rows, cols)
    packed = rng.integers(0, 256, size=ps, dtype=np.uint8)
    scale = rng.integers(lo, hi + 1, size=ss, dtype=np.uint8)
    return packed, scale


def expert_dims(cfg: LayerConfig):
    """[(rows, cols)] of w1, w3, w2 (out x in)."""
    return [(cfg.I, cfg.L), (cfg.I, cfg.L), (cfg.L, cfg.I)]


def shared_dims(cfg: LayerConfig):
    return [(cfg.S, cfg.H), (cfg.S, cfg.H), (cfg.H, cfg.S)]


def gen_expert(cfg: LayerConfig, e: int):
    """Expert e: [(packed, scale)] for w1, w3, w2."""
    return [_mx_matrix(_rng(cfg.wseed, _EXPERT, e, m), r, c, cfg.exp_lo, cfg.exp_hi)
            for m, (r, c) in enumerate(expert_dims(cfg))]


def gen_shared(cfg: LayerConfig):
    if cfg.S == 0:
        return None
    return [_mx_matrix(_rng(cfg.wseed, _SHARED, m), r, c, cfg.exp_lo, cfg.exp_hi)
            for m, (r, c) in enumerate(shared_dims(cfg))]


def gen_experts_into(cfg: LayerConfig, packed_out, scale_out, experts=None, threads=8):
    """Fill stacked per-matrix buffers: packed_out[m][e], scale_out[m][e].

    ``packed_out[m]`` has shape [E, rows, cols/2] (uint8), ``scale_out[m]``
    [E, rows, cols/32]; any array supporting slice assignment works (numpy,
    pinned torch CPU tensors viewed as numpy).
    """
    experts = range(cfg.E) if experts is None else experts

    def one(e):
        for m, (p, s) in enumerate(gen_expert(cfg, e)):
            packed_out[m][e] = p
            scale_out[m][e] = s

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(one, experts))


@dataclass
class DenseWeights:
    """Everything except the routed experts (host arrays)."""

    w_router: np.ndarray
    select_bias: np.ndarray | None
    w_down: np.ndarray
    w_up: np.ndarray
    gamma: np.ndarray
    shared: list | None


def gen_dense(cfg: LayerConfig) -> DenseWeights:
    return DenseWeights(gen_router(cfg), gen_bias(cfg), gen_down(cfg), gen_up(cfg),
                        gen_gamma(cfg), gen_shared(cfg))
