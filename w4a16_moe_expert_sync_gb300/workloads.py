"""Seeded synthetic workloads for the W4A16 routed-MoE layer.

This module is shared by the CUDA path's tests and benchmark and by the
oracle's tests, so it holds none of the layer's arithmetic: no quantisation,
no routing, no alignment, no matmul.  It only defines the workload shapes and
draws the random tensors they start from:

* activations x ~ N(0, 1), stored as bfloat16;
* expert weights W ~ N(0, 0.02^2), fp32, drawn expert by expert so that any
  subset of experts can be regenerated on its own;
* router logits ~ N(0, 1), fp32, plus (skewed workload only) a per-expert
  bias b_e = -1.2 * ln(r_e), with r a seeded permutation of 1..E, so that
  expert popularity follows a Zipf law with exponent 1.2.

The shapes follow the pages' layer: a 256-token canvas, hidden size 2816,
expert intermediate size 704, 128 experts, top-8 routing ("Inference: Making
every denoising pass fast" -- Quantisation alone leaves a sparse execution
problem; "diffusiongemma-26B-A4B-w4a16" -- What the model is, Checkpoint
format).  Random streams are numpy PCG64 keyed by (seed, tensor tag[, expert]).
"""
from __future__ import annotations

import dataclasses

import numpy as np

# tensor tags in the seed sequence
_TAG_X, _TAG_WGU, _TAG_WDN, _TAG_LOGITS, _TAG_ZIPF = 1, 2, 3, 4, 5


@dataclasses.dataclass(frozen=True)
class LayerShape:
    name: str
    M: int          # tokens (canvas rows)
    d: int          # hidden size (gate_up contraction dim)
    m: int          # expert intermediate size (down contraction dim)
    E: int          # experts
    k: int          # experts per token
    seed: int
    routing: str = "gaussian"   # or "zipf"
    gu_group: int = 128
    dn_group: int = 64
    weight_std: float = 0.02

    @property
    def A(self) -> int:
        return self.M * self.k


def _sweep():
    return {f"sweep_M{M}": LayerShape(f"sweep_M{M}", M, 2816, 704, 128, 8, seed=10 + i)
            for i, M in enumerate((1, 8, 32, 64, 128, 256))}


CONFIGS = {
    # small case the oracle finishes in well under a second
    "tiny": LayerShape("tiny", 16, 256, 128, 8, 2, seed=0),
    # several tiles in every dimension and a ragged contraction tail
    "ragged": LayerShape("ragged", 37, 384, 192, 12, 3, seed=6),
    # experts averaging 75 slots: the GEMMs' big-job mode (jobs of 16 to 64 slots)
    "bigjobs": LayerShape("bigjobs", 200, 384, 192, 8, 3, seed=7),
    # one 256-token canvas at the pages' layer shape
    "layer256": LayerShape("layer256", 256, 2816, 704, 128, 8, seed=1),
    # skewed routing: a few experts with >100 rows, many with none
    "zipf256": LayerShape("zipf256", 256, 2816, 704, 128, 8, seed=4, routing="zipf"),
    # eight overlapping canvases
    "canvas2048": LayerShape("canvas2048", 2048, 2816, 704, 128, 8, seed=5),
    **_sweep(),
}


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Store fp32 samples as bfloat16 (round to nearest even); returns uint16 bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def activations(cfg: LayerShape) -> np.ndarray:
    """x [M, d] as bfloat16 bits (uint16)."""
    x = _rng(cfg.seed, _TAG_X).standard_normal((cfg.M, cfg.d), dtype=np.float32)
    return f32_to_bf16_bits(x)


def gate_up_weight(cfg: LayerShape, e: int) -> np.ndarray:
    """W_gu[e] [2m, d] fp32 ~ N(0, std^2)."""
    w = _rng(cfg.seed, _TAG_WGU, e).standard_normal((2 * cfg.m, cfg.d), dtype=np.float32)
    return w * np.float32(cfg.weight_std)


def down_weight(cfg: LayerShape, e: int) -> np.ndarray:
    """W_dn[e] [d, m] fp32 ~ N(0, std^2)."""
    w = _rng(cfg.seed, _TAG_WDN, e).standard_normal((cfg.d, cfg.m), dtype=np.float32)
    return w * np.float32(cfg.weight_std)


def router_logits(cfg: LayerShape) -> np.ndarray:
    """Router logits [M, E] fp32: N(0, 1), plus the Zipf bias when skewed."""
    l = _rng(cfg.seed, _TAG_LOGITS).standard_normal((cfg.M, cfg.E), dtype=np.float32)
    if cfg.routing == "zipf":
        r = _rng(cfg.seed, _TAG_ZIPF).permutation(cfg.E).astype(np.float64) + 1.0
        bias = (-1.2 * np.log(r)).astype(np.float32)
        l = l + bias[None, :]
    return l


def all_gate_up_weights(cfg: LayerShape) -> np.ndarray:
    return np.stack([gate_up_weight(cfg, e) for e in range(cfg.E)])


def all_down_weights(cfg: LayerShape) -> np.ndarray:
    return np.stack([down_weight(cfg, e) for e in range(cfg.E)])


# --------------------------------------------------------------------------
# Beside the layer: RMSNorm inputs and vocabulary logits for the sampler
# ("dg-w4-kernels" -- RMSNorm, Sampler: [256, 262144] fp32 logits per
# denoising step).
# --------------------------------------------------------------------------
_TAG_NORM_X, _TAG_NORM_W, _TAG_VOCAB = 6, 7, 8


@dataclasses.dataclass(frozen=True)
class NormShape:
    name: str
    M: int
    d: int
    seed: int


NORM_CONFIGS = {
    "tiny": NormShape("tiny", 3, 64, seed=30),
    "ragged": NormShape("ragged", 37, 1032, seed=31),       # 129 vectors per row
    "layer256": NormShape("layer256", 256, 2816, seed=32),  # the pages' canvas x hidden
    "wide": NormShape("wide", 5, 8192, seed=33),            # the one-CTA-per-row path
    "canvas2048": NormShape("canvas2048", 2048, 2816, seed=34),
}


def norm_inputs(cfg: NormShape):
    """x [M, d] and weight [d] as bf16 bits: x row t ~ N(0, s_t^2) with s_t
    log-uniform in [0.1, 10] (residual-stream rows of different magnitude),
    weight ~ 1 + 0.1 N(0, 1)."""
    r = _rng(cfg.seed, _TAG_NORM_X)
    scale = np.exp(r.uniform(np.log(0.1), np.log(10.0), (cfg.M, 1)))
    x = (r.standard_normal((cfg.M, cfg.d)) * scale).astype(np.float32)
    w = (1.0 + 0.1 * _rng(cfg.seed, _TAG_NORM_W).standard_normal(cfg.d)).astype(np.float32)
    return f32_to_bf16_bits(x), f32_to_bf16_bits(w)


@dataclasses.dataclass(frozen=True)
class LogitsShape:
    name: str
    M: int          # canvas positions
    V: int          # vocabulary
    seed: int
    mask_frac: float = 0.0   # fraction of each row set to -inf


SAMPLER_CONFIGS = {
    "tiny": LogitsShape("tiny", 4, 1000, seed=40),
    # V % 4 == 3: the scalar-load path, several chunks and a ragged tail
    "ragged": LogitsShape("ragged", 5, 24579, seed=41),
    "masked": LogitsShape("masked", 6, 20000, seed=42, mask_frac=0.5),
    # one denoising step's logits at the pages' shape
    "canvas": LogitsShape("canvas", 256, 262144, seed=43),
}


def vocab_logits(cfg: LogitsShape) -> np.ndarray:
    """Logits [M, V] fp32 with a spread of entropies, as a canvas has between
    undecided and nearly committed positions: row t is N(0, sigma_t^2) with
    sigma_t log-uniform in [0.5, 4]; half the rows (chosen by a coin per row)
    add a peak h_t ~ U(5, 25) at one random column; with mask_frac > 0 that
    fraction of each row's columns (random) is -inf, never the peak column."""
    r = _rng(cfg.seed, _TAG_VOCAB)
    sigma = np.exp(r.uniform(np.log(0.5), np.log(4.0), (cfg.M, 1))).astype(np.float32)
    l = r.standard_normal((cfg.M, cfg.V), dtype=np.float32)
    l *= sigma
    peaked = r.random(cfg.M) < 0.5
    col = r.integers(0, cfg.V, cfg.M)
    h = r.uniform(5.0, 25.0, cfg.M).astype(np.float32)
    rows = np.nonzero(peaked)[0]
    l[rows, col[rows]] += h[rows]
    if cfg.mask_frac > 0:
        for t in range(cfg.M):
            masked = r.random(cfg.V) < cfg.mask_frac
            masked[col[t]] = False
            l[t, masked] = -np.inf
    return l


# --------------------------------------------------------------------------
# The dense W4A16 linear ("dg-w4-kernels" -- W4A16; "Inference: Making every
# denoising pass fast" -- Dense W4 everywhere: 256-row tests of QKV and of an
# LM-head tile).  The pages give neither the QKV width nor the tile width;
# qkv256 uses 4096 output rows (e.g. 16 query heads of 128 plus 8 key and 8
# value heads of 128 over the 2816 hidden size), lmhead256 a 16384-row tile of
# the 262144-row vocabulary head.
# --------------------------------------------------------------------------
_TAG_LIN_X, _TAG_LIN_W = 9, 10


@dataclasses.dataclass(frozen=True)
class LinearShape:
    name: str
    M: int      # rows (tokens)
    K: int      # input features (contraction dim)
    N: int      # output features
    seed: int
    group: int = 128


LINEAR_CONFIGS = {
    "tiny": LinearShape("tiny", 5, 256, 128, seed=50),
    "ragged": LinearShape("ragged", 37, 384, 256, seed=51),
    "wide_k": LinearShape("wide_k", 33, 2816, 384, seed=52),     # K > 768: streamed activations
    "qkv256": LinearShape("qkv256", 256, 2816, 4096, seed=53),
    "lmhead256": LinearShape("lmhead256", 256, 2816, 16384, seed=54),
}


def linear_inputs(cfg: LinearShape):
    """x [M, K] bf16 bits ~ N(0, 1); W [N, K] fp32 ~ N(0, 0.02^2)."""
    x = _rng(cfg.seed, _TAG_LIN_X).standard_normal((cfg.M, cfg.K), dtype=np.float32)
    W = (_rng(cfg.seed, _TAG_LIN_W).standard_normal((cfg.N, cfg.K), dtype=np.float32) * 0.02)
    return f32_to_bf16_bits(x), W.astype(np.float32)
