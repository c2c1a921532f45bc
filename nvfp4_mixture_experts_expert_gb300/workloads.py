"""Seeded synthetic inputs for the NVFP4 mixture-of-experts forward and its GEMMs.

This module holds no quantization, routing, GEMM or activation arithmetic:
only random draws (numpy ``default_rng``), the round-to-nearest-even of fp32
draws to bf16 (the storage type of every raw input), and the shapes and
value distributions of the five workloads.  The CPU oracle tests and the
CUDA tests / benchmark take their inputs from here, so both sides see
identical bytes.

Draw order per workload (fixed, so that a seed names one input set):
hidden/activations, router logits, logit bias or prior, outlier channels,
zero / tiny blocks, then W13 (expert by expert) and W2 (expert by expert).

Workload shapes follow the five configurations the method is measured on:
  tiny      T=64   H=256  I=128  E=8  top_k=2  (zero / underflow blocks)
  gemm      M=2048 K=3584 N=6144 single dense GEMM
  decode    T=128  H=4096 I=2048 E=32 top_k=6  (per-expert logit bias)
  prefill   T=8192 H=4096 I=2048 E=48 top_k=6  (Zipf(1.1) expert prior,
            2% outlier channels x20)
  grouped   G=8 T=2048 D=2048 R=1024 grouped linear on a (T,G,D) input
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "f32_to_bf16_bits", "bf16_bits_to_f32", "MoEWorkload", "GemmWorkload",
    "GroupedLinearWorkload", "moe_workload", "tiny_moe", "decode_moe",
    "prefill_moe", "dense_gemm", "grouped_linear", "gemm_workload", "random_nvfp4_codes",
]

GATE_LIMIT = 10.0
UP_LIMIT = 10.0


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32 values (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return f32_to_bf16_bits((rng.standard_normal(shape, dtype=np.float32) * np.float32(std)))


@dataclass
class MoEWorkload:
    """Inputs of one MoE layer forward.  Raw tensors are bf16 bit patterns.

    hidden  uint16 [T, H]        token activations (bf16)
    logits  float32 [T, E]       router logits
    w13     uint16 [E, 2I, H]    gate rows 0..I-1, up rows I..2I-1, K=H contiguous
    w2      uint16 [E, H, I]     down projection, K=I contiguous
    """
    name: str
    T: int
    H: int
    I: int
    E: int
    top_k: int
    hidden: np.ndarray
    logits: np.ndarray
    w13: np.ndarray
    w2: np.ndarray
    gate_limit: float = GATE_LIMIT
    up_limit: float = UP_LIMIT
    meta: dict = field(default_factory=dict)


def _expert_weights(rng, E, rows, cols, std=0.02):
    out = np.empty((E, rows, cols), dtype=np.uint16)
    for e in range(E):
        out[e] = _normal_bf16(rng, (rows, cols), std)
    return out


def moe_workload(T, H, I, E, top_k, seed=0, *, name="moe", logit_bias_std=0.0,
                 zipf_s=None, outlier_frac=0.0, outlier_gain=20.0,
                 zero_block_frac=0.0, tiny_block_frac=0.0, tiny_amax_range=(1e-9, 0.0117),
                 dead_experts=(), with_weights=True):
    """Generic seeded MoE layer input.

    logit_bias_std: per-expert bias N(0, std) added to N(0,1) logits.
    zipf_s: Zipf exponent of expert popularity, added to logits as log(p_rank)
            with ranks assigned by a seeded permutation of the experts.
    outlier_frac/gain: a seeded random fraction of hidden channels scaled by gain.
    zero_block_frac / tiny_block_frac: fraction of 16-element hidden blocks set to
            exact zero / rescaled so their raw amax is log-uniform in tiny_amax_range.
    dead_experts: experts whose logits are set to -inf (they receive no token).
    with_weights: False leaves w13 / w2 as None (activations and logits are
            drawn first, so they do not depend on this flag).
    """
    rng = np.random.default_rng(seed)
    hid = rng.standard_normal((T, H), dtype=np.float32)
    logits = rng.standard_normal((T, E), dtype=np.float32)
    meta = {}
    if logit_bias_std:
        bias = (rng.standard_normal(E, dtype=np.float32) * np.float32(logit_bias_std)).astype(np.float32)
        logits = (logits + bias[None, :]).astype(np.float32)
        meta["logit_bias"] = bias
    if zipf_s is not None:
        ranks = np.arange(1, E + 1, dtype=np.float64)
        p = ranks ** (-float(zipf_s))
        p /= p.sum()
        perm = rng.permutation(E)
        prior = np.empty(E, dtype=np.float64)
        prior[perm] = np.log(p)
        logits = (logits.astype(np.float64) + prior[None, :]).astype(np.float32)
        meta["zipf_prior"] = prior.astype(np.float32)
    if outlier_frac:
        n_out = int(round(outlier_frac * H))
        ch = np.sort(rng.choice(H, size=n_out, replace=False))
        hid[:, ch] *= np.float32(outlier_gain)
        meta["outlier_channels"] = ch
    if zero_block_frac or tiny_block_frac:
        nblk = T * (H // 16)
        n_zero = int(round(zero_block_frac * nblk))
        n_tiny = int(round(tiny_block_frac * nblk))
        pick = rng.choice(nblk, size=n_zero + n_tiny, replace=False)
        blocks = hid.reshape(nblk, 16)
        blocks[pick[:n_zero]] = 0.0
        lo, hi = np.log(tiny_amax_range[0]), np.log(tiny_amax_range[1])
        target = np.exp(rng.uniform(lo, hi, size=n_tiny)).astype(np.float32)
        tb = blocks[pick[n_zero:]]
        amax = np.max(np.abs(tb), axis=1)
        amax[amax == 0] = 1.0
        blocks[pick[n_zero:]] = tb / amax[:, None] * target[:, None]
        meta["zero_blocks"] = np.sort(pick[:n_zero])
        meta["tiny_blocks"] = np.sort(pick[n_zero:])
    for e in dead_experts:
        logits[:, e] = -np.inf
    w13 = _expert_weights(rng, E, 2 * I, H) if with_weights else None
    w2 = _expert_weights(rng, E, H, I) if with_weights else None
    return MoEWorkload(name=name, T=T, H=H, I=I, E=E, top_k=top_k,
                       hidden=f32_to_bf16_bits(hid), logits=np.ascontiguousarray(logits, np.float32),
                       w13=w13, w2=w2, meta=meta)


def tiny_moe(seed=0):
    """T=64, H=256, I=128, E=8, top_k=2; 5% zero blocks and 5% tiny blocks."""
    return moe_workload(64, 256, 128, 8, 2, seed, name="tiny_moe",
                        zero_block_frac=0.05, tiny_block_frac=0.05)


def decode_moe(seed=0, with_weights=True):
    """T=128, H=4096, I=2048, E=32, top_k=6; logits N(0,1) + per-expert bias N(0,0.5)."""
    return moe_workload(128, 4096, 2048, 32, 6, seed, name="decode_moe", logit_bias_std=0.5,
                        with_weights=with_weights)


def prefill_moe(seed=0, T=8192, with_weights=True):
    """T=8192, H=4096, I=2048, E=48, top_k=6; Zipf(1.1) prior, 2% outlier channels x20."""
    return moe_workload(T, 4096, 2048, 48, 6, seed, name="prefill_moe", zipf_s=1.1,
                        outlier_frac=0.02, outlier_gain=20.0, with_weights=with_weights)


@dataclass
class GemmWorkload:
    """One dense GEMM D = A . B^T.  A uint16 [M, K] bf16, B uint16 [N, K] bf16."""
    name: str
    M: int
    N: int
    K: int
    a: np.ndarray
    b: np.ndarray


def gemm_workload(M, N, K, seed=0, name="gemm", row_lognormal=True):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((M, K), dtype=np.float32)
    if row_lognormal:
        a *= np.exp(rng.standard_normal((M, 1))).astype(np.float32)
    b = rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)
    return GemmWorkload(name=name, M=M, N=N, K=K, a=f32_to_bf16_bits(a), b=f32_to_bf16_bits(b))


def dense_gemm(seed=0):
    """M=2048, K=3584, N=6144; A N(0,1) with per-row lognormal(0,1) gain, B N(0,0.02)."""
    return gemm_workload(2048, 6144, 3584, seed, name="dense_gemm")


@dataclass
class GroupedLinearWorkload:
    """Grouped linear: x uint16 [T, G, D] bf16, w uint16 [G, R, D] bf16,
    w_gs float32 [G] per-group weight global scales."""
    name: str
    T: int
    G: int
    D: int
    R: int
    x: np.ndarray
    w: np.ndarray
    w_gs: np.ndarray


def grouped_linear(seed=0, T=2048, G=8, D=2048, R=1024, name="grouped_linear"):
    """G=8, T=2048, D=2048, R=1024; weight global scales U[0.5, 2]."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, G, D), dtype=np.float32)
    w = rng.standard_normal((G, R, D), dtype=np.float32) * np.float32(0.02)
    w_gs = rng.uniform(0.5, 2.0, size=G).astype(np.float32)
    return GroupedLinearWorkload(name=name, T=T, G=G, D=D, R=R, x=f32_to_bf16_bits(x),
                                 w=f32_to_bf16_bits(w), w_gs=w_gs)


def random_nvfp4_codes(groups, rows, K, seed, scale_code_range=(0x28, 0x40)):
    """Random NVFP4 operand codes for timing runs (the arithmetic cost of a
    consumer does not depend on the values): E2M1 codes uniform over all 16,
    E4M3 scale codes uniform in scale_code_range, global scales 1.
    Returns (codes uint8 [groups, rows, K], scale codes uint8 [groups, rows, K/16],
    global scales float32 [groups])."""
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(groups, rows, K), dtype=np.uint8)
    scales = rng.integers(scale_code_range[0], scale_code_range[1], size=(groups, rows, K // 16), dtype=np.uint8)
    return codes, scales, np.ones(groups, dtype=np.float32)
