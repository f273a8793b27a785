"""Seeded synthetic inputs shaped like the workloads the method is described on.

This module only draws random inputs; it holds none of the method's arithmetic
(no rotation, scaling, snapping or packing).  Both the CUDA path's tests and the
fp64 oracle take their inputs from here, so they see identical bytes.

Every generator uses numpy ``Generator(PCG64(seed))`` and draws in the order
written.  Values stated as bf16 are drawn in fp64, cast to fp32 and rounded to
bf16 with round-to-nearest-even; they are returned both as the bf16 bit pattern
(uint16) and as the exactly equal fp32 array.

Workload shapes (sizes are those of the workloads, seeds fixed):

* dense tiny: W fp32 [512, 512] ~ N(0, 0.02^2) with 1% of entries x8
  outliers, x fp32 [1, 512] ~ N(0, 1); 4-bit codebook, group 64, seed 0.
* dense decode: W bf16 [11008, 4096] = Student-t(4) * 0.02 with a per-row
  lognormal(0, 0.5) scale; 3-bit, group 128; x bf16 [T, 4096] ~ N(0, 1); seed 2.
* MoE decode (Kimi-K2-shaped): 384 experts, top-8, hidden 7168, expert
  intermediate 2048, ternary group 16; router logits fp32 ~ N(0, 1);
  x bf16 [1, 7168]; seed 3.
* MoE prefill: 4096 tokens, 128 experts, top-8, hidden 4096, intermediate
  1536, 3-bit group 64; logits N(0, 1) plus a Zipf(1.1) expert bias; seed 4.
* KV cache: 131072 tokens, 8 kv heads, head dim 128, K 8-bit, V 3-bit,
  group 32; K, V bf16 = N(0, 1) * exp(sigma[h, c]), sigma ~ N(0, 1) per
  (head, channel), independent for K and V; q bf16 [32, 128]; seed 5.
"""
from __future__ import annotations

import numpy as np

SEED_DENSE_TINY = 0
SEED_DENSE_DECODE = 2
SEED_MOE_DECODE = 3
SEED_MOE_PREFILL = 4
SEED_KV = 5


def rng(seed: int, *stream: int) -> np.random.Generator:
    """A PCG64 generator for ``seed`` and an optional sub-stream key."""
    return np.random.Generator(np.random.PCG64([int(seed), *[int(s) for s in stream]]))


def sign_seed(seed: int, dim_index: int) -> int:
    """Seed of the rotation sign vector for the ``dim_index``-th input dim of a workload."""
    return int(seed) * 1000 + int(dim_index)


def to_bf16(a) -> tuple[np.ndarray, np.ndarray]:
    """Round to bf16 (nearest even). Returns (uint16 bits, float32 values)."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    nan = np.isnan(f)
    bits = rounded.astype(np.uint16)
    bits[nan] = 0x7FC0
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    return bits, vals


def dense_tiny(seed: int = SEED_DENSE_TINY, n: int = 512, k: int = 512):
    """W fp32 [n, k] ~ N(0, 0.02^2) with Bernoulli(0.01) entries scaled x8; x fp32 [1, k]."""
    g = rng(seed)
    W = g.normal(0.0, 0.02, size=(n, k))
    mask = g.random(size=(n, k)) < 0.01
    W = np.where(mask, W * 8.0, W).astype(np.float32)
    x = g.normal(0.0, 1.0, size=(1, k)).astype(np.float32)
    return W, x


def heavy_rows(g: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    """Student-t(4) * 0.02 entries with a per-row lognormal(0, 0.5) scale (fp32)."""
    t = g.standard_t(4.0, size=(rows, cols)) * 0.02
    s = np.exp(g.normal(0.0, 0.5, size=(rows, 1)))
    return (t * s).astype(np.float32)


def dense_decode_weights(seed: int = SEED_DENSE_DECODE, n: int = 11008, k: int = 4096, rows=None):
    """bf16 W [n, k] (or only the listed ``rows``, drawn from per-row sub-streams)."""
    if rows is None:
        rows = range(n)
    out = np.stack([heavy_rows(rng(seed, 1, r), 1, k)[0] for r in rows]) if len(rows) else np.zeros((0, k), np.float32)
    return to_bf16(out)


def dense_decode_x(seed: int = SEED_DENSE_DECODE, t: int = 1, k: int = 4096):
    return to_bf16(rng(seed, 2, t).normal(0.0, 1.0, size=(t, k)))


def expert_weights(seed: int, expert: int, which: int, rows: int, cols: int):
    """bf16 weights of one expert projection (which: 0 = gate||up, 1 = down)."""
    return to_bf16(heavy_rows(rng(seed, 3, which, expert), rows, cols))


def router_logits(seed: int, tokens: int, experts: int, zipf: float | None = None):
    """fp32 router logits [tokens, experts] ~ N(0, 1), plus an optional Zipf expert bias.

    The Zipf bias gives expert e the log-probability log(r_e^-a / sum_r r^-a)
    where r_e is its rank under a seeded permutation.
    """
    g = rng(seed, 4, tokens)
    logits = g.normal(0.0, 1.0, size=(tokens, experts))
    if zipf is not None:
        ranks = g.permutation(experts) + 1
        w = ranks.astype(np.float64) ** (-zipf)
        logits = logits + np.log(w / w.sum())[None, :]
    return logits.astype(np.float32)


def activations(seed: int, tokens: int, hidden: int, stream: int = 5):
    """bf16 activations [tokens, hidden] ~ N(0, 1)."""
    return to_bf16(rng(seed, stream, tokens).normal(0.0, 1.0, size=(tokens, hidden)))


def kv_cache(seed: int = SEED_KV, tokens: int = 131072, heads: int = 8, dim: int = 128, which: int = 0,
             token_offset: int = 0):
    """bf16 K (which=0) or V (which=1) [tokens, heads, dim] = N(0,1) * exp(sigma[h, c]).

    sigma ~ N(0, 1) per (head, channel) is drawn once per (seed, which); the
    N(0, 1) body is drawn per token block of 4096 so any token range can be
    regenerated on its own.
    """
    sigma = rng(seed, 6, which).normal(0.0, 1.0, size=(heads, dim))
    out = np.empty((tokens, heads, dim), dtype=np.float32)
    blk = 4096
    t = 0
    while t < tokens:
        a = token_offset + t
        b0 = a // blk
        body = rng(seed, 7, which, b0).normal(0.0, 1.0, size=(blk, heads, dim))
        lo = a - b0 * blk
        n = min(blk - lo, tokens - t)
        out[t:t + n] = body[lo:lo + n] * np.exp(sigma)[None]
        t += n
    return to_bf16(out)


def kv_query(seed: int = SEED_KV, heads: int = 32, dim: int = 128):
    return to_bf16(rng(seed, 8).normal(0.0, 1.0, size=(heads, dim)))
