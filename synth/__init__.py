"""Seeded synthetic inputs for the MoE permute / FP8-quant / combine path.

This module is shared by the CUDA path's tests and bench and by the CPU
oracle's tests. It holds only input generation: random activations, routing
and expert outputs with the shapes, value distributions and routing skew of
the workloads the SGLang pull-request digests describe. It holds none of the
method's arithmetic (no quantisation, no layout, no combine).

Every generator takes a seed and returns plain numpy arrays:
  * bf16 tensors are returned as ``uint16`` bit patterns;
  * e4m3 tensors are returned as ``uint8`` bit patterns;
  * ids / counts are ``int32``; weights and scales are ``float32``.

Workloads (all single GPU, every expert local):
  tiny      T=16,   H=256,  E=L=8,   K=2, uniform distinct ids
  decode    T=128,  H=7168, E=256, L=32 (ids 0..31 local), K=8, uniform
            distinct ids, x ~ N(0,1) with 1% of elements x50
  prefill   T=8192, H=7168, E=L=256, K=8, Gumbel-top-k over a Zipf(s=1.2)
            popularity with 12 experts forced empty
  mxfp8     24576-row receive buffer, H=7168, 112 live rows, rest garbage
            (NaN / Inf bit patterns), 256 experts, K=8
  requant   T=4096, H=7168, e4m3 payload of N(0,1)*64 (saturated to +-448),
            per-token scales log-uniform in [1e-3, 1e1]; repack over 64
            experts with 128-aligned prefix sums
"""
from __future__ import annotations

import numpy as np
import torch

__all__ = [
    "to_bf16_bits", "from_bf16_bits", "to_e4m3_bits",
    "normal_bf16", "uniform_topk", "zipf_topk", "softmax_weights",
    "repack_counts", "garbage_bf16_rows",
    "tiny", "decode", "prefill", "mxfp8", "requant",
    "PREFILL", "DECODE", "TINY", "MXFP8", "REQUANT",
]

# Workload shapes --------------------------------------------------------

TINY = dict(T=16, H=256, E=8, L=8, K=2, g=128, block_e=128)
DECODE = dict(T=128, H=7168, E=256, L=32, K=8, g=128, cap=128, align=128)
PREFILL = dict(T=8192, H=7168, E=256, L=256, K=8, g=128, block_e=128, n_empty=12)
MXFP8 = dict(T_cap=24576, n_live=112, H=7168, E=256, L=256, K=8, g=32)
REQUANT = dict(T=4096, H=7168, L=64, align=128, blocks=32)


# Conversions (input construction only) ---------------------------------

def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns (uint16), via torch's conversion."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_e4m3_bits(a: np.ndarray) -> np.ndarray:
    """float32 array with |a| <= 448 -> e4m3 bit patterns via torch (input
    construction only; never used to produce an expected value)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


# Primitive generators ---------------------------------------------------

def normal_bf16(rng: np.random.Generator, shape, outlier_frac=0.0, outlier_gain=50.0):
    x = rng.standard_normal(shape, dtype=np.float32)
    if outlier_frac > 0.0:
        mask = rng.random(shape) < outlier_frac
        x = np.where(mask, x * np.float32(outlier_gain), x)
    return to_bf16_bits(x)


def uniform_topk(rng: np.random.Generator, T: int, E: int, K: int) -> np.ndarray:
    """K distinct expert ids per token, uniform over [0, E)."""
    if T == 0:
        return np.zeros((0, K), dtype=np.int32)
    keys = rng.random((T, E))
    return np.argsort(keys, axis=1)[:, :K].astype(np.int32)


def zipf_topk(rng: np.random.Generator, T: int, E: int, K: int, s: float = 1.2,
              n_empty: int = 12) -> np.ndarray:
    """K distinct ids per token drawn without replacement (Gumbel-top-k) from
    a Zipf(s) popularity over a seeded permutation of expert ranks, with
    ``n_empty`` seeded experts forced to probability zero."""
    ranks = rng.permutation(E) + 1
    p = ranks.astype(np.float64) ** (-s)
    empty = rng.choice(E, size=n_empty, replace=False)
    p[empty] = 0.0
    p /= p.sum()
    with np.errstate(divide="ignore"):
        logp = np.log(p)
    g = rng.gumbel(size=(T, E))
    keys = logp[None, :] + g
    ids = np.argsort(-keys, axis=1)[:, :K].astype(np.int32)
    return ids


def softmax_weights(rng: np.random.Generator, T: int, K: int) -> np.ndarray:
    logits = rng.standard_normal((T, K)).astype(np.float64)
    logits -= logits.max(axis=1, keepdims=True) if T else 0.0
    w = np.exp(logits)
    w /= w.sum(axis=1, keepdims=True) if T else 1.0
    return w.astype(np.float32)


def garbage_bf16_rows(rows: int, H: int) -> np.ndarray:
    """Rows of bf16 NaN / +-Inf bit patterns: a live-row kernel must never read them."""
    pat = np.array([0x7FC0, 0x7F80, 0xFF80, 0xFFFF, 0x7FFF, 0xFFC1], dtype=np.uint16)
    n = rows * H
    return np.resize(pat, n).reshape(rows, H) if n else np.zeros((rows, H), np.uint16)


def repack_counts(rng: np.random.Generator, L: int, blocks: int, align: int) -> np.ndarray:
    """Per-expert row counts whose ``align``-rounded sum is ``blocks*align``:
    nb ~ Multinomial(blocks, 1/L); count = align*nb - U[0, align-1] when nb > 0,
    so some experts are empty and every non-empty one leaves a ragged tail."""
    nb = rng.multinomial(blocks, np.full(L, 1.0 / L))
    cut = rng.integers(0, align, size=L)
    counts = np.where(nb > 0, align * nb - cut, 0)
    return counts.astype(np.int32)


# Workloads --------------------------------------------------------------

def tiny(seed: int = 0, T: int | None = None, H: int | None = None):
    c = dict(TINY)
    if T is not None:
        c["T"] = T
    if H is not None:
        c["H"] = H
    rng = np.random.default_rng(1000 + seed)
    T, H, E, K = c["T"], c["H"], c["E"], c["K"]
    x = normal_bf16(rng, (T, H))
    ids = uniform_topk(rng, T, E, K)
    w = softmax_weights(rng, T, K)
    return dict(cfg=c, x=x, topk_ids=ids, topk_weights=w, rng=rng)


def decode(seed: int = 0, T: int | None = None):
    c = dict(DECODE)
    if T is not None:
        c["T"] = T
    rng = np.random.default_rng(2000 + seed)
    T, H, E, K = c["T"], c["H"], c["E"], c["K"]
    x = normal_bf16(rng, (T, H), outlier_frac=0.01, outlier_gain=50.0)
    ids = uniform_topk(rng, T, E, K)
    w = softmax_weights(rng, T, K)
    return dict(cfg=c, x=x, topk_ids=ids, topk_weights=w, rng=rng)


def prefill(seed: int = 0, T: int | None = None, H: int | None = None):
    c = dict(PREFILL)
    if T is not None:
        c["T"] = T
    if H is not None:
        c["H"] = H
    rng = np.random.default_rng(3000 + seed)
    T, H, E, K = c["T"], c["H"], c["E"], c["K"]
    ids = zipf_topk(rng, T, E, K, s=1.2, n_empty=c["n_empty"])
    w = softmax_weights(rng, T, K)
    x = normal_bf16(rng, (T, H))
    if T >= 1024:
        used = np.zeros(E, dtype=bool)
        used[ids.ravel()] = True
        assert (~used).sum() >= 10, "prefill workload must leave >= 10 experts empty"
    return dict(cfg=c, x=x, topk_ids=ids, topk_weights=w, rng=rng)


def expert_outputs(rng: np.random.Generator, rows: int, H: int) -> np.ndarray:
    """bf16 expert outputs y ~ N(0,1), [rows, H]."""
    return normal_bf16(rng, (rows, H))


def mxfp8(seed: int = 0, T_cap: int | None = None, n_live: int | None = None,
          H: int | None = None):
    c = dict(MXFP8)
    if T_cap is not None:
        c["T_cap"] = T_cap
    if n_live is not None:
        c["n_live"] = n_live
    if H is not None:
        c["H"] = H
    rng = np.random.default_rng(4000 + seed)
    T_cap, n, H, E, K = c["T_cap"], c["n_live"], c["H"], c["E"], c["K"]
    buf = np.empty((T_cap, H), dtype=np.uint16)
    buf[:n] = normal_bf16(rng, (n, H))
    buf[n:] = garbage_bf16_rows(T_cap - n, H)
    ids = np.full((T_cap, K), -1, dtype=np.int32)
    ids[:n] = uniform_topk(rng, n, E, K)
    w = np.zeros((T_cap, K), dtype=np.float32)
    w[:n] = softmax_weights(rng, n, K)
    return dict(cfg=c, x=buf, topk_ids=ids, topk_weights=w, rng=rng)


def requant(seed: int = 0, T: int | None = None, H: int | None = None):
    c = dict(REQUANT)
    if T is not None:
        c["T"] = T
    if H is not None:
        c["H"] = H
    rng = np.random.default_rng(5000 + seed)
    T, H = c["T"], c["H"]
    v = np.clip(rng.standard_normal((T, H), dtype=np.float32) * np.float32(64.0), -448.0, 448.0)
    q = to_e4m3_bits(v)
    s = np.exp(rng.uniform(np.log(1e-3), np.log(1e1), size=T)).astype(np.float32)
    return dict(cfg=c, q=q, s_tok=s, rng=rng)
