"""Seeded synthetic inputs shaped like the workloads of the logit-masking and
sampling pages.

This module only draws random inputs; it holds none of the masking or sampling
arithmetic.  It is the one module that both the CUDA path's tests/benchmark and
the CPU oracle's tests use, so both sides see identical inputs.  Arrays are numpy,
on the host; bfloat16 logits are returned as their uint16 bit patterns (round to
nearest even from float32, done by PyTorch's CPU conversion).

No public benchmark or dataset is named by the pages; real grammar masks need a
grammar engine, grammars and tokenizers that are not part of this project.  The
"grammar-like" mask below stands in for them: most allowed tokens come in runs
(token families such as digits or identifier pieces), the rest are isolated bits,
and the bits past ``vocab_size`` in the last word are random garbage so that a
kernel which reads them is caught.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

DTYPES = ("f32", "f16", "bf16")


def to_storage(x32: np.ndarray, dtype: str) -> np.ndarray:
    """float32 array -> storage array of ``dtype`` (bf16 as uint16 bit patterns)."""
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    if dtype == "f32":
        return x32
    if dtype == "f16":
        return x32.astype(np.float16)
    import torch

    t = torch.from_numpy(x32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def storage_to_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float32 values of a storage array (bf16 widened by a 16-bit shift)."""
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a.astype(np.float32)


def pack_bits(allowed: np.ndarray) -> np.ndarray:
    """bool [rows, n] -> int32 words [rows, ceil(n/32)], token j at bit j % 32 of
    word j // 32 (little-endian bit order within each word)."""
    rows, n = allowed.shape
    words = (n + 31) // 32
    padded = np.zeros((rows, words * 32), dtype=bool)
    padded[:, :n] = allowed
    by = np.packbits(padded, axis=1, bitorder="little")
    return np.ascontiguousarray(by).view("<u4").astype(np.uint32).view(np.int32).reshape(rows, words)


def garbage_tail(bitmask: np.ndarray, vocab_size: int, rng: np.random.Generator) -> None:
    """Fill the bits at positions >= vocab_size of every row with random garbage."""
    words = bitmask.shape[1]
    u = bitmask.view(np.uint32)
    first_word, first_bit = divmod(vocab_size, 32)
    if first_word < words:
        junk = rng.integers(0, 2**32, size=bitmask.shape[0], dtype=np.uint64).astype(np.uint32)
        keep = np.uint32((1 << first_bit) - 1) if first_bit else np.uint32(0)
        u[:, first_word] = (u[:, first_word] & keep) | (junk & ~keep)
        if first_word + 1 < words:
            u[:, first_word + 1:] = rng.integers(0, 2**32, size=(bitmask.shape[0],
                                                 words - first_word - 1),
                                                 dtype=np.uint64).astype(np.uint32)


def grammar_like_allowed(rng: np.random.Generator, vocab_size: int, density: float,
                         run_share: float = 0.8, run_min: int = 16,
                         run_max: int = 256) -> np.ndarray:
    """One row of allowed flags with ``round(density * vocab_size)`` tokens set:
    about ``run_share`` of them in runs of U{run_min..run_max} tokens at random
    starts, the rest isolated bits at random free positions."""
    target = int(round(density * vocab_size))
    a = np.zeros(vocab_size, dtype=bool)
    if target <= 0:
        return a
    run_goal = int(run_share * target)
    covered = 0
    while covered < run_goal:
        length = int(rng.integers(run_min, run_max + 1))
        length = min(length, run_goal - covered, vocab_size)
        start = int(rng.integers(0, vocab_size - length + 1))
        seg = a[start:start + length]
        covered += int(length - seg.sum())
        seg[:] = True
    rest = target - int(a.sum())
    if rest > 0:
        free = np.flatnonzero(~a)
        a[rng.choice(free, size=min(rest, free.size), replace=False)] = True
    return a


@dataclass
class Workload:
    """One batch of inputs.  ``logits`` is a 2-D storage array whose width is the
    row stride; ``cols`` is the logical row width (<= stride)."""

    name: str
    dtype: str
    logits: np.ndarray
    cols: int
    vocab_size: int
    bitmask: np.ndarray | None = None
    indices: np.ndarray | None = None
    temperature: np.ndarray | float = 1.0
    top_k: np.ndarray | int = 0
    top_p: np.ndarray | float = 1.0
    min_p: np.ndarray | float = 0.0
    seed: int = 0
    offsets: list = field(default_factory=lambda: [0])
    notes: str = ""

    @property
    def B(self) -> int:
        return self.logits.shape[0]

    @property
    def stride(self) -> int:
        return self.logits.shape[1]

    def per_row(self, name: str) -> np.ndarray:
        v = getattr(self, name)
        dt = np.int32 if name == "top_k" else np.float32
        a = np.asarray(v, dtype=dt)
        return np.full(self.B, a, dtype=dt) if a.ndim == 0 else a.astype(dt)


# ----------------------------------------------------------------- workloads


def tiny_greedy(B: int = 4, V: int = 1003, seed: int = 0) -> Workload:
    """B=4, V=1003 (not a multiple of 32) float32 logits ~N(0,1); bitmask
    [4, 32] with Bernoulli(0.5) bits and the last row all zero (unsatisfiable);
    applied in place to -inf, then greedy."""
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((B, V), dtype=np.float32)
    words = (V + 31) // 32
    bits = rng.integers(0, 2**32, size=(B, words), dtype=np.uint64).astype(np.uint32)
    bits[B - 1, :] = 0
    return Workload("tiny_greedy", "f32", logits, V, V, bitmask=bits.view(np.int32),
                    temperature=0.0, seed=seed)


def apply_only(B: int = 64, V: int = 128256, padded_cols: int = 128512, n_indexed: int = 32,
               density: float = 0.01, sigma: float = 2.0, seed: int = 1,
               dtype: str = "bf16") -> Workload:
    """Bitmask apply only: B rows of bf16 logits ~N(0, sigma) in a buffer padded to
    ``padded_cols`` columns, vocab_size V, a grammar-like mask of ``density``, and
    ``n_indexed`` random unique row indices."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, padded_cols), dtype=np.float32) * np.float32(sigma)
    logits = to_storage(x, dtype)
    allowed = np.stack([grammar_like_allowed(rng, V, density) for _ in range(B)])
    bm = pack_bits(allowed)
    garbage_tail(bm, V, rng)
    idx = np.sort(rng.choice(B, size=min(n_indexed, B), replace=False)).astype(np.int32)
    rng.shuffle(idx)
    return Workload("apply_only", dtype, logits, padded_cols, V, bitmask=bm, indices=idx,
                    seed=seed)


def fused_sample(B: int = 256, V: int = 131072, density: float = 0.10, sigma: float = 3.0,
                 boost_share: float = 0.05, boost: float = 6.0, seed: int = 7,
                 steps: int = 100, dtype: str = "bf16") -> Workload:
    """Fused mask + sample: bf16 logits ~N(0, sigma) with ``boost_share`` of each
    row's tokens raised by ``boost``; grammar-like mask of ``density``; per-row
    temperature U[0.5, 1.2]; top_k 50, top_p 0.9, min_p 0.05; offsets 0..steps-1."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, V), dtype=np.float32) * np.float32(sigma)
    nb = int(round(boost_share * V))
    for b in range(B):
        x[b, rng.choice(V, size=nb, replace=False)] += np.float32(boost)
    logits = to_storage(x, dtype)
    allowed = np.stack([grammar_like_allowed(rng, V, density) for _ in range(B)])
    bm = pack_bits(allowed)
    garbage_tail(bm, V, rng)
    temp = rng.uniform(0.5, 1.2, size=B).astype(np.float32)
    return Workload("fused_sample", dtype, logits, V, V, bitmask=bm, temperature=temp,
                    top_k=50, top_p=0.9, min_p=0.05, seed=seed, offsets=list(range(steps)))


def zipf_top_p(B: int = 1024, V: int = 32000, top_p: float = 0.9, temperature: float = 0.7,
               exponent: float = 1.1, noise: float = 0.1, seed: int = 11) -> Workload:
    """Top-p / greedy sweep without a mask: float32 logits whose ranked values are
    Zipf log-probabilities, -exponent * ln(rank), plus N(0, noise), placed at a
    random permutation of the vocabulary per row."""
    rng = np.random.default_rng(seed)
    base = (-exponent * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
    logits = np.empty((B, V), dtype=np.float32)
    for b in range(B):
        perm = rng.permutation(V)
        logits[b, perm] = base + rng.standard_normal(V, dtype=np.float32) * np.float32(noise)
    return Workload("zipf_top_p", "f32", logits, V, V, temperature=temperature, top_k=0,
                    top_p=top_p, min_p=0.0, seed=seed)


def speculative_verify(slots: int = 128, rows_per_slot: int = 8, V: int = 202048,
                       sigma: float = 2.0, constrained_slots: int = 64, seed: int = 3,
                       dtype: str = "f16") -> Workload:
    """Speculative verify: slots x draft rows, fp16 logits ~N(0, sigma); the rows of
    ``constrained_slots`` random slots are masked (listed in ``indices``) with
    per-row grammar-like densities log-uniform in [0.1%, 30%], two of them all
    zero; the other slots are unconstrained.  Per-row parameters: temperature
    U[0.3, 1.5] with 10% greedy (0), top_k from {0, 1, 20, 50, 1000}, top_p
    U[0.5, 1] with 25% exactly 1, min_p from {0, 0.02, 0.1}."""
    rng = np.random.default_rng(seed)
    B = slots * rows_per_slot
    x = rng.standard_normal((B, V), dtype=np.float32) * np.float32(sigma)
    logits = to_storage(x, dtype)
    words = (V + 31) // 32
    bm = np.full((B, words), -1, dtype=np.int32)
    cslots = np.sort(rng.choice(slots, size=min(constrained_slots, slots), replace=False))
    rows = (cslots[:, None] * rows_per_slot + np.arange(rows_per_slot)[None, :]).reshape(-1)
    dens = np.exp(rng.uniform(np.log(0.001), np.log(0.30), size=rows.size))
    allowed = np.stack([grammar_like_allowed(rng, V, d) for d in dens])
    bm[rows] = pack_bits(allowed)
    if rows.size >= 2:
        bm[rng.choice(rows, size=2, replace=False)] = 0
    garbage_tail(bm, V, rng)
    temp = rng.uniform(0.3, 1.5, size=B).astype(np.float32)
    temp[rng.random(B) < 0.10] = 0.0
    top_k = rng.choice(np.array([0, 1, 20, 50, 1000], dtype=np.int32), size=B)
    top_p = rng.uniform(0.5, 1.0, size=B).astype(np.float32)
    top_p[rng.random(B) < 0.25] = 1.0
    min_p = rng.choice(np.array([0.0, 0.02, 0.1], dtype=np.float32), size=B)
    idx = rows.astype(np.int32)
    return Workload("speculative_verify", dtype, logits, V, V, bitmask=bm, indices=idx,
                    temperature=temp, top_k=top_k, top_p=top_p, min_p=min_p, seed=seed)


WORKLOADS = {
    "tiny_greedy": tiny_greedy,
    "apply_only": apply_only,
    "fused_sample": fused_sample,
    "zipf_top_p": zipf_top_p,
    "speculative_verify": speculative_verify,
}
