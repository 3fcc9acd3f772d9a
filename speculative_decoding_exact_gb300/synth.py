"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the oracle.

This module draws random numbers and lays them out in the input formats; it
holds none of the verify step's arithmetic.  Every tensor is keyed by
(seed, tensor_id) through NumPy's PCG64 bit generator (``random_raw`` only, so
the stream does not depend on NumPy's distribution code).

Distributions (the workload descriptions of the benchmark configurations):
  * Q4_K weights: 4-bit codes uniform in 0..15, 6-bit sub-scales and sub-mins
    uniform in 0..63 (uniform random bytes in the packed field), d and dmin
    uniform in [1e-3, 1e-2) rounded to binary16;
  * hidden rows and activations: N(0, 1) via Box-Muller in fp64, stored fp32;
  * KV context: N(0, 1) rounded to bf16 (round to nearest even).
"""
from __future__ import annotations

import numpy as np

SUPERBLOCK_BYTES = 144


def generator(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(tensor_id)])))


def raw_u64(seed: int, tensor_id: int, n: int) -> np.ndarray:
    return generator(seed, tensor_id).bit_generator.random_raw(int(n)).astype(np.uint64)


def random_bytes(seed: int, tensor_id: int, nbytes: int) -> np.ndarray:
    words = raw_u64(seed, tensor_id, (nbytes + 7) // 8)
    return words.view(np.uint8)[:nbytes].copy()


def uniform01(seed: int, tensor_id: int, n: int) -> np.ndarray:
    """Uniform in [0, 1) with 53 random bits (fp64)."""
    return (raw_u64(seed, tensor_id, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(shape, seed: int, tensor_id: int) -> np.ndarray:
    """Standard normal, Box-Muller in fp64, returned as fp32."""
    n = int(np.prod(shape))
    m = (n + 1) // 2
    u = uniform01(seed, tensor_id, 2 * m)
    u1 = 1.0 - u[:m]                      # (0, 1]
    u2 = u[m:]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.concatenate([r * np.cos(2.0 * np.pi * u2), r * np.sin(2.0 * np.pi * u2)])[:n]
    return z.astype(np.float32).reshape(shape)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep = u >> np.uint64(16)
    rest = u & np.uint64(0xFFFF)
    up = (rest > 0x8000) | ((rest == 0x8000) & ((keep & np.uint64(1)) == 1))
    return (keep + up.astype(np.uint64)).astype(np.uint16)


def q4k_matrix(N: int, K: int, seed: int, tensor_id: int,
               d_lo: float = 1e-3, d_hi: float = 1e-2, dmin_over_d: float | None = None) -> np.ndarray:
    """Canonical Q4_K bytes of an N x K matrix (N*(K/256) superblocks of 144 B).

    With dmin_over_d = None (the benchmark workload) d and dmin are drawn
    independently from U[d_lo, d_hi).  With a ratio r, dmin = r * d: r = 7.5
    makes every weight's expectation zero (E[sc] = E[m], E[q] = 7.5), so the
    logits are no longer dominated by one direction and rows disagree on
    their argmax (used by tests that exercise the argmax)."""
    assert K % 256 == 0
    nsb = N * (K // 256)
    sb = random_bytes(seed, tensor_id, nsb * SUPERBLOCK_BYTES).reshape(nsb, SUPERBLOCK_BYTES)
    u = uniform01(seed, tensor_id + (1 << 40), 2 * nsb)
    dd = (d_lo + (d_hi - d_lo) * u).reshape(2, nsb)
    if dmin_over_d is not None:
        dd[1] = dd[0] * dmin_over_d
    d = dd.astype(np.float16).view(np.uint16)
    sb[:, 0] = (d[0] & 0xFF).astype(np.uint8)
    sb[:, 1] = (d[0] >> 8).astype(np.uint8)
    sb[:, 2] = (d[1] & 0xFF).astype(np.uint8)
    sb[:, 3] = (d[1] >> 8).astype(np.uint8)
    return sb.reshape(-1)


def tokens(n: int, vocab: int, seed: int, tensor_id: int) -> np.ndarray:
    return (raw_u64(seed, tensor_id, n) % np.uint64(vocab)).astype(np.int32)


def plant_draft(target: np.ndarray, accepted: int, vocab: int, seed: int, tensor_id: int) -> np.ndarray:
    """Draft tokens for k = len(target)-1 whose greedy accepted length is `accepted`:
    draft[i] = target[i] for i < accepted, draft[accepted] = target[accepted]+1 mod V,
    the rest random (their value cannot matter)."""
    k = len(target) - 1
    d = tokens(k, vocab, seed, tensor_id)
    d[:accepted] = target[:accepted]
    if accepted < k:
        d[accepted] = (int(target[accepted]) + 1) % vocab
    return d.astype(np.int32)


# Model geometries used by tests and the benchmark --------------------------------
FULL = dict(hidden=6656, n_layers=52, n_q_heads=52, n_kv_heads=4, head_dim=128, ffn=17920,
            vocab=131072)
SMALL = dict(hidden=1664, n_layers=2, n_q_heads=13, n_kv_heads=1, head_dim=128, ffn=4608,
             vocab=4096)
