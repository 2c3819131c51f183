"""Seeded synthetic bf16 weight generators (input side only).

This module is shared by the oracle tests, the CUDA parity tests and the
benchmark.  It holds no part of the codec: it only draws random numbers and
rounds them to bf16 bit patterns (``numpy.uint16`` arrays, little-endian in
memory, so byte ``2i+1`` of the buffer is the high -- sign and exponent --
byte of value ``i``).

Recipe (the source pages use real Kimi K3 trunk weights, which are not
available; these synthetic tensors stand in for them):

* every draw is float64 from numpy's PCG64 ``default_rng``, cast to float32
  and then rounded to bf16 with round-to-nearest-even;
* large tensors are drawn in blocks of ``BLOCK`` values, block ``b`` of a
  stream with seed ``s`` using ``default_rng([s, tag, b])``, so the bytes do
  not depend on the number of worker threads;
* the shapes and distributions are those of the five workloads below.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

BLOCK = 1 << 22  # values per independently seeded block

# Tensor shapes of one trunk layer: four square attention projections, the
# two low-rank latent projections, and the three MLP matrices.
TRUNK_LAYER_SHAPES = [
    (8192, 8192), (8192, 8192), (8192, 8192), (8192, 8192),
    (576, 8192), (8192, 576),
    (8192, 24576), (8192, 24576), (24576, 8192),
]

WORKLOADS = {
    "tiny": "one 4 MiB bf16 tensor 1024x2048 ~ N(0, 0.02), seed 0",
    "projection": "bf16 8192x16384 (256 MiB): N(0,1) x per-row lognormal(ln 0.02, 0.5) scale, seed 1",
    "heavy_tail": "1 GiB bf16: 0.01 * Student-t(3), 1% replaced by a 20-step power-of-two ladder, seed 2",
    "trunk_layer": "one trunk layer of 9 tensors N(0, 1/sqrt(fan_in)), one code table each, seed 3",
    "ring": "14 trunk layers (seeds 10..23) streamed from pinned host memory",
    "ring_file": "trunk layers (seeds 10..) read from a container file (O_DIRECT where allowed) into the pinned ring",
    "encode": "GPU encoder: the heavy-tail 1 GiB bf16 tensor (seed 2) packed into a container on the device",
    "gemv": "y = W x with the projection matrix W (8192x16384, seed 1) held compressed, x ~ N(0,1) bf16 (seed 4)",
}

_THREADS = max(1, min(16, os.cpu_count() or 1))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even).

    Returns the 16-bit patterns.  NaN is not expected from the generators.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (h.astype(np.uint32) << 16).view(np.float32)


def _blocked(n: int, seed: int, tag: int, fill) -> np.ndarray:
    """Fill ``n`` bf16 values block by block; ``fill(rng, start, count)``
    returns float64 (or float32) values for positions [start, start+count)."""
    out = np.empty(n, dtype=np.uint16)
    nb = (n + BLOCK - 1) // BLOCK

    def one(b):
        s = b * BLOCK
        c = min(BLOCK, n - s)
        rng = np.random.default_rng([seed, tag, b])
        out[s:s + c] = f32_to_bf16_bits(np.asarray(fill(rng, s, c), dtype=np.float64).astype(np.float32))

    if nb <= 1:
        for b in range(nb):
            one(b)
    else:
        with ThreadPoolExecutor(_THREADS) as ex:
            list(ex.map(one, range(nb)))
    return out


def normal_tensor(shape, std: float, seed: int, tag: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    return _blocked(n, seed, tag, lambda r, s, c: r.normal(0.0, std, c))


def tiny(seed: int = 0) -> np.ndarray:
    """1024x2048 values ~ N(0, 0.02): one stripe, the small parity case."""
    return normal_tensor((1024, 2048), 0.02, seed)


def projection(seed: int = 1, rows: int = 8192, cols: int = 16384) -> np.ndarray:
    """Projection matrix: N(0,1) times a per-row log-normal scale."""
    scale = np.random.default_rng([seed, 1 << 30]).lognormal(math.log(0.02), 0.5, rows)

    def fill(r, s, c):
        idx = np.arange(s, s + c) // cols
        return r.standard_normal(c) * scale[idx]

    return _blocked(rows * cols, seed, 0, fill)


def heavy_tail(seed: int = 2, n: int = 1 << 29) -> np.ndarray:
    """0.01 * Student-t(3); 1% of the values replaced by +-2^k (1 + m/128),
    k in 0..19 with P(k) proportional to 2^-k, m uniform in 0..127.  The
    ladder's exponents reach far past the bulk, so an unconstrained Huffman
    code on the high bytes is deeper than 12 bits."""
    pk = 2.0 ** -np.arange(20)
    pk /= pk.sum()

    def fill(r, s, c):
        v = 0.01 * r.standard_t(3.0, c)
        mask = r.random(c) < 0.01
        m = int(mask.sum())
        k = r.choice(20, size=m, p=pk)
        sign = np.where(r.random(m) < 0.5, -1.0, 1.0)
        mant = r.integers(0, 128, m)
        v[mask] = sign * np.ldexp(1.0 + mant / 128.0, k)
        return v

    return _blocked(n, seed, 0, fill)


def trunk_layer(seed: int = 3, shapes=None):
    """The tensors of one trunk layer, each N(0, 1/sqrt(fan_in)) with
    fan_in = number of columns (PyTorch [out, in] layout)."""
    shapes = TRUNK_LAYER_SHAPES if shapes is None else shapes
    return [normal_tensor(shp, 1.0 / math.sqrt(shp[1]), seed, tag=i) for i, shp in enumerate(shapes)]


def ring_layers(first_seed: int = 10, n_layers: int = 14, shapes=None):
    """Seeds of the streamed layers; generate one at a time with trunk_layer."""
    return [first_seed + i for i in range(n_layers)]


# --- edge cases -----------------------------------------------------------

def single_symbol(n: int, seed: int = 100) -> np.ndarray:
    """Every value is +1.0 with a random low byte: one high-byte symbol."""
    lo = np.random.default_rng(seed).integers(0, 256, n).astype(np.uint16)
    return (np.uint16(0x3F00) | lo).astype(np.uint16)


def two_symbol(n: int, seed: int = 101) -> np.ndarray:
    """Values +-1.x with random low bytes: two high-byte symbols."""
    r = np.random.default_rng(seed)
    lo = r.integers(0, 256, n).astype(np.uint16)
    hi = np.where(r.random(n) < 0.5, 0x3F, 0xBF).astype(np.uint16)
    return ((hi << 8) | lo).astype(np.uint16)


def uniform_bytes(n: int, seed: int = 102) -> np.ndarray:
    """Uniformly random 16-bit patterns: all 256 high bytes, near 8-bit entropy."""
    return np.random.default_rng(seed).integers(0, 1 << 16, n).astype(np.uint16)


def dyadic_long_codes(n: int, seed: int = 104) -> np.ndarray:
    """High bytes drawn with dyadic probabilities: four symbols of probability
    1/2, 1/4, 1/8, 1/16, two of 1/64 and 128 of 1/4096, so that about 3% of
    the values carry the rarest symbols and about one pair in a thousand
    consecutive values is two of them; random low bytes."""
    r = np.random.default_rng(seed)
    probs = np.array([2.0 ** -1, 2.0 ** -2, 2.0 ** -3, 2.0 ** -4] + [2.0 ** -6] * 2 + [2.0 ** -12] * 128)
    syms = r.permutation(256)[: probs.size]
    hi = syms[r.choice(probs.size, n, p=probs / probs.sum())].astype(np.uint16)
    lo = r.integers(0, 256, n).astype(np.uint16)
    return ((hi << 8) | lo).astype(np.uint16)


def geometric_exponent_symbols(n: int, alpha: float, seed: int = 103) -> np.ndarray:
    """Integers k with P(k) = (1-q)/(1+q) q^|k|, q = 2^-alpha (two-sided
    geometric law of a floating-point exponent), via the difference of two
    independent geometric variables."""
    q = 2.0 ** -alpha
    r = np.random.default_rng(seed)
    a = r.geometric(1.0 - q, n) - 1
    b = r.geometric(1.0 - q, n) - 1
    return a - b


def workload(name: str):
    """List of tensors (uint16 arrays) of a named workload (not 'ring')."""
    if name == "tiny":
        return [tiny()]
    if name == "projection":
        return [projection()]
    if name == "heavy_tail":
        return [heavy_tail()]
    if name == "trunk_layer":
        return trunk_layer()
    raise KeyError(name)
