"""Seeded synthetic inputs for the Q1_0 GEMV: weights, activations, raw quants.

This module draws random numbers and lays them out in the input formats; it
holds none of the product's arithmetic.  Both the CUDA path and the CPU oracle
receive exactly the arrays made here.

Input formats:
  Q1_0 weight blocks  uint8 [rows, n/128, 18]: bytes 0-1 the block scale d0 as
                      little-endian IEEE binary16, bytes 2-17 the 128 sign bits
                      (element j in byte 2 + j//8, bit j%8; 1 = +d0, 0 = -d0).
  Q2_0 weight blocks  uint8 [rows, n/128, 34]: bytes 0-1 the block scale d0 as
                      above, bytes 2-33 the 128 2-bit codes (element j in byte
                      2 + j//4, bits 2*(j%4)..2*(j%4)+1; code 0/1/2 = -1/0/+1
                      times d0)
  activations         float32 [B, n]
  raw q8_0 quants     int8 [B, n] and binary16 scale bits uint16 [B, n/32]

Distributions (the shapes of the workloads the pages and the benchmark name):
  sign bits           Bernoulli(0.5), i.e. uniform random bytes
  ternary values      -1, 0, +1 with probabilities (1-p0)/2, p0, (1-p0)/2
                      (p0 = 1/3 unless a test asks otherwise); for the
                      full-size sets, uniform random bytes with the code 3
                      read as 1 (p0 = 1/2), which is cheap at 7.5 G weights
  d0 "halfnormal"     |N(0, 0.02)| rounded to binary16 (about 0.24 % of blocks
                      land in the binary16 subnormal range)
  d0 "lognormal"      exp(N(ln 0.02, 1)) rounded to binary16 (scales that vary
                      per block over several binades: the "layer-shaped" regime)
  activations         N(0, 1) float32, optionally with 1 % outliers of
                      magnitude 20 at positions drawn without replacement
"""
from __future__ import annotations

import numpy as np

QK1 = 128          # weights per Q1_0 block
QK8 = 32           # activation values per q8_0 scale
BLOCK_BYTES = 18
Q2_BLOCK_BYTES = 34

# Llama-3-8B-shaped decode step: per layer q, k, v, o, gate, up, down; then lm_head.
LLAMA3_8B_LAYER = (
    ("q", 4096, 4096),
    ("k", 1024, 4096),
    ("v", 1024, 4096),
    ("o", 4096, 4096),
    ("gate", 14336, 4096),
    ("up", 14336, 4096),
    ("down", 4096, 14336),
)
LLAMA3_8B_LAYERS = 32
LLAMA3_8B_LM_HEAD = ("lm_head", 128256, 4096)


def decode_set_shapes():
    """The 225 (name, rows, n) products of one Llama-3-8B-shaped decode step."""
    out = []
    for layer in range(LLAMA3_8B_LAYERS):
        for name, rows, n in LLAMA3_8B_LAYER:
            out.append((f"L{layer}.{name}", rows, n))
    out.append(LLAMA3_8B_LM_HEAD)
    return out


def rng_for(*keys: int) -> np.random.Generator:
    """A generator seeded from a tuple of non-negative integers."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in keys])))


def fp16_bits(values: np.ndarray) -> np.ndarray:
    """Binary16 bit patterns of `values` (numpy's own float16 rounding)."""
    return np.asarray(values, dtype=np.float64).astype(np.float16).view(np.uint16)


def block_scales(rng: np.random.Generator, shape, kind: str = "halfnormal") -> np.ndarray:
    """Binary16 bits of block scales with the named distribution."""
    if kind == "halfnormal":
        v = np.abs(rng.standard_normal(shape)) * 0.02
    elif kind == "lognormal":
        v = np.exp(rng.standard_normal(shape) + np.log(0.02))
    elif kind == "ones":
        v = np.ones(shape)
    elif kind == "signed":
        v = rng.standard_normal(shape) * 0.02
    else:
        raise ValueError(f"unknown scale distribution {kind!r}")
    return fp16_bits(v)


def assemble_blocks(scale_bits: np.ndarray, sign_bytes: np.ndarray) -> np.ndarray:
    """Lay out [rows, nb] scale bits and [rows, nb, 16] sign bytes as 18-byte blocks."""
    rows, nb = scale_bits.shape
    if sign_bytes.shape != (rows, nb, 16):
        raise ValueError("sign bytes must be [rows, nb, 16]")
    blocks = np.empty((rows, nb, BLOCK_BYTES), dtype=np.uint8)
    s = np.ascontiguousarray(scale_bits, dtype=np.uint16)
    blocks[:, :, 0] = (s & 0xFF).astype(np.uint8)
    blocks[:, :, 1] = (s >> 8).astype(np.uint8)
    blocks[:, :, 2:] = sign_bytes
    return blocks


def weight_blocks(rng: np.random.Generator, rows: int, n: int, scale: str = "halfnormal") -> np.ndarray:
    """Random Q1_0 weight blocks uint8 [rows, n/128, 18]."""
    if n % QK1:
        raise ValueError("n must be a multiple of 128")
    nb = n // QK1
    signs = rng.integers(0, 256, size=(rows, nb, 16), dtype=np.uint8)
    scales = block_scales(rng, (rows, nb), scale)
    return assemble_blocks(scales, signs)


def sign_bytes_from_bits(bits: np.ndarray) -> np.ndarray:
    """Pack a {0,1} array [..., 128] into the block's 16 sign bytes (bit j%8 of byte j//8)."""
    bits = np.asarray(bits, dtype=np.uint8)
    return np.packbits(bits.reshape(bits.shape[:-1] + (16, 8)), axis=-1, bitorder="little")[..., 0]


def activations(rng: np.random.Generator, nvec: int, n: int, outliers: float = 0.0,
                outlier_value: float = 20.0) -> np.ndarray:
    """float32 [nvec, n] N(0,1) activations; a fraction `outliers` of positions
    per vector (drawn without replacement) set to +-outlier_value."""
    x = rng.standard_normal((nvec, n)).astype(np.float32)
    k = int(round(outliers * n))
    for v in range(nvec if k else 0):
        pos = rng.choice(n, size=k, replace=False)
        sgn = np.where(rng.integers(0, 2, size=k) == 1, 1.0, -1.0)
        x[v, pos] = (sgn * outlier_value).astype(np.float32)
    return x


def raw_quants(rng: np.random.Generator, nvec: int, n: int, scale: str = "lognormal",
               m128_frac: float = 0.02):
    """Raw q8_0 activations not produced by the quantizer: quants uniform over
    [-128, 127] with a further fraction `m128_frac` forced to -128, and binary16
    scale bits from `scale`.  Returns (q int8 [nvec, n], d uint16 [nvec, n/32])."""
    if n % QK8:
        raise ValueError("n must be a multiple of 32")
    q = rng.integers(-128, 128, size=(nvec, n), dtype=np.int16)
    if m128_frac > 0:
        mask = rng.random((nvec, n)) < m128_frac
        q[mask] = -128
    d = block_scales(rng, (nvec, n // QK8), scale)
    return q.astype(np.int8), d


def ternary_codes(rng: np.random.Generator, shape, p_zero: float = 1.0 / 3.0) -> np.ndarray:
    """uint8 codes 0/1/2 (values -1/0/+1): zero with probability p_zero, the
    two signs equally likely otherwise."""
    u = rng.random(shape)
    half = (1.0 - p_zero) / 2.0
    return np.where(u < half, 0, np.where(u < half + p_zero, 1, 2)).astype(np.uint8)


def assemble_ternary_blocks(scale_bits: np.ndarray, codes: np.ndarray) -> np.ndarray:
    """Lay out [rows, nb] scale bits and [rows, nb, 128] codes as 34-byte blocks."""
    rows, nb = scale_bits.shape
    codes = np.asarray(codes, dtype=np.uint8)
    if codes.shape != (rows, nb, 128) or codes.max(initial=0) > 3:
        raise ValueError("codes must be [rows, nb, 128] values 0..3")
    c = codes.reshape(rows, nb, 32, 4)
    packed = c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)
    blocks = np.empty((rows, nb, Q2_BLOCK_BYTES), dtype=np.uint8)
    s = np.ascontiguousarray(scale_bits, dtype=np.uint16)
    blocks[:, :, 0] = (s & 0xFF).astype(np.uint8)
    blocks[:, :, 1] = (s >> 8).astype(np.uint8)
    blocks[:, :, 2:] = packed
    return blocks


def ternary_blocks(rng: np.random.Generator, rows: int, n: int, scale: str = "halfnormal",
                   p_zero: float = 1.0 / 3.0) -> np.ndarray:
    """Random Q2_0 weight blocks uint8 [rows, n/128, 34]."""
    if n % QK1:
        raise ValueError("n must be a multiple of 128")
    nb = n // QK1
    codes = ternary_codes(rng, (rows, nb, QK1), p_zero)
    scales = block_scales(rng, (rows, nb), scale)
    return assemble_ternary_blocks(scales, codes)


def ternary_blocks_fast(rng: np.random.Generator, rows: int, n: int, scale: str = "halfnormal") -> np.ndarray:
    """Random Q2_0 blocks for full-size sets: uniform random code bytes with
    every code 3 replaced by 1, i.e. P(-1) = P(+1) = 1/4, P(0) = 1/2."""
    if n % QK1:
        raise ValueError("n must be a multiple of 128")
    nb = n // QK1
    b = rng.integers(0, 256, size=(rows, nb, 32), dtype=np.uint8)
    both = b & (b >> 1) & np.uint8(0x55)      # low bit of every 2-bit field that is 3
    b &= ~(both << 1).astype(np.uint8)        # 3 -> 1
    blocks = np.empty((rows, nb, Q2_BLOCK_BYTES), dtype=np.uint8)
    sbits = block_scales(rng, (rows, nb), scale)
    blocks[:, :, 0] = (sbits & 0xFF).astype(np.uint8)
    blocks[:, :, 1] = (sbits >> 8).astype(np.uint8)
    blocks[:, :, 2:] = b
    return blocks
