"""fp64 CPU definition of the FP8 forward: rotation, block quantisation, and
the exact attention of the quantised operands.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product never
imports this module.

[Interrogating-5] "What did FlashAttention-3 do with Hopper?": FP8 attention
quantises per block after a random Hadamard rotation, which spreads outliers
across the block and cuts the error well below plain FP8.  [FA-versions]
"FlashAttention-3 (2024)", "FP8 with incoherent processing": block-level
quantisation instead of a naive per-tensor quantisation that degrades on
outliers.

Readings taken here (the pages give no formulas):
* the rotation is R = diag(s) H / sqrt(d), with H the Sylvester Hadamard
  matrix and s a vector of random signs; a row x becomes x R.  Queries and
  keys are rotated by the same R, so (Q R)(K R)^T = Q K^T exactly;
* FP8 is the OCP E4M3 format (4 exponent bits, bias 7, 3 fraction bits,
  largest finite value 448), rounding to nearest with ties to even and
  saturating at +-448;
* queries and keys are quantised per block of 128 rows of one head, with the
  scale max|x R| / 448 of the block; values are quantised per channel of one
  head over the whole sequence (scale max_n |v_nc| / 448), so that the scale
  is constant along the P V sum and applies once to the output;
* a quantised code is a decision that floating point takes, so it is taken
  in the kernel's precision: the value (x R rounded to fp32, or the bf16 v
  itself) is multiplied in fp32 by the fp32 reciprocal scale 448 / max, and
  that fp32 product is rounded to E4M3.  (In fp64 the products that land
  exactly on an E4M3 midpoint would round differently from fp32 about half
  of the time when 448 / max is not exact.)  The scales used to dequantise
  stay fp64;
* "plain FP8" is one per-tensor scale max|x| / 448 for each of Q, K, V of a
  head, no rotation.
"""

from __future__ import annotations

import numpy as np

from .attention import attention_fwd_ref

E4M3_MAX = 448.0
BLOCK = 128


def e4m3_round(x) -> np.ndarray:
    """Nearest E4M3 value (ties to even), saturating at +-448.

    A normal E4M3 number of binade 2^e (e >= -6) is a multiple of 2^(e-3)
    (three fraction bits); below 2^-6 the values are the subnormal multiples
    of 2^-9.  np.round rounds half to even.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    quantum = np.exp2(np.maximum(e, -6.0) - 3.0)
    r = np.minimum(np.round(a / quantum) * quantum, E4M3_MAX)
    return np.copysign(r, x)


def sylvester_hadamard(d: int) -> np.ndarray:
    """H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]] (d a power of two)."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def rotation_matrix(signs) -> np.ndarray:
    """R = diag(s) H / sqrt(d): orthogonal, so (Q R)(K R)^T = Q K^T."""
    s = np.asarray(signs, dtype=np.float64)
    d = s.shape[0]
    return (s[:, None] * sylvester_hadamard(d)) / np.sqrt(d)


def _scale_of(amax: np.ndarray) -> np.ndarray:
    """max|x| / 448, and 1 where the block is all zeros."""
    return np.where(amax > 0, amax / E4M3_MAX, 1.0)


def _codes(x: np.ndarray, amax) -> np.ndarray:
    """E4M3 codes of x / (max / 448), decided in fp32 (see the module notes):
    RN(fp32(x) * RN_fp32(448 / max)), then rounded to E4M3."""
    amax32 = np.asarray(amax, dtype=np.float32)
    inv = np.where(amax32 > 0, np.float32(E4M3_MAX) / np.where(amax32 > 0, amax32, np.float32(1)), np.float32(1))
    prod = np.asarray(x, dtype=np.float32) * inv.astype(np.float32)
    return e4m3_round(prod.astype(np.float64))


def quantize_rows_per_block(x, signs=None, block: int = BLOCK):
    """x [N, d] of one head -> (x8 [N, d] E4M3 values, scales [ceil(N/block)]).

    Rows are rotated by R when ``signs`` is given, then each block of
    ``block`` rows gets its own scale.  x8 * scale of its block is the
    dequantised (rotated) operand.
    """
    x = np.asarray(x, dtype=np.float64)
    xr = x @ rotation_matrix(signs) if signs is not None else x
    n = xr.shape[0]
    nb = (n + block - 1) // block
    scales = np.empty(nb)
    x8 = np.empty_like(xr)
    for b in range(nb):
        rows = slice(b * block, min(n, (b + 1) * block))
        amax = np.abs(xr[rows].astype(np.float32)).max()
        scales[b] = _scale_of(np.float64(amax))
        x8[rows] = _codes(xr[rows], amax)
    return x8, scales


def quantize_columns(x):
    """x [N, d] of one head -> (x8, scales [d]): one scale per channel."""
    x = np.asarray(x, dtype=np.float64)
    amax = np.abs(x).max(axis=0)
    return _codes(x, amax[None, :]), _scale_of(amax)


def quantize_per_tensor(x):
    """Plain FP8: one scale for the whole [N, d] operand of one head."""
    x = np.asarray(x, dtype=np.float64)
    amax = np.abs(x).max()
    return _codes(x, amax), float(_scale_of(amax))


def dequantized_operands(q, k, v, signs):
    """The operands the FP8 forward multiplies, dequantised to fp64:
    Q R and K R quantised per 128-row block, V quantised per channel."""
    q8, sq = quantize_rows_per_block(q, signs)
    k8, sk = quantize_rows_per_block(k, signs)
    v8, sv = quantize_columns(v)
    qd = q8 * np.repeat(sq, BLOCK)[: q8.shape[0], None]
    kd = k8 * np.repeat(sk, BLOCK)[: k8.shape[0], None]
    return qd, kd, v8 * sv[None, :]


def attention_fwd_fp8_ref(q, k, v, signs, scale: float, causal: bool):
    """Exact (fp64) attention of the quantised operands of one head.

    The FP8 forward computes this up to the rounding of the probabilities P
    to E4M3 before the P V product (and fp32 accumulation); the rotation
    leaves the scores unchanged, so no inverse rotation is needed.
    """
    qd, kd, vd = dequantized_operands(q, k, v, signs)
    return attention_fwd_ref(qd, kd, vd, scale, causal)


def attention_fwd_fp8_plain_ref(q, k, v, scale: float, causal: bool):
    """Exact attention of per-tensor quantised operands (plain FP8, no rotation)."""
    q8, sq = quantize_per_tensor(q)
    k8, sk = quantize_per_tensor(k)
    v8, sv = quantize_per_tensor(v)
    return attention_fwd_ref(q8 * sq, k8 * sk, v8 * sv, scale, causal)
