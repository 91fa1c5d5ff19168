"""Pins of the FP8 oracle (oracle/fp8.py) against things other than itself.

* E4M3 rounding: torch's float8_e4m3fn cast of float32 values (a library
  routine), the format's 256 codes as fixed points, saturation;
* the Hadamard rotation: the 2 x 2 closed form, H H^T = d I, R orthogonal,
  (Q R)(K R)^T = Q K^T;
* block quantisation: the block maximum maps to +-448 exactly, and every
  element is within half an E4M3 quantum of its input;
* the error claim of the pages (rotation + per-block quantisation against
  per-tensor FP8, on inputs with scattered outliers): the direction and a
  lower bound on the ratio, and no harm on outlier-free inputs.
"""

import math

import numpy as np
import pytest
import torch

from exact_tiled_attention_08_gb300.workloads import make_inputs, make_outlier_inputs, rotation_signs, to_f32_numpy
from oracle import attention_fwd_ref
from oracle.fp8 import (
    E4M3_MAX,
    attention_fwd_fp8_plain_ref,
    attention_fwd_fp8_ref,
    dequantized_operands,
    e4m3_round,
    quantize_columns,
    quantize_per_tensor,
    quantize_rows_per_block,
    rotation_matrix,
    sylvester_hadamard,
)


def test_e4m3_matches_torch_cast_of_float32():
    rng = np.random.default_rng(0)
    x = np.concatenate([np.linspace(-448, 448, 100001), rng.standard_normal(50000) * 3,
                        np.linspace(-0.02, 0.02, 20001), rng.standard_normal(20000) * 1e-3]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(e4m3_round(x), ref)


def test_e4m3_codes_are_fixed_points_and_saturation():
    codes = torch.arange(256, dtype=torch.int16).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = codes[np.isfinite(codes)]
    assert finite.size == 254  # 0x7f and 0xff are NaN in E4M3
    assert np.array_equal(e4m3_round(finite), finite)
    assert np.abs(finite).max() == E4M3_MAX
    assert e4m3_round(1e6) == E4M3_MAX and e4m3_round(-1e6) == -E4M3_MAX
    # spacing: 3 fraction bits in the binade [1, 2), subnormal quantum 2^-9
    assert e4m3_round(1.0 + 1 / 16) == 1.0 and e4m3_round(1.0 + 3 / 16) == 1.25
    assert e4m3_round(2.0 ** -10) == 0.0 and e4m3_round(3 * 2.0 ** -10) == 2 * 2.0 ** -9


def test_hadamard_closed_form_and_orthogonality():
    assert np.array_equal(sylvester_hadamard(2), np.array([[1.0, 1.0], [1.0, -1.0]]))
    for d in (4, 64, 128):
        h = sylvester_hadamard(d)
        assert np.array_equal(h @ h.T, d * np.eye(d))
        r = rotation_matrix(rotation_signs(d, 3).numpy())
        assert np.abs(r @ r.T - np.eye(d)).max() < 1e-12
    with pytest.raises(ValueError):
        sylvester_hadamard(96)


def test_rotation_leaves_scores_unchanged():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal((40, 128)), rng.standard_normal((50, 128))
    r = rotation_matrix(rotation_signs(128, 4).numpy())
    assert np.abs((q @ r) @ (k @ r).T - q @ k.T).max() < 1e-11


def test_block_quantisation_bounds():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((300, 128)) * np.exp(rng.standard_normal((300, 1)))
    signs = rotation_signs(128, 5).numpy()
    x8, sc = quantize_rows_per_block(x, signs)
    assert sc.shape == (3,)
    xr = x @ rotation_matrix(signs)
    for b in range(3):
        rows = slice(128 * b, min(300, 128 * (b + 1)))
        assert np.abs(x8[rows]).max() == E4M3_MAX  # the block maximum maps to +-448 exactly
        err = np.abs(x8[rows] * sc[b] - xr[rows])
        # half a quantum: 2^-4 relative for normal numbers, 2^-10 * scale below 2^-6 * scale
        # (plus the fp32 rounding of the rotated value and of the product, 2^-23 relative)
        bound = np.maximum(2.0 ** -4 * np.abs(xr[rows]), 2.0 ** -10 * sc[b]) + 2.0 ** -22 * np.abs(xr[rows])
        assert (err <= bound).all()
    v8, sv = quantize_columns(x)
    assert (np.abs(v8).max(axis=0) == E4M3_MAX).all()
    t8, st = quantize_per_tensor(x)
    assert np.abs(t8).max() == E4M3_MAX and st == np.abs(x).max() / E4M3_MAX


def test_codes_are_decided_in_fp32():
    # v / (max / 448) on an exact E4M3 midpoint when 448 / max is not exact:
    # the code follows RN_fp32(v * RN_fp32(448 / max)), not the fp64 quotient
    v = np.array([[1.0], [1.2890625 * 1.1875]])  # a bf16 value and the column maximum
    x8, sv = quantize_columns(v)
    inv = np.float32(448) / np.float32(v.max())
    assert x8[0, 0] == e4m3_round(np.float64(np.float32(1.0) * inv))
    assert x8[1, 0] == E4M3_MAX and sv[0] == v.max() / E4M3_MAX


def test_fp8_reference_is_attention_of_dequantised_operands():
    inp = make_inputs(1, 1, 200, 128, seed=6, with_dout=False)
    q, k, v = (to_f32_numpy(inp[x][0, 0]) for x in "qkv")
    signs = rotation_signs(128, 7).numpy()
    qd, kd, vd = dequantized_operands(q, k, v, signs)
    for causal in (False, True):
        o, lse = attention_fwd_fp8_ref(q, k, v, signs, 0.09, causal)
        o2, lse2 = attention_fwd_ref(qd, kd, vd, 0.09, causal)
        assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
        # FP8 operands stay close to exact attention: each quantised value is
        # within 2^-4 of itself relative, so a row that averages few values
        # (early causal rows) can be off by ~2^-4 max|V|; the RMS is far smaller
        oe, _ = attention_fwd_ref(q, k, v, 0.09, causal)
        assert np.abs(o - oe).max() <= 2.0 ** -3 * np.abs(v).max()
        assert _rmse(o, oe) < 0.02


def _rmse(a, b):
    return float(np.sqrt(np.mean((a - b) ** 2)))


@pytest.mark.parametrize("N,d", [(512, 128), (1024, 128), (512, 64)])
def test_rotation_and_blocks_beat_plain_fp8_on_outliers(N, d):
    """[Interrogating-5] "What did FlashAttention-3 do with Hopper?": per-block
    quantisation after a random Hadamard rotation cuts the error below plain
    FP8 (the page quotes 2.6x for its own, unstated, inputs).  Here, on
    N(0,1) entries with 0.1% of them given an extra N(0, 100): the O error of
    the rotated, block-quantised operands is below that of per-tensor FP8 by
    at least 1.25x (measured 1.36-1.76x), and the error that the query and key
    quantisation alone causes drops by at least 1.3x (measured 1.42-2.03x); on
    outlier-free inputs the two schemes are within 5% of each other."""
    scale = 1 / math.sqrt(d)
    signs = rotation_signs(d, 11).numpy()
    out = make_outlier_inputs(1, 2, N, d, seed=5)
    plain = make_inputs(1, 2, N, d, seed=5, with_dout=False)
    e_rot, e_plain, e_qk_rot, e_qk_plain, n_rot, n_plain = [], [], [], [], [], []
    for h in range(2):
        q, k, v = (to_f32_numpy(out[x][0, h]).astype(np.float64) for x in "qkv")
        o, _ = attention_fwd_ref(q, k, v, scale, False)
        e_rot.append(_rmse(attention_fwd_fp8_ref(q, k, v, signs, scale, False)[0], o))
        e_plain.append(_rmse(attention_fwd_fp8_plain_ref(q, k, v, scale, False)[0], o))
        qd, kd, _ = dequantized_operands(q, k, v, signs)
        e_qk_rot.append(_rmse(attention_fwd_ref(qd, kd, v, scale, False)[0], o))
        q8, sq = quantize_per_tensor(q)
        k8, sk = quantize_per_tensor(k)
        e_qk_plain.append(_rmse(attention_fwd_ref(q8 * sq, k8 * sk, v, scale, False)[0], o))
        # the rotated, dequantised scores approximate the exact ones (rotation is exact)
        assert np.abs(qd @ kd.T - q @ k.T).max() <= 0.1 * np.abs(q @ k.T).max()
        qn, kn, vn = (to_f32_numpy(plain[x][0, h]).astype(np.float64) for x in "qkv")
        on, _ = attention_fwd_ref(qn, kn, vn, scale, False)
        n_rot.append(_rmse(attention_fwd_fp8_ref(qn, kn, vn, signs, scale, False)[0], on))
        n_plain.append(_rmse(attention_fwd_fp8_plain_ref(qn, kn, vn, scale, False)[0], on))
    assert np.mean(e_plain) >= 1.25 * np.mean(e_rot)
    assert np.mean(e_qk_plain) >= 1.3 * np.mean(e_qk_rot)
    assert abs(np.mean(n_plain) / np.mean(n_rot) - 1) < 0.05
