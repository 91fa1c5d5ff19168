"""FP8 forward (fa_fwd_fp8, through the C ABI) against the FP8 oracle.

Three checks, from the step that is exact to the one that rounds:
* the quantised operands the library writes into its workspace (documented
  layout) equal the oracle's rotation and block quantisation, element by
  element up to one E4M3 quantum where fp32 and fp64 rotations land on
  different sides of a rounding boundary (rare), scales to fp32 rounding;
* O against the exact attention of the oracle's quantised operands, within a
  bound derived from the one remaining rounding, P to E4M3 before the P V
  product: with p_j = e_j scaled so that the largest is >= 1 (the kernel's
  exponent reference is at most 8 binades below the row maximum), rounding
  moves p_j by at most max(2^-4 p_j, 2^-10), and
      |O_gpu - O_ref|_ic <= sum_j max(2^-4 e_j, 2^-10) |v_jc - O_ic| / sum_j e_j
  (the worst case of the scaling), plus bf16 rounding of O (2^-8 |O|) and
  fp32 accumulation slack (2e-3); LSE (unrounded sums) within 2e-3;
* against exact attention of the bf16 inputs: the FP8 error stays small on
  normal inputs and, on inputs with scattered outliers, below the error of
  plain per-tensor FP8 operands (the pages' claim for the rotation and block
  scales).
"""

import math

import numpy as np
import pytest
import torch

from exact_tiled_attention_08_gb300 import fa
from exact_tiled_attention_08_gb300.workloads import (
    WORKLOADS,
    make_inputs,
    make_outlier_inputs,
    rotation_signs,
    to_f32_numpy,
    workload_inputs,
)
from oracle import attention_fwd_ref
from oracle.fp8 import attention_fwd_fp8_plain_ref, dequantized_operands, quantize_columns, quantize_rows_per_block

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_tiled_attention_08_gb300.build import build_library

    build_library()
    fa.load_library()
    assert torch.cuda.is_available()


def run_fp8(inp, signs, scale, causal):
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    B, H, N, d = q.shape
    ws = torch.full((fa.fa_fwd_fp8_workspace_bytes(B, H, N, d),), 0x5A, dtype=torch.uint8, device="cuda")
    o, lse = fa.attention_forward_fp8(q, k, v, signs.cuda(), scale, causal, workspace=ws)
    st = fa.fa_check_device_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return o, lse, ws


def decode_workspace(ws, B, H, N):
    """The quantised operands and scales, from the layout fa.h documents."""
    bh, nkb = B * H, (N + 127) // 128

    def up(x):
        return (x + 255) // 256 * 256

    sizes = [bh * N * D, bh * N * D, bh * nkb * D * 128, bh * nkb * 4, bh * nkb * 4, bh * D * 4, bh * D * 4]
    offs = np.cumsum([0] + [up(s) for s in sizes])
    raw = ws.cpu()

    def e4m3(lo, n, shape):
        return raw[lo:lo + n].view(torch.float8_e4m3fn).to(torch.float64).numpy().reshape(shape)

    def f32(lo, n, shape):
        return raw[lo:lo + 4 * n].view(torch.float32).to(torch.float64).numpy().reshape(shape)

    q8 = e4m3(offs[0], sizes[0], (bh, N, D))
    k8 = e4m3(offs[1], sizes[1], (bh, N, D))
    v8t = e4m3(offs[2], sizes[2], (bh, nkb, D, 128))
    qs = f32(offs[3], bh * nkb, (bh, nkb))
    ks = f32(offs[4], bh * nkb, (bh, nkb))
    vs = f32(offs[6], bh * D, (bh, D))
    return q8, k8, v8t, qs, ks, vs


def within_one_quantum(a, b):
    """|a - b| <= one E4M3 quantum at b's magnitude (2^-3 relative, 2^-9 below 2^-6)."""
    return np.abs(a - b) <= np.maximum(2.0 ** -3 * np.abs(b), 2.0 ** -9) * (1 + 1e-9)


def p_rounding_bound(qd, kd, vd, scale, causal, row_chunk=64):
    """Exact attention of the dequantised operands and the bound above."""
    n = qd.shape[0]
    o_ref, lse_ref = attention_fwd_ref(qd, kd, vd, scale, causal)
    bound = np.empty_like(o_ref)
    for r0 in range(0, n, row_chunk):
        rows = slice(r0, min(n, r0 + row_chunk))
        s = scale * (qd[rows] @ kd.T)
        if causal:
            i = np.arange(rows.start, rows.stop)[:, None]
            s = np.where(np.arange(n)[None, :] > i, -np.inf, s)
        e = np.exp(s - s.max(axis=1, keepdims=True))
        wgt = np.where(np.isfinite(s), np.maximum(2.0 ** -4 * e, 2.0 ** -10), 0.0)
        dev = np.abs(vd[None, :, :] - o_ref[rows][:, None, :])  # [rows, keys, d]
        bound[rows] = np.einsum("rk,rkc->rc", wgt, dev) / e.sum(axis=1, keepdims=True)
    return o_ref, lse_ref, bound


def check_head(inp, b, h, o, lse, signs_np, scale, causal, rows=None):
    """The bound on head (b, h); with ``rows`` (causal only, a multiple of 128)
    on its first ``rows`` query rows, which see only the first ``rows`` keys:
    their query and key blocks are quantised exactly as in the full sequence,
    and V's channel scales are taken over the whole sequence."""
    q, k, v = (to_f32_numpy(inp[x][b, h]).astype(np.float64) for x in ("q", "k", "v"))
    qd, kd, vd = dequantized_operands(q, k, v, signs_np)
    if rows is not None:
        assert causal and rows % 128 == 0
        q, k, v, qd, kd, vd = (t[:rows] for t in (q, k, v, qd, kd, vd))
    o_ref, lse_ref, bound = p_rounding_bound(qd, kd, vd, scale, causal)
    og = to_f32_numpy(o[b, h, : q.shape[0]]).astype(np.float64)
    err = np.abs(og - o_ref)
    limit = bound + 2.0 ** -8 * np.abs(o_ref) + 2e-3
    assert (err <= limit).all(), (b, h, float((err - limit).max()))
    assert np.abs(lse[b, h, : q.shape[0]].cpu().numpy() - lse_ref).max() <= 2e-3
    return og, q, k, v


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [129, 300])
def test_fp8_quantised_operands_match_oracle(N, causal):
    inp = make_inputs(1, 2, N, D, seed=500 + N, with_dout=False)
    signs = rotation_signs(D, 21)
    _, _, ws = run_fp8(inp, signs, 1 / math.sqrt(D), causal)
    q8, k8, v8t, qs, ks, vs = decode_workspace(ws, 1, 2, N)
    nkb = (N + 127) // 128
    for h in range(2):
        for name, g8, gs in (("q", q8, qs), ("k", k8, ks)):
            x8, sc = quantize_rows_per_block(to_f32_numpy(inp[name][0, h]), signs.numpy())
            assert np.allclose(gs[h], sc, rtol=1e-6, atol=0)
            assert within_one_quantum(g8[h], x8).all()
            assert np.mean(g8[h] == x8) >= 0.995
        v8, sv = quantize_columns(to_f32_numpy(inp["v"][0, h]))
        assert np.allclose(vs[h], sv, rtol=1e-6, atol=0)
        pad = np.zeros((nkb * 128, D))
        pad[:N] = v8
        want = pad.reshape(nkb, 128, D).transpose(0, 2, 1)  # per key block: channel rows of 128 keys
        assert within_one_quantum(v8t[h], want).all() and np.mean(v8t[h] == want) >= 0.995


def test_fp8_quantised_operands_many_blocks_per_cta():
    """3 operands x 32 heads x 17 blocks = 1632 blocks of 128 rows: more than
    the preparation has CTAs, so each CTA walks several blocks through both of
    its staging buffers and their barrier phases; N = 2148 leaves a ragged
    last block in every head.  Every head's quantised Q, K and V against the
    oracle, as above."""
    B, H, N = 2, 16, 2148
    inp = make_inputs(B, H, N, D, seed=505, with_dout=False)
    signs = rotation_signs(D, 26)
    _, _, ws = run_fp8(inp, signs, 1 / math.sqrt(D), False)
    q8, k8, v8t, qs, ks, vs = decode_workspace(ws, B, H, N)
    nkb = (N + 127) // 128
    for bh in range(B * H):
        b, h = divmod(bh, H)
        for name, g8, gs in (("q", q8, qs), ("k", k8, ks)):
            x8, sc = quantize_rows_per_block(to_f32_numpy(inp[name][b, h]), signs.numpy())
            assert np.allclose(gs[bh], sc, rtol=1e-6, atol=0), (name, bh)
            assert within_one_quantum(g8[bh], x8).all(), (name, bh)
            assert np.mean(g8[bh] == x8) >= 0.995, (name, bh)
        v8, sv = quantize_columns(to_f32_numpy(inp["v"][b, h]))
        assert np.allclose(vs[bh], sv, rtol=1e-6, atol=0), bh
        pad = np.zeros((nkb * 128, D))
        pad[:N] = v8
        want = pad.reshape(nkb, 128, D).transpose(0, 2, 1)
        assert within_one_quantum(v8t[bh], want).all() and np.mean(v8t[bh] == want) >= 0.995, bh


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 128, 129, 255, 300, 1000])
def test_fp8_forward_small_and_ragged(N, causal):
    inp = make_inputs(1, 2, N, D, seed=600 + N, with_dout=False)
    signs = rotation_signs(D, 22)
    scale = 1 / math.sqrt(D)
    o, lse, _ = run_fp8(inp, signs, scale, causal)
    for h in range(2):
        og, q, k, v = check_head(inp, 0, h, o, lse, signs.numpy(), scale, causal)
        oe, _ = attention_fwd_ref(q, k, v, scale, causal)
        assert np.abs(og - oe).max() <= 2.0 ** -3 * np.abs(v).max()
        assert np.sqrt(np.mean((og - oe) ** 2)) <= 0.03


def test_fp8_several_heads_and_batches():
    inp = make_inputs(2, 3, 640, D, seed=61, with_dout=False)
    signs = rotation_signs(D, 23)
    for causal in (False, True):
        o, lse, _ = run_fp8(inp, signs, 0.07, causal)
        for b, h in ((0, 0), (1, 2), (0, 1)):
            check_head(inp, b, h, o, lse, signs.numpy(), 0.07, causal)


def test_fp8_beats_plain_fp8_on_outliers():
    """On N(0,1) inputs with 0.1% of the entries given an extra N(0, 100),
    the GPU's FP8 forward (rotation, block scales, and P rounded to E4M3) is
    closer to exact attention than exact attention of plain per-tensor FP8
    operands, which does not even round P."""
    N = 1024
    inp = make_outlier_inputs(1, 4, N, D, seed=62)
    signs = rotation_signs(D, 24)
    scale = 1 / math.sqrt(D)
    o, lse, _ = run_fp8(inp, signs, scale, False)
    e_gpu, e_plain = [], []
    for h in range(4):
        og, q, k, v = check_head(inp, 0, h, o, lse, signs.numpy(), scale, False)
        oe, _ = attention_fwd_ref(q, k, v, scale, False)
        op, _ = attention_fwd_fp8_plain_ref(q, k, v, scale, False)
        e_gpu.append(np.sqrt(np.mean((og - oe) ** 2)))
        e_plain.append(np.sqrt(np.mean((op - oe) ** 2)))
    assert np.mean(e_gpu) < np.mean(e_plain), (np.mean(e_gpu), np.mean(e_plain))


@pytest.mark.parametrize("name", ["b4_h16_n2048_d128", "causal_b2_h32_n8192_d128", "causal_long_b1_h8_n32768_d128"])
def test_fp8_full_size_workloads(name):
    """Full-size d = 128 workloads: the bound on a sampled head where the
    oracle's N x N x d bound fits in seconds (N = 2048, every row); with the
    causal mask at N = 8192 and 32768, on the first 1024 query rows of two
    heads (which see only the first 1024 keys), plus all-head sanity."""
    w = WORKLOADS[name]
    inp = workload_inputs(w, with_dout=False)
    signs = rotation_signs(D, 25)
    o, lse, _ = run_fp8(inp, signs, w.scale, w.causal)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    if w.N <= 2048:
        check_head(inp, w.B - 1, w.H - 1, o, lse, signs.numpy(), w.scale, w.causal)
        return
    assert w.causal
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        check_head(inp, b, h, o, lse, signs.numpy(), w.scale, True, rows=1024)
