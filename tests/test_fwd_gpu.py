"""Forward parity: the CUDA kernel (through the C ABI) against the fp64 oracle.

Tolerances: O max abs error <= 1e-2, LSE max abs error <= 1e-3.
"""

import math

import numpy as np
import pytest
import torch

from exact_tiled_attention_08_gb300 import fa
from exact_tiled_attention_08_gb300.workloads import WORKLOADS, make_inputs, to_f32_numpy, workload_inputs
from oracle import attention_fwd_ref

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_tiled_attention_08_gb300.build import build_library

    build_library()
    fa.load_library()
    assert torch.cuda.is_available()


def gpu_forward(inp, scale, causal):
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    o, lse = fa.attention_forward(q, k, v, scale, causal)
    st = fa.fa_check_device_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return o, lse


def check_heads(inp, o, lse, scale, causal, heads=None):
    B, H = inp["q"].shape[:2]
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    worst_o = worst_l = 0.0
    for b, h in heads:
        qn, kn, vn = (to_f32_numpy(inp[x][b, h]) for x in ("q", "k", "v"))
        o_ref, l_ref = attention_fwd_ref(qn, kn, vn, scale, causal)
        eo = np.abs(to_f32_numpy(o[b, h]) - o_ref).max()
        el = np.abs(lse[b, h].cpu().numpy() - l_ref).max()
        worst_o, worst_l = max(worst_o, eo), max(worst_l, el)
    assert worst_o <= O_TOL, worst_o
    assert worst_l <= LSE_TOL, worst_l
    return worst_o, worst_l


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 127, 128, 129, 255, 256, 257, 384, 1000])
@pytest.mark.parametrize("d", [64, 128])
def test_forward_small_and_ragged(N, d, causal):
    inp = make_inputs(1, 2, N, d, seed=100 + N + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = gpu_forward(inp, scale, causal)
    check_heads(inp, o, lse, scale, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_several_heads_and_batches(causal):
    inp = make_inputs(3, 5, 640, 128, seed=5)
    o, lse = gpu_forward(inp, 0.07, causal)
    check_heads(inp, o, lse, 0.07, causal)


@pytest.mark.parametrize("d", [64, 128])
def test_forward_rescale_stress(d):
    # keys scaled x8 late in the sequence: the running max jumps after several
    # blocks have been accumulated, exercising the conditional rescale
    inp = make_inputs(2, 2, 1024, d, seed=11, key_outliers=True)
    scale = 1.0 / math.sqrt(d)
    for causal in (False, True):
        o, lse = gpu_forward(inp, scale, causal)
        check_heads(inp, o, lse, scale, causal)


def test_forward_large_scale_forces_every_rescale():
    # A scale of 1 with N(0,1) inputs at d=128 gives scores with s.d. ~11: most
    # blocks raise the row maximum by more than the rescale threshold and each
    # row puts nearly all its weight on one or two keys.  The bound here is the
    # one bf16 arithmetic itself imposes, larger than the 1e-2 bar of the
    # standard workloads:
    #  * P is rounded to bf16 before P V, |p^/p - 1| <= 2^-9, and O's
    #    normaliser (the fp32 sum plus the rounding error of each key block's
    #    largest p) is within 2^-9 of the sum of the p^ that weight V, so each
    #    weight moves by at most 2^-8 w_k and O by at most 2^-8 max|V|;
    #  * storing O in bf16 costs at most half an ulp, 2^-8 |O|;
    #  * plus 1e-3 for fp32 accumulation.
    # The observed error is reported (and held to half the bound, where it has
    # stayed: 0.35-0.36 of it at d = 128 and d = 64, causal or not).
    for d in (128, 64):
        for causal in (False, True):
            inp = make_inputs(1, 2, 1024, d, seed=12)
            o, lse = gpu_forward(inp, 1.0, causal)
            for h in range(2):
                qn, kn, vn = (to_f32_numpy(inp[x][0, h]) for x in ("q", "k", "v"))
                o_ref, l_ref = attention_fwd_ref(qn, kn, vn, 1.0, causal)
                err = np.abs(to_f32_numpy(o[0, h]) - o_ref)
                bound = 2.0 ** -8 * (np.abs(vn).max() + np.abs(o_ref)) + 1e-3
                ratio = float((err / bound).max())
                print(f"d={d} causal={causal} head {h}: max |O - ref| {err.max():.3e}, {ratio:.3f} of the bound")
                assert ratio <= 0.5, (d, causal, h, ratio)
                assert np.abs(lse[0, h].cpu().numpy() - l_ref).max() <= LSE_TOL


def test_equal_scores_give_mean_and_log_count():
    N, d = 700, 128
    inp = make_inputs(1, 1, N, d, seed=13)
    inp["q"] = torch.zeros_like(inp["q"])
    v = to_f32_numpy(inp["v"][0, 0]).astype(np.float64)
    o, lse = gpu_forward(inp, 0.1, False)
    assert np.abs(to_f32_numpy(o[0, 0]) - v.mean(0)).max() <= O_TOL
    assert np.abs(lse[0, 0].cpu().numpy() - math.log(N)).max() <= LSE_TOL
    o, lse = gpu_forward(inp, 0.1, True)
    prefix = np.cumsum(v, axis=0) / np.arange(1, N + 1)[:, None]
    assert np.abs(to_f32_numpy(o[0, 0]) - prefix).max() <= O_TOL
    assert np.abs(lse[0, 0].cpu().numpy() - np.log(np.arange(1, N + 1))).max() <= LSE_TOL


def test_constant_values_and_single_key():
    inp = make_inputs(1, 2, 300, 64, seed=14)
    row = inp["v"][:, :, :1, :]
    inp["v"] = row.expand_as(inp["v"]).contiguous()
    o, _ = gpu_forward(inp, 0.125, False)
    ref = to_f32_numpy(row).astype(np.float64)
    assert np.abs(to_f32_numpy(o) - ref).max() <= O_TOL
    one = make_inputs(2, 2, 1, 128, seed=15)
    o, lse = gpu_forward(one, 0.3, True)
    assert np.abs(to_f32_numpy(o) - to_f32_numpy(one["v"])).max() == 0.0
    dot = (to_f32_numpy(one["q"]).astype(np.float64) * to_f32_numpy(one["k"])).sum(-1) * 0.3
    assert np.abs(lse.cpu().numpy() - dot).max() <= LSE_TOL


def sampled_heads(B, H, seed):
    g = np.random.default_rng(seed)
    return sorted({(0, 0), (B - 1, H - 1), (int(g.integers(B)), int(g.integers(H)))})


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_forward_full_size_workloads(name):
    w = WORKLOADS[name]
    inp = workload_inputs(w, with_dout=False)
    o, lse = gpu_forward(inp, w.scale, w.causal)
    heads = None if w.B * w.H == 1 else sampled_heads(w.B, w.H, w.seed)
    check_heads(inp, o, lse, w.scale, w.causal, heads)
    # every head: outputs finite, LSE at least the largest visible scaled score
    # of row 0 (key 0 is visible to every row)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    q0 = inp["q"][:, :, 0, :].float().cuda()
    k0 = inp["k"][:, :, 0, :].float().cuda()
    assert (lse[:, :, 0] >= (q0 * k0).sum(-1) * w.scale - LSE_TOL).all()


@pytest.mark.parametrize("soft_quarters", [1, 2])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_forward_with_software_exp2(soft_quarters, causal, d):
    """Part of the exponentials by the pages' cubic 2^n p(f) on the FMA pipe
    (fa_set_exp2_split): same tolerances.  Ragged N, the rescale-stress keys
    (arguments far below 0 and up to the rescale threshold) and a masked
    diagonal all pass through the software path."""
    inp = make_inputs(2, 2, 777, d, seed=300 + d + soft_quarters, key_outliers=True)
    scale = 1.0 / math.sqrt(d)
    fa.fa_set_exp2_split(soft_quarters)
    try:
        o, lse = gpu_forward(inp, scale, causal)
    finally:
        fa.fa_set_exp2_split(0)
    check_heads(inp, o, lse, scale, causal)


def test_exp2_split_rejects_other_values():
    with pytest.raises(fa.FaError):
        fa.fa_set_exp2_split(3)
    with pytest.raises(fa.FaError):
        fa.fa_set_exp2_split(-1)
