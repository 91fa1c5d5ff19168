"""Deterministic backward (fa_bwd_deterministic, through the C ABI): parity
with the fp64 oracle, bitwise repeatability, and agreement with fa_bwd.

dQ comes from a separate query-major pass that sums dS K over the key blocks
in a fixed order, so two runs on the same inputs give identical bits; dK and dV
come from the same key-major products as in fa_bwd (same order of
accumulation), so they equal fa_bwd's bit for bit.

Tolerance against the oracle: max abs error <= 2e-2 * max|reference| per
tensor (1e-5 absolute where the reference is identically zero, N = 1), as for
fa_bwd.
"""

import math

import numpy as np
import pytest
import torch

from exact_tiled_attention_08_gb300 import fa
from exact_tiled_attention_08_gb300.workloads import WORKLOADS, make_inputs, to_f32_numpy, workload_inputs
from oracle import attention_bwd_ref

pytestmark = pytest.mark.gpu

GRAD_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_tiled_attention_08_gb300.build import build_library

    build_library()
    fa.load_library()
    assert torch.cuda.is_available()


def run_both(inp, scale, causal):
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    o, lse = fa.attention_forward(q, k, v, scale, causal)
    det = [fa.attention_backward(q, k, v, o, do, lse, scale, causal, deterministic=True) for _ in range(2)]
    atomic = fa.attention_backward(q, k, v, o, do, lse, scale, causal)
    st = fa.fa_check_device_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return det, atomic


def check_oracle(inp, grads, scale, causal, heads):
    for b, h in heads:
        qn, kn, vn, don = (to_f32_numpy(inp[x][b, h]) for x in ("q", "k", "v", "do"))
        refs = attention_bwd_ref(qn, kn, vn, don, scale, causal)
        for name, g, r in zip(("dq", "dk", "dv"), grads, refs):
            err = np.abs(to_f32_numpy(g[b, h]) - r).max()
            ref_max = np.abs(r).max()
            if ref_max > 0:
                assert err <= GRAD_TOL * ref_max, (name, b, h, err / ref_max)
            else:
                assert err <= 1e-5, (name, b, h, err)


def check_det(det, atomic):
    (dq0, dk0, dv0), (dq1, dk1, dv1) = det
    dq_a, dk_a, dv_a = atomic
    # bitwise repeatable
    assert torch.equal(dq0, dq1) and torch.equal(dk0, dk1) and torch.equal(dv0, dv1)
    # dK, dV: the same products in the same order as fa_bwd
    assert torch.equal(dk0, dk_a) and torch.equal(dv0, dv_a)
    # dQ: the same sum in another order
    ref = dq_a.float()
    assert (dq0.float() - ref).abs().max().item() <= 1e-2 * max(ref.abs().max().item(), 1e-30) or \
        (dq0.float() - ref).abs().max().item() <= 1e-5


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 127, 128, 129, 257, 384, 1000])
@pytest.mark.parametrize("d", [64, 128])
def test_deterministic_small_and_ragged(N, d, causal):
    inp = make_inputs(1, 2, N, d, seed=400 + N + d)
    scale = 1.0 / math.sqrt(d)
    det, atomic = run_both(inp, scale, causal)
    check_oracle(inp, det[0], scale, causal, [(0, 0), (0, 1)])
    check_det(det, atomic)


@pytest.mark.parametrize("d", [64, 128])
def test_deterministic_rescale_stress_and_heads(d):
    inp = make_inputs(2, 3, 700, d, seed=41, key_outliers=True)
    scale = 1.0 / math.sqrt(d)
    for causal in (False, True):
        det, atomic = run_both(inp, scale, causal)
        check_oracle(inp, det[0], scale, causal, [(0, 0), (1, 2)])
        check_det(det, atomic)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_deterministic_full_size_workloads(name):
    w = WORKLOADS[name]
    inp = workload_inputs(w)
    det, atomic = run_both(inp, w.scale, w.causal)
    check_det(det, atomic)
    # one sampled head against the oracle where it finishes in seconds (the
    # 32k-token workload is covered through fa_bwd, itself checked against the
    # oracle on sampled heads)
    if w.N <= 8192:
        check_oracle(inp, det[0], w.scale, w.causal, [(w.B - 1, w.H - 1)])
