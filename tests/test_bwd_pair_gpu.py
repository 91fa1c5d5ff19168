"""fa_bwd_deterministic with its dK/dV products on CTA pairs (fa_set_bwd_pair_mma):
two CTAs on adjacent key blocks run each product as one 256-row tcgen05 MMA
(cta_group::2).  Checked through the C ABI against the fp64 oracle (the same
tolerances as every backward path), for bitwise repeatability, and against
the single-CTA path of the same entry point.

Shapes cover an odd number of key blocks (the last block's partner lies past
N), a first query block that is entirely in the future of the second CTA's
keys (causal), persistent pairs taking several items, causal head groups, and
the full-size d = 128 workloads.
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
    yield
    fa.fa_set_bwd_pair_mma(False)


def backward(q, k, v, o, do, lse, scale, causal, pair):
    fa.fa_set_bwd_pair_mma(pair)
    try:
        return fa.attention_backward(q, k, v, o, do, lse, scale, causal, deterministic=True)
    finally:
        fa.fa_set_bwd_pair_mma(False)


def run(inp, scale, causal):
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    o, lse = fa.attention_forward(q, k, v, scale, causal)
    pair = [backward(q, k, v, o, do, lse, scale, causal, True) for _ in range(2)]
    single = backward(q, k, v, o, do, lse, scale, causal, False)
    assert fa.fa_check_device_status() == fa.FA_OK
    return pair, single


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


def check_pair(pair, single):
    (dq0, dk0, dv0), (dq1, dk1, dv1) = pair
    # bitwise repeatable
    assert torch.equal(dq0, dq1) and torch.equal(dk0, dk1) and torch.equal(dv0, dv1)
    # dQ comes from the same query-major pass
    assert torch.equal(dq0, single[0])
    # dK, dV: the same products on one CTA or two (same sums, possibly in another order)
    for g, r in ((dk0, single[1]), (dv0, single[2])):
        ref = r.float()
        err = (g.float() - ref).abs().max().item()
        assert err <= 1e-2 * max(ref.abs().max().item(), 1e-30) or err <= 1e-5, err


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 127, 128, 129, 255, 257, 384, 640, 1000])
def test_pair_small_and_ragged(N, causal):
    inp = make_inputs(1, 2, N, 128, seed=500 + N)
    scale = 1.0 / math.sqrt(128)
    pair, single = run(inp, scale, causal)
    check_oracle(inp, pair[0], scale, causal, [(0, 0), (0, 1)])
    check_pair(pair, single)


def test_pair_rescale_stress_and_heads():
    inp = make_inputs(2, 3, 700, 128, seed=51, key_outliers=True)
    scale = 1.0 / math.sqrt(128)
    for causal in (False, True):
        pair, single = run(inp, scale, causal)
        check_oracle(inp, pair[0], scale, causal, [(0, 0), (1, 2)])
        check_pair(pair, single)


def test_pair_persistent_items():
    # without the mask the pairs are persistent: 3 * 70 heads x 3 pair items
    # (N = 640: five key blocks, the fifth unpaired) is more than the pairs that
    # run at once, so pairs take several items
    inp = make_inputs(3, 70, 640, 128, seed=52)
    scale = 1.0 / math.sqrt(128)
    pair, single = run(inp, scale, False)
    check_oracle(inp, pair[0], scale, False, [(0, 0), (1, 33), (2, 69)])
    check_pair(pair, single)


def test_pair_causal_head_groups():
    inp = make_inputs(2, 72, 1024, 128, seed=53)
    scale = 1.0 / math.sqrt(128)
    pair, single = run(inp, scale, True)
    check_oracle(inp, pair[0], scale, True, [(0, 0), (0, 71), (1, 37)])
    check_pair(pair, single)


@pytest.mark.parametrize("name", [n for n, w in WORKLOADS.items() if w.d == 128])
def test_pair_full_size_workloads(name):
    w = WORKLOADS[name]
    inp = workload_inputs(w)
    pair, single = run(inp, w.scale, w.causal)
    check_pair(pair, single)
    if w.N <= 8192:
        check_oracle(inp, pair[0], w.scale, w.causal, [(w.B - 1, w.H - 1)])
    else:
        # every head: dK sums to zero over the keys, dV to the sum of dO over the queries
        dk, dv = pair[0][1].double(), pair[0][2].double()
        do = inp["do"].cuda().double()
        scale_dk = dk.abs().max().item() * math.sqrt(w.N)
        assert (dk.sum(dim=2).abs().max().item()) <= GRAD_TOL * scale_dk
        assert ((dv.sum(dim=2) - do.sum(dim=2)).abs().max().item()) <= GRAD_TOL * dv.abs().max().item() * math.sqrt(w.N)
