"""Backward parity: fa_bwd_preprocess and fa_bwd (through the C ABI) against
the fp64 oracle.  The backward consumes the O and LSE that fa_fwd wrote.

Tolerance: dQ, dK, dV max abs error <= 2e-2 * max|reference| per tensor.  When
the reference is identically zero (N = 1: a softmax over a single key has no
gradient with respect to its score, so dQ = dK = 0 exactly) the bound becomes
1e-5 absolute, the size of the fp32 rounding of dP - delta.
"""

import math

import numpy as np
import pytest
import torch

from exact_tiled_attention_08_gb300 import fa
from exact_tiled_attention_08_gb300.workloads import WORKLOADS, make_inputs, to_f32_numpy, workload_inputs
from oracle import attention_bwd_preprocess_ref, attention_bwd_ref

pytestmark = pytest.mark.gpu

GRAD_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_tiled_attention_08_gb300.build import build_library

    build_library()
    fa.load_library()
    assert torch.cuda.is_available()


def gpu_fwd_bwd(inp, scale, causal):
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    o, lse = fa.attention_forward(q, k, v, scale, causal)
    dq, dk, dv = fa.attention_backward(q, k, v, o, do, lse, scale, causal)
    st = fa.fa_check_device_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return o, lse, dq, dk, dv


def check_grads(inp, grads, scale, causal, heads=None):
    B, H = inp["q"].shape[:2]
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    worst = {}
    for b, h in heads:
        qn, kn, vn, don = (to_f32_numpy(inp[x][b, h]) for x in ("q", "k", "v", "do"))
        refs = attention_bwd_ref(qn, kn, vn, don, scale, causal)
        for name, g, r in zip(("dq", "dk", "dv"), grads, refs):
            err = np.abs(to_f32_numpy(g[b, h]) - r).max()
            ref_max = np.abs(r).max()
            rel = err / ref_max if ref_max > 0 else (0.0 if err <= 1e-5 else np.inf)
            worst[name] = max(worst.get(name, 0.0), rel)
    for name, rel in worst.items():
        assert rel <= GRAD_TOL, (name, rel)
    return worst


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 127, 128, 129, 255, 257, 384, 1000])
@pytest.mark.parametrize("d", [64, 128])
def test_backward_small_and_ragged(N, d, causal):
    inp = make_inputs(1, 2, N, d, seed=200 + N + d)
    scale = 1.0 / math.sqrt(d)
    _, _, dq, dk, dv = gpu_fwd_bwd(inp, scale, causal)
    check_grads(inp, (dq, dk, dv), scale, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_several_heads_and_batches(causal):
    inp = make_inputs(2, 3, 640, 128, seed=21)
    _, _, dq, dk, dv = gpu_fwd_bwd(inp, 0.07, causal)
    check_grads(inp, (dq, dk, dv), 0.07, causal)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [128, 300])
def test_backward_ctas_over_several_items(N, d):
    """Without the mask the backward's CTAs stay resident, one per SM, and walk
    the (key block, batch, head) items; with about 2.5 items per SM most CTAs
    take two or three, carrying barrier phases, ring positions and statistics
    entries from one item to the next.  Every head is checked, for fa_bwd and
    for fa_bwd_deterministic (whose dK and dV come from the same kernel)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nkb = (N + 127) // 128
    H = -(-5 * sms // (2 * nkb))
    inp = make_inputs(1, H, N, d, seed=25 + N + d)
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    o, lse = fa.attention_forward(q, k, v, scale, False)
    runs = [fa.attention_backward(q, k, v, o, do, lse, scale, False, deterministic=det) for det in (False, True)]
    st = fa.fa_check_device_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    check_grads(inp, runs[0], scale, False)
    # the deterministic dQ against the oracle; dK, dV bit for bit as fa_bwd's
    check_grads(inp, (runs[1][0], runs[0][1], runs[0][2]), scale, False)
    assert torch.equal(runs[0][1], runs[1][1]) and torch.equal(runs[0][2], runs[1][2])


def test_backward_causal_item_groups():
    """With the mask the key-block items run in groups of heads, costliest key
    block first inside a group.  B = 2, H = 72, N = 1024 (8 key blocks) gives
    two groups of 72 heads on a 152-SM part (the smallest divisor of 144 that
    is at least 4 x 152 / 9); every head is checked, for fa_bwd and for
    fa_bwd_deterministic (whose dQ pass orders its query blocks the same way)."""
    inp = make_inputs(2, 72, 1024, 64, seed=26)
    scale = 1.0 / math.sqrt(64)
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    o, lse = fa.attention_forward(q, k, v, scale, True)
    runs = [fa.attention_backward(q, k, v, o, do, lse, scale, True, deterministic=det) for det in (False, True)]
    st = fa.fa_check_device_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    check_grads(inp, runs[0], scale, True)
    check_grads(inp, (runs[1][0], runs[0][1], runs[0][2]), scale, True)
    assert torch.equal(runs[0][1], runs[1][1]) and torch.equal(runs[0][2], runs[1][2])


@pytest.mark.parametrize("d", [64, 128])
def test_backward_rescale_stress(d):
    inp = make_inputs(2, 2, 1024, d, seed=22, key_outliers=True)
    scale = 1.0 / math.sqrt(d)
    for causal in (False, True):
        _, _, dq, dk, dv = gpu_fwd_bwd(inp, scale, causal)
        check_grads(inp, (dq, dk, dv), scale, causal)


@pytest.mark.parametrize("d", [64, 128])
def test_preprocess_matches_rowsum(d):
    inp = make_inputs(2, 3, 333, d, seed=23)
    o, do = inp["q"].cuda(), inp["do"].cuda()   # any bf16 tensors serve as O and dO
    delta = torch.empty((2, 3, 333), dtype=torch.float32, device="cuda")
    fa.fa_bwd_preprocess(o, do, delta)
    assert fa.fa_check_device_status() == fa.FA_OK
    ref = attention_bwd_preprocess_ref(to_f32_numpy(inp["q"]), to_f32_numpy(inp["do"]))
    assert np.abs(delta.cpu().numpy() - ref).max() <= 1e-5 * np.abs(ref).max()


def test_backward_overwrites_outputs_and_ignores_stale_workspace():
    inp = make_inputs(1, 2, 300, 128, seed=24)
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(128)
    o, lse = fa.attention_forward(q, k, v, scale, True)
    ws = torch.full((fa.fa_bwd_workspace_bytes(1, 2, 300, 128),), 0x7F, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, scale, True)
        assert fa.fa_check_device_status() == fa.FA_OK
        outs.append((dq, dk, dv))
    check_grads(inp, outs[0], scale, True)
    for a, b in zip(*outs):
        # dK, dV are deterministic; dQ differs only by the order of fp32 atomics
        assert (a.float() - b.float()).abs().max().item() <= 1e-2 * b.float().abs().max().item()


def sampled_heads(B, H, seed):
    g = np.random.default_rng(seed)
    return sorted({(0, 0), (B - 1, H - 1), (int(g.integers(B)), int(g.integers(H)))})


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_backward_full_size_workloads(name):
    w = WORKLOADS[name]
    inp = workload_inputs(w)
    _, _, dq, dk, dv = gpu_fwd_bwd(inp, w.scale, w.causal)
    heads = None if w.B * w.H == 1 else sampled_heads(w.B, w.H, w.seed)
    check_grads(inp, (dq, dk, dv), w.scale, w.causal, heads)
    # every head: the exact-arithmetic invariants sum_j dK_j = 0 and
    # sum_j dV_j = sum_i dO_i, to within bf16 accumulation noise
    do = inp["do"].cuda().float()
    sum_dk = dk.float().sum(dim=2)
    sum_dv = dv.float().sum(dim=2)
    tol_k = 2e-2 * dk.float().abs().amax(dim=(2, 3)) * math.sqrt(w.N)
    tol_v = 2e-2 * dv.float().abs().amax(dim=(2, 3)) * math.sqrt(w.N)
    assert ((sum_dk.abs().amax(dim=-1)) <= tol_k).all()
    assert (((sum_dv - do.sum(dim=2)).abs().amax(dim=-1)) <= tol_v).all()
    assert torch.isfinite(dq.float()).all()
