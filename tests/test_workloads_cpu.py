"""The seeded synthetic inputs (workloads.py) follow their stated recipe.

Every tensor is fp32 ``randn`` from ``torch.Generator('cpu')`` seeded per
workload, drawn in the order Q, K, V, dO and cast to bf16; the rescale-stress
workload multiplies ceil(1% of N) key rows from the last quarter of the
sequence by 8, the same rows for every (batch, head).  Both the GPU parity
tests and the oracle tests draw their inputs here, so these checks pin what
both sides see.
"""

import math

import numpy as np
import torch

from exact_tiled_attention_08_gb300.workloads import (
    WORKLOADS,
    make_inputs,
    make_outlier_inputs,
    outlier_key_rows,
    rotation_signs,
    to_f32_numpy,
    workload_inputs,
)


def test_the_five_workloads():
    want = {
        "tiny_b1_h1_n128_d128": (1, 1, 128, 128, False, False),
        "b4_h16_n2048_d128": (4, 16, 2048, 128, False, False),
        "causal_b2_h32_n8192_d128": (2, 32, 8192, 128, True, False),
        "causal_long_b1_h8_n32768_d128": (1, 8, 32768, 128, True, False),
        "rescale_stress_b16_h16_n1024_d64": (16, 16, 1024, 64, False, True),
    }
    assert set(WORKLOADS) == set(want)
    seeds = set()
    for name, (B, H, N, d, causal, outliers) in want.items():
        w = WORKLOADS[name]
        assert (w.B, w.H, w.N, w.d, w.causal, w.key_outliers) == (B, H, N, d, causal, outliers)
        assert w.scale == 1.0 / math.sqrt(d)
        f = 4.0 * N * N * d * B * H * (0.5 if causal else 1.0)
        assert w.fwd_flops() == f and w.bwd_flops() == 2.5 * f
        seeds.add(w.seed)
    assert len(seeds) == len(want)


def test_inputs_are_reproducible_and_seeded():
    a = make_inputs(1, 2, 100, 64, seed=5)
    b = make_inputs(1, 2, 100, 64, seed=5)
    c = make_inputs(1, 2, 100, 64, seed=6)
    for x in ("q", "k", "v", "do"):
        assert a[x].dtype == torch.bfloat16 and a[x].shape == (1, 2, 100, 64)
        assert torch.equal(a[x], b[x])
        assert not torch.equal(a[x], c[x])


def test_draw_order_and_bf16_rounding():
    """Q, K, V, dO are the first four randn draws of the seeded generator, in
    that order, each rounded to bf16; dropping dO leaves Q, K, V unchanged."""
    shape = (2, 3, 50, 64)
    gen = torch.Generator("cpu").manual_seed(11)
    draws = [torch.randn(shape, generator=gen, dtype=torch.float32) for _ in range(4)]
    got = make_inputs(*shape, seed=11)
    for x, ref in zip(("q", "k", "v", "do"), draws):
        assert torch.equal(got[x], ref.to(torch.bfloat16))
    no_do = make_inputs(*shape, seed=11, with_dout=False)
    assert "do" not in no_do and all(torch.equal(no_do[x], got[x]) for x in ("q", "k", "v"))
    # the widening to float32 on the host is exact
    f = to_f32_numpy(got["q"])
    assert f.dtype == np.float32 and torch.equal(torch.from_numpy(f).to(torch.bfloat16), got["q"])


def test_outlier_rows_of_the_rescale_stress_workload():
    w = WORKLOADS["rescale_stress_b16_h16_n1024_d64"]
    # a small batch of heads with the workload's N and d: against the same
    # draws without outliers, exactly the outlier rows change, by x8
    plain = make_inputs(2, 3, w.N, w.d, w.seed)
    stress = make_inputs(2, 3, w.N, w.d, w.seed, key_outliers=True)
    for x in ("q", "v", "do"):
        assert torch.equal(plain[x], stress[x])
    kp, ks = plain["k"].float(), stress["k"].float()
    scaled = (ks != kp).any(dim=-1)  # [B, H, N]: rows that changed
    rows = torch.nonzero(scaled[0, 0]).flatten()
    assert len(rows) == math.ceil(0.01 * w.N) == 11
    assert (rows >= 3 * w.N // 4).all() and (rows < w.N).all()
    assert (scaled == scaled[0, 0]).all()  # the same rows for every (batch, head)
    assert torch.equal(ks[:, :, rows], 8.0 * kp[:, :, rows])  # exact: times 8 in bf16
    # the full workload: 11 rows per head whose keys are ~8x larger (mean
    # |k| ~ 6.4 against ~0.8), the same rows for every (batch, head), in the
    # last quarter of the sequence
    full = workload_inputs(w, with_dout=False)["k"].float().abs().mean(dim=-1)  # [B, H, N]
    big = full > 3.0
    assert (big.sum(dim=-1) == 11).all() and (big == big[0, 0]).all()
    big_rows = torch.nonzero(big[0, 0]).flatten()
    assert (big_rows >= 3 * w.N // 4).all()
    gen = torch.Generator("cpu").manual_seed(0)
    r = outlier_key_rows(w.N, gen)
    assert len(set(r.tolist())) == len(r) == 11


def test_rotation_signs():
    s = rotation_signs(128, 21)
    assert s.dtype == torch.int8 and s.shape == (128,)
    assert set(s.tolist()) == {-1, 1}
    assert torch.equal(s, rotation_signs(128, 21)) and not torch.equal(s, rotation_signs(128, 22))
    assert 32 <= int((s == 1).sum()) <= 96


def test_scattered_outlier_inputs():
    """Entries are N(0, 1) plus, with probability frac, an extra N(0, 10^2):
    against frac = 0 (the same draws, no hits) about frac of the entries move."""
    shape = (1, 4, 1024, 128)
    base = make_outlier_inputs(*shape, seed=62, frac=0.0)
    hit = make_outlier_inputs(*shape, seed=62, frac=1e-3)
    n = math.prod(shape)
    for x in ("q", "k", "v"):
        moved = int((hit[x] != base[x]).sum())
        assert abs(moved - 1e-3 * n) <= 5 * math.sqrt(1e-3 * n), (x, moved)
        s = base[x].float()
        assert abs(float(s.mean())) < 0.01 and abs(float(s.std()) - 1.0) < 0.01
