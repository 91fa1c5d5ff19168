"""Memory stays linear in N: the library keeps no N x N buffer and allocates
nothing.

On the 32k-token workload (B = 1, H = 8, N = 32768, d = 128, causal) one
head's N x N bf16 score matrix alone would be 2 GiB.  With every caller
buffer (inputs, outputs, the backward workspace of an fp32 dQ accumulator and
two padded per-row vectors, about 135 MB) allocated beforehand, a forward and
a backward through the C ABI must leave torch's allocator untouched and move
the driver's free device memory by at most 64 MB.  A first call on a small
problem loads the kernels before anything is measured.
"""

import math

import pytest
import torch

from exact_tiled_attention_08_gb300 import fa
from exact_tiled_attention_08_gb300.workloads import WORKLOADS, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_tiled_attention_08_gb300.build import build_library

    build_library()
    fa.load_library()
    assert torch.cuda.is_available()


def fwd_bwd(t, scale, causal):
    fa.fa_fwd(t["q"], t["k"], t["v"], t["o"], t["lse"], scale, causal)
    fa.fa_bwd(t["q"], t["k"], t["v"], t["o"], t["do"], t["lse"], t["dq"], t["dk"], t["dv"], t["ws"], scale, causal)


def buffers(inp):
    t = {x: inp[x].cuda() for x in ("q", "k", "v", "do")}
    B, H, N, d = t["q"].shape
    t["o"], t["dq"], t["dk"], t["dv"] = (torch.empty_like(t["q"]) for _ in range(4))
    t["lse"] = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    t["ws"] = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    return t


def test_memory_linear_in_n_on_the_32k_workload():
    w = WORKLOADS["causal_long_b1_h8_n32768_d128"]
    # load the kernels (same instantiations) on a small problem first
    small = buffers(make_inputs(1, 1, 256, w.d, seed=31))
    fwd_bwd(small, w.scale, w.causal)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK

    t = buffers(workload_inputs(w))
    # the workspace: the fp32 dQ accumulator and two padded fp32 per-row
    # vectors (each part rounded up to 256 bytes), O(N d), not O(N^2)
    rows, npad = w.B * w.H * w.N, w.B * w.H * (-(-w.N // 128) * 128)
    assert t["ws"].numel() <= rows * w.d * 4 + 2 * npad * 4 + 3 * 256
    assert t["ws"].numel() < w.N * w.N * 2 // 8
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    allocated0 = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    fwd_bwd(t, w.scale, w.causal)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert fa.fa_check_device_status() == fa.FA_OK
    assert torch.cuda.max_memory_allocated() == allocated0
    assert free0 - free1 <= 64 << 20, (free0 - free1) / 2**20
    assert torch.isfinite(t["dq"].float()).all() and torch.isfinite(t["o"].float()).all()
    assert math.isfinite(float(t["lse"].min()))
