"""fa_bwd_static_scratch: the backward pass for callers that cannot allocate
device memory when they call it (for example a plug-in inside a runtime that
owns all device memory through its own arena, or a program that must keep a
fixed device-memory footprint once started).  It takes no workspace and uses a
fixed array inside the library instead.

The test calls it through the C ABI twice in a row, on different inputs, and
compares each result with fa_bwd's on the same inputs within the backward
tolerance the other tests use (2e-2 x max|reference|).  The second call would
see the first call's leftovers in the shared array if the entry point did not
re-initialise them.  This file is named so that pytest collects it last.
"""

import ctypes
import gc
import math

import pytest
import torch

from exact_tiled_attention_08_gb300 import fa
from exact_tiled_attention_08_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_tiled_attention_08_gb300.build import build_library

    build_library()
    fa.load_library()
    assert torch.cuda.is_available()


def forward(q, k, v, scale, causal):
    o, lse = fa.attention_forward(q, k, v, scale, causal)
    assert fa.fa_check_device_status() == fa.FA_OK
    return o, lse


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_static_scratch_matches_workspace_backward_twice(d, causal):
    B, H, N = 2, 3, 700
    scale = 1.0 / math.sqrt(d)
    lib = fa.load_library()
    for call, seed in enumerate((41, 42)):
        inp = make_inputs(B, H, N, d, seed=seed)
        q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
        o, lse = forward(q, k, v, scale, causal)
        ref = fa.attention_backward(q, k, v, o, do, lse, scale, causal)
        assert fa.fa_check_device_status() == fa.FA_OK
        got = [torch.full_like(q, float("nan")) for _ in range(3)]
        torch.cuda.synchronize()
        # torch's count of allocated bytes must not move across the call.  Cyclic
        # garbage left by earlier tests (tracebacks that hold tensors) is
        # collected first, and the collector stays off while the count is
        # compared, so that it cannot free tensors in between.
        gc.collect()
        gc.disable()
        try:
            allocated = torch.cuda.memory_allocated()
            st = lib.fa_bwd_static_scratch(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                                           lse.data_ptr(), got[0].data_ptr(), got[1].data_ptr(), got[2].data_ptr(),
                                           B, H, N, d, ctypes.c_float(scale), int(causal),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
            assert st == fa.FA_OK, fa.fa_status_string(st)
            assert fa.fa_check_device_status() == fa.FA_OK
            assert torch.cuda.memory_allocated() == allocated
        finally:
            gc.enable()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            r = r.float()
            err = (g.float() - r).abs().max().item()
            assert err <= TOL * r.abs().max().item(), (call, name, err)


def test_static_scratch_rejects_shapes_beyond_its_size():
    # B=1, H=16, N=16384, d=128 needs a 128 MiB dQ accumulator, more than the
    # 72 MiB array: the call must be refused before any work is enqueued (the
    # pointers are never dereferenced).  The default bench workload fits.
    lib = fa.load_library()
    assert fa.fa_bwd_workspace_bytes(1, 16, 16384, 128) > fa.FA_STATIC_SCRATCH_BYTES
    p = ctypes.c_void_p(0x7F0000000000)
    st = lib.fa_bwd_static_scratch(p, p, p, p, p, p, p, p, p, 1, 16, 16384, 128, ctypes.c_float(0.1), 0, None)
    assert st == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_workspace_bytes(4, 16, 2048, 128) <= fa.FA_STATIC_SCRATCH_BYTES
