"""The boundary's limits on a GPU: pointers the device cannot use are refused
before anything runs, and shapes whose element count passes 2^31 (the
kernels' 64-bit addressing) give the same results as the oracle."""

import ctypes
import math

import numpy as np
import pytest
import torch

from exact_tiled_attention_08_gb300 import fa
from exact_tiled_attention_08_gb300.workloads import make_inputs, to_f32_numpy
from oracle import attention_bwd_ref, attention_fwd_ref

pytestmark = pytest.mark.gpu

VP = ctypes.c_void_p


@pytest.fixture(scope="module")
def lib():
    from exact_tiled_attention_08_gb300.build import build_library

    build_library()
    return fa.load_library()


def test_host_and_unmapped_pointers_are_refused(lib):
    B, H, N, d = 1, 2, 256, 128
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, H, N), dtype=torch.float32, device="cuda")
    host = torch.zeros((B, H, N, d), dtype=torch.bfloat16)            # pageable host memory
    pinned = torch.zeros((B, H, N, d), dtype=torch.bfloat16).pin_memory()
    fake = 0x7F0000000000                                             # aligned, covered by nothing
    dp, lp = q.data_ptr(), lse.data_ptr()
    torch.cuda.synchronize()
    for bad in (host.data_ptr(), pinned.data_ptr(), fake):
        assert lib.fa_fwd(VP(bad), VP(dp), VP(dp), VP(dp), VP(lp), B, H, N, d, 0.1, 0, None) == fa.FA_ERR_INVALID_ARG
        assert lib.fa_fwd(VP(dp), VP(dp), VP(dp), VP(bad), VP(lp), B, H, N, d, 0.1, 0, None) == fa.FA_ERR_INVALID_ARG
        assert lib.fa_bwd_preprocess(VP(dp), VP(bad), VP(lp), B, H, N, d, None) == fa.FA_ERR_INVALID_ARG
    # nothing was enqueued and the context is healthy: a valid call still works
    assert lib.fa_fwd(VP(dp), VP(dp), VP(dp), VP(dp), VP(lp), B, H, N, d, 0.1, 0, None) == fa.FA_OK
    assert fa.fa_check_device_status() == fa.FA_OK
    assert torch.isfinite(lse).all()


def test_binding_refuses_tensors_on_mixed_devices():
    q = torch.zeros((1, 1, 128, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 1, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q, q, torch.zeros((1, 1, 128, 128), dtype=torch.bfloat16), lse, 0.1, False)


def test_more_than_2_31_elements_match_the_oracle(lib):
    """B*H*N*d = 8193 * 2048 * 128 > 2^31: head 8192 starts exactly 2^31
    elements in.  The heads cycle through a pool of 7 seeded heads, so that the
    oracle needs only the pool; a 32-bit wrap of any offset would read another
    pool head's data (head 8192 -> head 0) and fail the comparison."""
    B, H, N, d = 1, 8193, 2048, 128
    assert (8192 * N * d) == 1 << 31
    free, _ = torch.cuda.mem_get_info()
    need = 8 * B * H * N * d * 2 + fa.fa_bwd_workspace_bytes(B, H, N, d) + (1 << 30)
    if free < need:
        pytest.skip(f"needs {need / 2**30:.1f} GiB of device memory, {free / 2**30:.1f} free")
    pool_n = 7
    pool = make_inputs(1, pool_n, N, d, seed=2031)
    scale = 1.0 / math.sqrt(d)
    big = {}
    for name in ("q", "k", "v", "do"):
        t = torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")
        src = pool[name][0].cuda()
        flat = t.view(H, N, d)
        for r in range(pool_n):
            flat[r::pool_n] = src[r]
        big[name] = t
    q, k, v, do = big["q"], big["k"], big["v"], big["do"]
    o, lse = fa.attention_forward(q, k, v, scale, False)
    dq, dk, dv = fa.attention_backward(q, k, v, o, do, lse, scale, False)
    for h in (0, 4096, 8191, 8192):
        r = h % pool_n
        qn, kn, vn, don = (to_f32_numpy(pool[x][0, r]) for x in ("q", "k", "v", "do"))
        o_ref, l_ref = attention_fwd_ref(qn, kn, vn, scale, False)
        dq_ref, dk_ref, dv_ref = attention_bwd_ref(qn, kn, vn, don, scale, False)
        assert np.abs(to_f32_numpy(o[0, h]) - o_ref).max() <= 1e-2, h
        assert np.abs(lse[0, h].cpu().numpy() - l_ref).max() <= 1e-3, h
        for name, g, ref in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
            err = np.abs(to_f32_numpy(g[0, h]) - ref).max()
            assert err <= 2e-2 * np.abs(ref).max(), (h, name, err)
    # every head is one of the pool's: outputs of equal heads are equal, so a
    # wrong offset anywhere would show as a mismatch against head h % 7
    for h in (8192, 8186):
        assert torch.equal(o[0, h], o[0, h % pool_n]), h
        assert torch.equal(dk[0, h], dk[0, h % pool_n]), h
