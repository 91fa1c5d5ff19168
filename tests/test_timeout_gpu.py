"""The bounded waits: with the debug stall on, each kernel's MMA thread waits
on a barrier that nothing signals; after the (short) wait limit the kernel
reports FA_ERR_TIMEOUT through the status word, drains the copies it started
and returns; the checking conveniences raise it as FaError.  The context
stays usable and the next call, with the stall off and the default limit, is
correct.  Nothing here traps or hangs."""

import math

import numpy as np
import pytest
import torch

from exact_tiled_attention_08_gb300 import fa
from exact_tiled_attention_08_gb300.workloads import make_inputs, to_f32_numpy
from oracle import attention_fwd_ref

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def restore_limit():
    from exact_tiled_attention_08_gb300.build import build_library

    build_library()
    fa.load_library()
    yield
    fa.fa_debug_stall(False)
    fa.fa_set_wait_limit_ns(0)


def test_forward_wait_timeout_is_reported_and_recoverable():
    inp = make_inputs(1, 2, 512, 128, seed=31)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(128)
    assert fa.fa_check_device_status() == fa.FA_OK
    fa.fa_set_wait_limit_ns(1_000_000)  # 1 ms
    fa.fa_debug_stall(True)
    # asynchronous form: the call returns FA_OK, the status word holds the timeout
    fa.attention_forward(q, k, v, scale, False, check_status=False)
    assert fa.fa_check_device_status() == fa.FA_ERR_TIMEOUT
    assert fa.fa_check_device_status() == fa.FA_OK  # cleared by the read
    # checked form (the conveniences' default): the timeout is raised
    with pytest.raises(fa.FaError) as err:
        fa.attention_forward(q, k, v, scale, False)
    assert err.value.status == fa.FA_ERR_TIMEOUT
    assert fa.fa_check_device_status() == fa.FA_OK
    fa.fa_debug_stall(False)
    fa.fa_set_wait_limit_ns(0)
    o, lse = fa.attention_forward(q, k, v, scale, False)
    assert fa.fa_check_device_status() == fa.FA_OK
    o_ref, l_ref = attention_fwd_ref(*(to_f32_numpy(inp[x][0, 1]) for x in ("q", "k", "v")), scale, False)
    assert np.abs(to_f32_numpy(o[0, 1]) - o_ref).max() <= 1e-2
    assert np.abs(lse[0, 1].cpu().numpy() - l_ref).max() <= 1e-3


def test_backward_wait_timeout_is_reported_and_recoverable():
    inp = make_inputs(1, 2, 512, 64, seed=32)
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    scale = 0.125
    o, lse = fa.attention_forward(q, k, v, scale, True)
    assert fa.fa_check_device_status() == fa.FA_OK
    fa.fa_set_wait_limit_ns(1_000_000)
    fa.fa_debug_stall(True)
    with pytest.raises(fa.FaError) as err:
        fa.attention_backward(q, k, v, o, do, lse, scale, True)
    assert err.value.status == fa.FA_ERR_TIMEOUT
    assert fa.fa_check_device_status() == fa.FA_OK
    fa.fa_debug_stall(False)
    fa.fa_set_wait_limit_ns(0)
    dq, dk, dv = fa.attention_backward(q, k, v, o, do, lse, scale, True)
    assert fa.fa_check_device_status() == fa.FA_OK
    assert torch.isfinite(dq.float()).all() and torch.isfinite(dk.float()).all()
