"""C-ABI checks that need no GPU: the library loads, exports every entry point
declared in include/fa.h, and rejects bad arguments before touching CUDA."""

import ctypes
import os
import re

import pytest

from exact_tiled_attention_08_gb300 import fa
from exact_tiled_attention_08_gb300.build import INCLUDE_DIR, build_library


@pytest.fixture(scope="module")
def lib():
    build_library()
    return fa.load_library()


def declared_functions():
    src = open(os.path.join(INCLUDE_DIR, "fa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fa_fwd", "fa_bwd", "fa_bwd_preprocess", "fa_bwd_workspace_bytes", "fa_check_device_status",
                     "fa_status_string", "fa_set_wait_limit_ns", "fa_debug_stall", "fa_set_timing_events",
                     "fa_set_exp2_split"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_exp2_split_validation(lib):
    assert lib.fa_set_exp2_split(3) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_set_exp2_split(-1) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_set_exp2_split(0) == fa.FA_OK


def test_status_strings(lib):
    for code, name in fa._STATUS_NAMES.items():
        assert fa.fa_status_string(code) == name
    assert fa.fa_status_string(99) == "FA_ERR_UNKNOWN"


# A fake but 16-byte-aligned address: validation must reject the call before any
# CUDA work is enqueued, so the pointer is never dereferenced.
P = 0x7F0000000000
BAD = P + 8
VP = ctypes.c_void_p


def fwd(lib, q=P, k=P, v=P, o=P, lse=P, B=1, H=1, N=128, d=128, scale=0.1, causal=0):
    return lib.fa_fwd(VP(q), VP(k), VP(v), VP(o), VP(lse), B, H, N, d, scale, causal, None)


def test_fwd_validation(lib):
    assert fwd(lib, q=0) == fa.FA_ERR_INVALID_ARG
    assert fwd(lib, lse=0) == fa.FA_ERR_INVALID_ARG
    assert fwd(lib, B=0) == fa.FA_ERR_INVALID_ARG
    assert fwd(lib, H=-1) == fa.FA_ERR_INVALID_ARG
    assert fwd(lib, N=0) == fa.FA_ERR_INVALID_ARG
    assert fwd(lib, d=96) == fa.FA_ERR_UNSUPPORTED
    assert fwd(lib, d=256) == fa.FA_ERR_UNSUPPORTED
    assert fwd(lib, scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert fwd(lib, scale=-1.0) == fa.FA_ERR_INVALID_ARG
    assert fwd(lib, scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert fwd(lib, scale=float("inf")) == fa.FA_ERR_INVALID_ARG
    assert fwd(lib, causal=2) == fa.FA_ERR_INVALID_ARG
    assert fwd(lib, B=1 << 16, H=1 << 15) == fa.FA_ERR_INVALID_ARG   # B*H = 2^31
    assert fwd(lib, B=1 << 15, H=1 << 15, N=1 << 20) == fa.FA_ERR_INVALID_ARG  # 128-row blocks x B*H >= 2^31
    assert fwd(lib, B=1 << 10, H=1 << 8, N=1 << 14, q=BAD) == fa.FA_ERR_MISALIGNED  # 2^39 elements: shape accepted
    assert fwd(lib, q=BAD) == fa.FA_ERR_MISALIGNED
    assert fwd(lib, o=BAD) == fa.FA_ERR_MISALIGNED
    assert fwd(lib, lse=P + 4) == fa.FA_ERR_MISALIGNED


def bwd(lib, ws_bytes=None, ws=P, dq=P, B=1, H=1, N=128, d=128, scale=0.1, causal=0, entry="fa_bwd"):
    if ws_bytes is None:
        ws_bytes = lib.fa_bwd_workspace_bytes(B, H, N, d)
    return getattr(lib, entry)(VP(P), VP(P), VP(P), VP(P), VP(P), VP(P), VP(dq), VP(P), VP(P), VP(ws), ws_bytes,
                               B, H, N, d, scale, causal, None)


@pytest.mark.parametrize("entry", ["fa_bwd", "fa_bwd_deterministic"])
def test_bwd_validation(lib, entry):
    assert bwd(lib, ws=0, entry=entry) == fa.FA_ERR_INVALID_ARG
    assert bwd(lib, dq=0, entry=entry) == fa.FA_ERR_INVALID_ARG
    assert bwd(lib, d=32, entry=entry) == fa.FA_ERR_UNSUPPORTED
    assert bwd(lib, scale=float("nan"), entry=entry) == fa.FA_ERR_INVALID_ARG
    assert bwd(lib, causal=-1, entry=entry) == fa.FA_ERR_INVALID_ARG
    need = lib.fa_bwd_workspace_bytes(1, 1, 128, 128)
    assert bwd(lib, ws_bytes=need - 1, entry=entry) == fa.FA_ERR_INVALID_ARG
    assert bwd(lib, dq=BAD, entry=entry) == fa.FA_ERR_MISALIGNED
    assert bwd(lib, ws=BAD, entry=entry) == fa.FA_ERR_MISALIGNED


def test_preprocess_validation(lib):
    f = lib.fa_bwd_preprocess
    assert f(VP(0), VP(P), VP(P), 1, 1, 8, 128, None) == fa.FA_ERR_INVALID_ARG
    assert f(VP(P), VP(P), VP(P), 1, 1, 8, 100, None) == fa.FA_ERR_UNSUPPORTED
    assert f(VP(P), VP(BAD), VP(P), 1, 1, 8, 128, None) == fa.FA_ERR_MISALIGNED


@pytest.mark.parametrize("B,H,N,d", [(1, 1, 128, 128), (2, 3, 1000, 64), (1, 8, 32768, 128), (16, 16, 1024, 64)])
def test_workspace_bytes(lib, B, H, N, d):
    # fp32 dQ accumulator, then delta and LSE*log2(e) padded to whole 128-row blocks
    rows = B * H * N
    npad = (N + 127) // 128 * 128
    dq = (rows * d * 4 + 255) // 256 * 256
    stat = (B * H * npad * 4 + 255) // 256 * 256
    assert lib.fa_bwd_workspace_bytes(B, H, N, d) == dq + 2 * stat


def test_workspace_bytes_rejects_bad_shapes(lib):
    assert lib.fa_bwd_workspace_bytes(0, 1, 1, 128) == 0
    assert lib.fa_bwd_workspace_bytes(1, 1, 1, 80) == 0


def test_binding_checks_tensors_before_calling(lib):
    import torch

    q = torch.zeros((1, 1, 8, 128), dtype=torch.float32)
    with pytest.raises(TypeError):
        fa.fa_fwd(q, q, q, q, torch.zeros((1, 1, 8)), 0.1, False, stream=0)
    qb = torch.zeros((1, 1, 8, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fa_fwd(qb, qb, qb, qb, torch.zeros((1, 1, 7)), 0.1, False, stream=0)


def test_fwd_fp8_validation(lib):
    f = lib.fa_fwd_fp8
    need = lib.fa_fwd_fp8_workspace_bytes(1, 1, 128, 128)
    assert need > 0 and lib.fa_fwd_fp8_workspace_bytes(1, 1, 128, 64) == 0

    def call(signs=P, ws=P, ws_bytes=need, d=128, scale=0.1, causal=0):
        return f(VP(P), VP(P), VP(P), VP(signs), VP(P), VP(P), VP(ws), ws_bytes, 1, 1, 128, d, scale, causal, None)

    assert call(signs=0) == fa.FA_ERR_INVALID_ARG
    assert call(ws=0) == fa.FA_ERR_INVALID_ARG
    assert call(ws_bytes=need - 1) == fa.FA_ERR_INVALID_ARG
    assert call(d=64) == fa.FA_ERR_UNSUPPORTED
    assert call(scale=-1.0) == fa.FA_ERR_INVALID_ARG
    assert call(ws=BAD) == fa.FA_ERR_MISALIGNED


@pytest.mark.parametrize("B,H,N", [(1, 1, 1), (1, 2, 129), (4, 16, 2048), (1, 8, 32768)])
def test_fwd_fp8_workspace_bytes_follow_the_documented_layout(lib, B, H, N):
    # Q R, K R [B][H][N][128] E4M3; V^T [B][H][nkb][128][128] E4M3; query and key
    # block scales [B][H][nkb] fp32; channel maxima and scales [B][H][128] fp32;
    # each part on a 256-byte boundary
    bh, nkb = B * H, (N + 127) // 128

    def up(x):
        return (x + 255) // 256 * 256

    want = 2 * up(bh * N * 128) + up(bh * nkb * 128 * 128) + 2 * up(bh * nkb * 4) + 2 * up(bh * 128 * 4)
    assert lib.fa_fwd_fp8_workspace_bytes(B, H, N, 128) == want


def test_fwd_fp8_rejects_more_than_65535_heads(lib):
    # the V quantisation's grid has one y index per (batch, head)
    B, H, N = 256, 257, 128
    need = lib.fa_fwd_fp8_workspace_bytes(B, H, N, 128)
    assert need > 0
    assert lib.fa_fwd_fp8(VP(P), VP(P), VP(P), VP(P), VP(P), VP(P), VP(P), need, B, H, N, 128, 0.1, 0,
                          None) == fa.FA_ERR_UNSUPPORTED


def test_workspace_bytes_past_2_31_elements(lib):
    # B*H*N*d above 2^31 is accepted; sizes are computed in 64 bits
    B, H, N, d = 1, 8193, 2048, 128
    rows = B * H * N
    assert rows * d > 1 << 31
    assert lib.fa_bwd_workspace_bytes(B, H, N, d) == (rows * d * 4 + 255) // 256 * 256 + 2 * ((rows * 4 + 255) // 256 * 256)

