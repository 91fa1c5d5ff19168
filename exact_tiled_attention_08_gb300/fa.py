"""Thin Python binding of the C ABI in ``include/fa.h`` (ctypes).

Every function here has the name of the C entry point it wraps and does
argument marshalling only: it checks dtypes, shapes, contiguity and devices of
the torch tensors it is given, passes their device pointers and sizes to the
library, and raises ``FaError`` on a non-OK status.  All arithmetic runs in the
library's CUDA kernels; there is no other implementation behind these names.
If the compiled library is missing, loading fails loudly.
"""

from __future__ import annotations

import contextlib
import ctypes
import os

import torch

from .build import LIB_PATH

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_MISALIGNED = 2
FA_ERR_UNSUPPORTED = 3
FA_ERR_CUDA = 4
FA_ERR_TIMEOUT = 5

_STATUS_NAMES = {
    FA_OK: "FA_OK",
    FA_ERR_INVALID_ARG: "FA_ERR_INVALID_ARG",
    FA_ERR_MISALIGNED: "FA_ERR_MISALIGNED",
    FA_ERR_UNSUPPORTED: "FA_ERR_UNSUPPORTED",
    FA_ERR_CUDA: "FA_ERR_CUDA",
    FA_ERR_TIMEOUT: "FA_ERR_TIMEOUT",
}


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_STATUS_NAMES.get(status, status)}")


_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libfa.so (built by ``build.build_library``); raises if it is absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libfa.so not found at {p}: run __graft_entry__.build() (no fallback exists)")
    lib = ctypes.CDLL(p)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.fa_fwd.restype = i
    lib.fa_fwd_fp8_workspace_bytes.argtypes = [i, i, i, i]
    lib.fa_fwd_fp8_workspace_bytes.restype = sz
    lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, f, i, vp]
    lib.fa_fwd_fp8.restype = i
    lib.fa_bwd_preprocess.argtypes = [vp, vp, vp, i, i, i, i, vp]
    lib.fa_bwd_preprocess.restype = i
    lib.fa_bwd_workspace_bytes.argtypes = [i, i, i, i]
    lib.fa_bwd_workspace_bytes.restype = sz
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, f, i, vp]
    lib.fa_bwd.restype = i
    lib.fa_bwd_deterministic.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, f, i, vp]
    lib.fa_bwd_deterministic.restype = i
    lib.fa_bwd_static_scratch.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.fa_bwd_static_scratch.restype = i
    lib.fa_check_device_status.argtypes = [vp]
    lib.fa_check_device_status.restype = i
    lib.fa_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.fa_set_wait_limit_ns.restype = None
    lib.fa_debug_stall.argtypes = [i]
    lib.fa_debug_stall.restype = None
    lib.fa_set_bwd_pair_mma.argtypes = [i]
    lib.fa_set_bwd_pair_mma.restype = None
    lib.fa_set_exp2_split.argtypes = [i]
    lib.fa_set_exp2_split.restype = i
    lib.fa_set_timing_events.argtypes = [vp, vp, vp, vp]
    lib.fa_set_timing_events.restype = None
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def _stream_handle(stream, device=None) -> int:
    """The raw handle of ``stream``: None is the current stream of ``device``
    (or of the current device); a torch stream must live on ``device``."""
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        if device is not None and stream.device != device:
            raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
        return stream.cuda_stream
    return int(stream)


def _on_device(device: torch.device):
    """The library launches on the current device, so each call makes the
    tensors' device current for its duration."""
    return torch.cuda.device(device) if device.type == "cuda" else contextlib.nullcontext()


def _shape4(t: torch.Tensor, name: str):
    if t.dim() != 4:
        raise ValueError(f"{name} must be [B, H, N, d], got {tuple(t.shape)}")
    return tuple(t.shape)


def _check(t: torch.Tensor, name: str, dtype, shape, device):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor, got one on {t.device}")


def _raise(status: int, where: str):
    if status != FA_OK:
        raise FaError(status, where)


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


def fa_set_wait_limit_ns(limit_ns: int) -> None:
    load_library().fa_set_wait_limit_ns(int(limit_ns))


def fa_debug_stall(enable: bool) -> None:
    """Test hook: kernels launched while enabled stall on a barrier nothing signals."""
    load_library().fa_debug_stall(int(bool(enable)))


def fa_set_bwd_pair_mma(enable: bool) -> None:
    """fa_bwd_deterministic at d = 128: dK, dV products as 2-CTA (256-row) MMAs on CTA pairs."""
    load_library().fa_set_bwd_pair_mma(int(bool(enable)))


def fa_set_exp2_split(soft_quarters: int) -> None:
    """0 (default): every forward exponential on the special-function unit;
    1 or 2: that many of every four pairs by the cubic 2^n p(f) on the FMA pipe."""
    _raise(load_library().fa_set_exp2_split(int(soft_quarters)), "fa_set_exp2_split")


def _event_handle(ev) -> int:
    if ev is None:
        return 0
    if isinstance(ev, torch.cuda.Event):
        if ev.cuda_event == 0:
            raise ValueError("record a torch.cuda.Event once before passing it (it is created lazily)")
        return ev.cuda_event
    return int(ev)


def fa_set_timing_events(fwd_start=None, fwd_stop=None, bwd_start=None, bwd_stop=None) -> None:
    """Events recorded around the forward kernel and the main backward kernel (profiling)."""
    load_library().fa_set_timing_events(_event_handle(fwd_start), _event_handle(fwd_stop),
                                        _event_handle(bwd_start), _event_handle(bwd_stop))


def fa_check_device_status(stream=None) -> int:
    """Synchronize the stream; return (and clear) the status word of the
    stream's device (of the current device for None or a raw handle)."""
    dev = stream.device if isinstance(stream, torch.cuda.Stream) else None
    with (torch.cuda.device(dev) if dev is not None else contextlib.nullcontext()):
        return int(load_library().fa_check_device_status(_stream_handle(stream)))


def fa_fwd(q, k, v, o, lse, scale: float, causal: bool, stream=None) -> None:
    """O and LSE of softmax(scale Q K^T) V; tensors [B,H,N,d] bf16 and [B,H,N] fp32."""
    B, H, N, d = _shape4(q, "q")
    dev = q.device
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _check(t, name, torch.bfloat16, (B, H, N, d), dev)
    _check(lse, "lse", torch.float32, (B, H, N), dev)
    with _on_device(dev):
        st = load_library().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                   B, H, N, d, float(scale), int(bool(causal)), _stream_handle(stream, dev))
    _raise(st, "fa_fwd")


def fa_fwd_fp8_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().fa_fwd_fp8_workspace_bytes(B, H, N, d))


def fa_fwd_fp8(q, k, v, signs, o, lse, workspace, scale: float, causal: bool, stream=None) -> None:
    """FP8 forward: Q, K rotated by diag(signs) H / sqrt(d) and quantised per
    128-row block, V per channel, E4M3 products; signs is an int8 device
    tensor of +1 / -1 [d]; workspace a uint8 device tensor."""
    B, H, N, d = _shape4(q, "q")
    dev = q.device
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _check(t, name, torch.bfloat16, (B, H, N, d), dev)
    _check(lse, "lse", torch.float32, (B, H, N), dev)
    _check(signs, "signs", torch.int8, (d,), dev)
    if workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on the inputs' device")
    ws_bytes = workspace.numel() * workspace.element_size()
    with _on_device(dev):
        st = load_library().fa_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), signs.data_ptr(), o.data_ptr(),
                                       lse.data_ptr(), workspace.data_ptr(), ws_bytes, B, H, N, d, float(scale),
                                       int(bool(causal)), _stream_handle(stream, dev))
    _raise(st, "fa_fwd_fp8")


def fa_bwd_preprocess(o, dout, delta, stream=None) -> None:
    """delta = rowsum(dO * O) in fp32, [B,H,N]."""
    B, H, N, d = _shape4(o, "o")
    dev = o.device
    _check(o, "o", torch.bfloat16, (B, H, N, d), dev)
    _check(dout, "dout", torch.bfloat16, (B, H, N, d), dev)
    _check(delta, "delta", torch.float32, (B, H, N), dev)
    with _on_device(dev):
        st = load_library().fa_bwd_preprocess(o.data_ptr(), dout.data_ptr(), delta.data_ptr(), B, H, N, d,
                                              _stream_handle(stream, dev))
    _raise(st, "fa_bwd_preprocess")


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().fa_bwd_workspace_bytes(B, H, N, d))


def _bwd_call(entry: str, q, k, v, o, dout, lse, dq, dk, dv, workspace, scale: float, causal: bool, stream):
    B, H, N, d = _shape4(q, "q")
    dev = q.device
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check(t, name, torch.bfloat16, (B, H, N, d), dev)
    _check(lse, "lse", torch.float32, (B, H, N), dev)
    if workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on the inputs' device")
    ws_bytes = workspace.numel() * workspace.element_size()
    with _on_device(dev):
        st = getattr(load_library(), entry)(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                            dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                            dv.data_ptr(), workspace.data_ptr(), ws_bytes, B, H, N, d, float(scale),
                                            int(bool(causal)), _stream_handle(stream, dev))
    _raise(st, entry)


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, scale: float, causal: bool, stream=None) -> None:
    """dQ, dK, dV of attention by recomputation; workspace is a uint8 device tensor."""
    _bwd_call("fa_bwd", q, k, v, o, dout, lse, dq, dk, dv, workspace, scale, causal, stream)


def fa_bwd_deterministic(q, k, v, o, dout, lse, dq, dk, dv, workspace, scale: float, causal: bool,
                         stream=None) -> None:
    """fa_bwd with dQ summed by a separate query-major pass: bitwise repeatable."""
    _bwd_call("fa_bwd_deterministic", q, k, v, o, dout, lse, dq, dk, dv, workspace, scale, causal, stream)


FA_STATIC_SCRATCH_BYTES = 72 * 1024 * 1024


def fa_bwd_static_scratch(q, k, v, o, dout, lse, dq, dk, dv, scale: float, causal: bool, stream=None) -> None:
    """fa_bwd without a workspace argument, for callers that cannot allocate device
    memory at call time: the scratch is a fixed array inside the library (see
    include/fa.h for the size limit, the first-call set-up and the rule that
    calls overlapping on the GPU race)."""
    B, H, N, d = _shape4(q, "q")
    dev = q.device
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check(t, name, torch.bfloat16, (B, H, N, d), dev)
    _check(lse, "lse", torch.float32, (B, H, N), dev)
    with _on_device(dev):
        st = load_library().fa_bwd_static_scratch(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                                  dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                                  dv.data_ptr(), B, H, N, d, float(scale), int(bool(causal)),
                                                  _stream_handle(stream, dev))
    _raise(st, "fa_bwd_static_scratch")


# ---------------------------------------------------------------------------
# conveniences that allocate the outputs with torch and call the entry points.
# With check_status (the default) they wait for the work and raise FaError if
# a kernel reported a timeout, so what they return is known to be valid; pass
# check_status=False to keep the call asynchronous and check later with
# fa_check_device_status.
# ---------------------------------------------------------------------------
def _checked(stream, device, where: str):
    with _on_device(device):
        st = int(load_library().fa_check_device_status(_stream_handle(stream, device)))
    _raise(st, where)


def attention_forward(q, k, v, scale: float, causal: bool = False, stream=None, check_status: bool = True):
    B, H, N, d = _shape4(q, "q")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, scale, causal, stream)
    if check_status:
        _checked(stream, q.device, "attention_forward")
    return o, lse


def attention_forward_fp8(q, k, v, signs, scale: float, causal: bool = False, workspace=None, stream=None,
                          check_status: bool = True):
    B, H, N, d = _shape4(q, "q")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(fa_fwd_fp8_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=q.device)
    fa_fwd_fp8(q, k, v, signs, o, lse, workspace, scale, causal, stream)
    if check_status:
        _checked(stream, q.device, "attention_forward_fp8")
    return o, lse


def attention_backward(q, k, v, o, dout, lse, scale: float, causal: bool = False, workspace=None, stream=None,
                       deterministic: bool = False, check_status: bool = True):
    B, H, N, d = _shape4(q, "q")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=q.device)
    (fa_bwd_deterministic if deterministic else fa_bwd)(q, k, v, o, dout, lse, dq, dk, dv, workspace, scale, causal,
                                                        stream)
    if check_status:
        _checked(stream, q.device, "attention_backward")
    return dq, dk, dv
