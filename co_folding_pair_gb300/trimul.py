"""Python binding of the TriMul C ABI (include/trimul.h): argument marshalling only.

Every step of the forward runs in the CUDA library; PyTorch supplies device
memory and streams.  The functions keep the C names; ``TriMul`` wraps them in
the construct / prepare / call / free life cycle of the fold-cp-ops README
("Use" section).  There is no fallback: if the library cannot be built or
loaded, or the device is not sm_103, the calls raise.
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib

OUTGOING = 0
INCOMING = 1
FLAG_CHECK = 1
FLAG_INJECT_STALL = 2
FLAG_DEFER_OUTPUT = 4
FLAG_FP8 = 8  # trimul_forward only, outgoing only: e4m3 triangle contraction (less accurate)

STATUS_NAMES = {
    0: "TRIMUL_OK",
    1: "TRIMUL_ERR_INVALID_ARG",
    2: "TRIMUL_ERR_SHAPE",
    3: "TRIMUL_ERR_UNSUPPORTED_ARCH",
    4: "TRIMUL_ERR_OOM",
    5: "TRIMUL_ERR_CUDA",
    6: "TRIMUL_ERR_TIMEOUT",
}

PARAM_DTYPES = {
    "W_a": torch.bfloat16, "W_ga": torch.bfloat16, "W_b": torch.bfloat16, "W_gb": torch.bfloat16,
    "W_o": torch.bfloat16, "W_g": torch.bfloat16,
    "ln_in_gamma": torch.float32, "ln_in_beta": torch.float32,
    "ln_out_gamma": torch.float32, "ln_out_beta": torch.float32,
}


class TrimulError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class Handle:
    """An opaque trimul_handle plus the layer sizes it was created with."""

    def __init__(self, ptr: ctypes.c_void_p, D: int, C: int, device: int):
        self.ptr = ptr
        self.D = D
        self.C = C
        self.device = device


def _check(status: int):
    if status != 0:
        raise TrimulError(status, trimul_last_error())


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _direction(direction) -> int:
    if direction in ("outgoing", OUTGOING):
        return OUTGOING
    if direction in ("incoming", INCOMING):
        return INCOMING
    raise ValueError(f"direction must be 'outgoing' or 'incoming', got {direction!r}")


def _need(t, dtype, name, device=None):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and (t.device.type != "cuda" or t.device.index != device):
        raise ValueError(f"{name} must be on cuda:{device}, got {t.device}")


def trimul_last_error() -> str:
    msg = _lib.load().trimul_last_error()
    return msg.decode() if msg else ""


def trimul_kernels_per_forward(h: Handle, B: int, N: int) -> int:
    """Kernel launches one trimul_forward enqueues for a B x N input."""
    n = int(_lib.load().trimul_kernels_per_forward(h.ptr, B, N))
    if n < 0:
        raise TrimulError(1, trimul_last_error())
    return n


def trimul_kernels_per_forward_host(h: Handle, B: int, N: int) -> int:
    """Kernels one trimul_forward_host call launches for a B x N input."""
    n = int(_lib.load().trimul_kernels_per_forward_host(h.ptr, B, N))
    if n < 0:
        raise TrimulError(1, trimul_last_error())
    return n


def trimul_create(params: dict, eps: float = 1e-5, device=None) -> Handle:
    """Create a handle from W_a, W_ga, W_b, W_gb [C, D], W_o [D, C], W_g [D, D] (bf16)
    and the LayerNorm affine parameters (float32)."""
    lib = _lib.load()
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else torch.device(device).index or 0)
    on_dev = {}
    for k, dt in PARAM_DTYPES.items():
        on_dev[k] = params[k].to(device=dev, dtype=dt).contiguous()
    C, D = on_dev["W_a"].shape
    p = _lib.TrimulParams()
    p.D, p.C, p.eps = int(D), int(C), float(eps)
    for k in PARAM_DTYPES:
        setattr(p, k, on_dev[k].data_ptr())
    out = ctypes.c_void_p()
    with torch.cuda.device(dev):
        torch.cuda.current_stream(dev).synchronize()
        _check(lib.trimul_create(ctypes.byref(out), ctypes.byref(p), dev.index))
    return Handle(out, int(D), int(C), dev.index)


def trimul_prepare(h: Handle, B: int, N: int, masked: bool = True):
    _check(_lib.load().trimul_prepare(h.ptr, B, N, int(bool(masked))))


def trimul_forward(h: Handle, z, mask, direction, out=None, stream=None, flags: int = 0):
    """out[B, N, N, D] (bf16) = TriMul(z[B, N, N, D] bf16, mask[B, N, N] bf16 or None)."""
    _need(z, torch.bfloat16, "z", h.device)
    if mask is not None:
        _need(mask, torch.bfloat16, "mask", h.device)
    B, N = z.shape[0], z.shape[1]
    if out is None:
        out = torch.empty_like(z)
    _need(out, torch.bfloat16, "out", h.device)
    _check(_lib.load().trimul_forward(h.ptr, _vp(z), _vp(mask), B, N, _direction(direction), _vp(out),
                                      _stream(stream, h.device), flags))
    return out


def trimul_forward_noalloc(h: Handle, z, mask, direction, out, stream=None, flags: int = 0):
    """trimul_forward without any device allocation: a, b and x live in the
    library's fixed scratch array (see include/trimul.h).  ``out`` must be
    given, so this call allocates nothing, not even through torch."""
    _need(z, torch.bfloat16, "z", h.device)
    if mask is not None:
        _need(mask, torch.bfloat16, "mask", h.device)
    _need(out, torch.bfloat16, "out", h.device)
    B, N = z.shape[0], z.shape[1]
    _check(_lib.load().trimul_forward_noalloc(h.ptr, _vp(z), _vp(mask), B, N, _direction(direction), _vp(out),
                                              _stream(stream, h.device), flags))
    return out


def trimul_noalloc_scratch_bytes() -> int:
    return int(_lib.load().trimul_noalloc_scratch_bytes())


def trimul_forward_host(h: Handle, z_host, mask_host, direction, out_host=None, stream=None, flags: int = 0):
    """Same as trimul_forward on CPU tensors (pinned memory for asynchronous copies).
    Returns after enqueueing; synchronise the stream before reading out_host."""
    if z_host.device.type != "cpu":
        raise ValueError("z_host must be a CPU tensor")
    _need(z_host, torch.bfloat16, "z_host")
    if mask_host is not None:
        _need(mask_host, torch.bfloat16, "mask_host")
    if out_host is None:
        out_host = torch.empty_like(z_host, pin_memory=z_host.is_pinned())
    _need(out_host, torch.bfloat16, "out_host")
    B, N = z_host.shape[0], z_host.shape[1]
    _check(_lib.load().trimul_forward_host(h.ptr, _vp(z_host), _vp(mask_host), B, N, _direction(direction),
                                           _vp(out_host), _stream(stream, h.device), flags))
    return out_host


def trimul_host_join(h: Handle, stream=None):
    """Make `stream` wait for every output copy of earlier host-buffer calls
    (needed before reading out_host of calls made with FLAG_DEFER_OUTPUT)."""
    _check(_lib.load().trimul_host_join(h.ptr, _stream(stream, h.device)))


def trimul_inproj(h: Handle, z, mask, a_out=None, b_out=None, stream=None, flags: int = 0):
    """Stage 1: a, b as fp16 [B, C, N, N] channel-major planes."""
    _need(z, torch.bfloat16, "z", h.device)
    B, N = z.shape[0], z.shape[1]
    shape = (B, h.C, N, N)
    a_out = torch.empty(shape, dtype=torch.float16, device=z.device) if a_out is None else a_out
    b_out = torch.empty(shape, dtype=torch.float16, device=z.device) if b_out is None else b_out
    _need(a_out, torch.float16, "a_out", h.device)
    _need(b_out, torch.float16, "b_out", h.device)
    if mask is not None:
        _need(mask, torch.bfloat16, "mask", h.device)
    _check(_lib.load().trimul_inproj(h.ptr, _vp(z), _vp(mask), B, N, _vp(a_out), _vp(b_out),
                                     _stream(stream, h.device), flags))
    return a_out, b_out


def trimul_x_scale_log2(h: Handle, N: int) -> int:
    """s such that stage 2 stores x * 2^-s (fp16) for token count N."""
    s = int(_lib.load().trimul_x_scale_log2(h.ptr, N))
    if s < 0:
        raise TrimulError(1, trimul_last_error())
    return s


def trimul_triangle(h: Handle, a, b, direction, x_out=None, stream=None, flags: int = 0):
    """Stage 2: x * 2^-s (fp16 [B, C, N, N], s = trimul_x_scale_log2) from fp16 a, b planes."""
    _need(a, torch.float16, "a", h.device)
    _need(b, torch.float16, "b", h.device)
    B, N = a.shape[0], a.shape[2]
    x_out = torch.empty(a.shape, dtype=torch.float16, device=a.device) if x_out is None else x_out
    _need(x_out, torch.float16, "x_out", h.device)
    _check(_lib.load().trimul_triangle(h.ptr, _vp(a), _vp(b), B, N, _direction(direction), _vp(x_out),
                                       _stream(stream, h.device), flags))
    return x_out


def trimul_outproj(h: Handle, x, z, out=None, stream=None, flags: int = 0):
    """Stage 3: out (bf16 [B, N, N, D]) from x * 2^-s (fp16 [B, C, N, N]) and z."""
    _need(x, torch.float16, "x", h.device)
    _need(z, torch.bfloat16, "z", h.device)
    B, N = z.shape[0], z.shape[1]
    out = torch.empty_like(z) if out is None else out
    _need(out, torch.bfloat16, "out", h.device)
    _check(_lib.load().trimul_outproj(h.ptr, _vp(x), _vp(z), B, N, _vp(out), _stream(stream, h.device), flags))
    return out


# Parameter names of the gradients trimul_backward returns, with their C fields.
GRAD_NAMES = {"W_a": "dW_a", "W_ga": "dW_ga", "W_b": "dW_b", "W_gb": "dW_gb", "W_o": "dW_o", "W_g": "dW_g",
              "ln_in_gamma": "d_ln_in_gamma", "ln_in_beta": "d_ln_in_beta",
              "ln_out_gamma": "d_ln_out_gamma", "ln_out_beta": "d_ln_out_beta"}


def trimul_backward(h: Handle, z, mask, dout, direction, dz=None, grads=None, stream=None, flags: int = 0):
    """Gradients of the layer for dout = dL/d out: returns (dz, grads) with dz
    bf16 [B, N, N, D] and grads a dict of float32 tensors keyed by parameter
    name (W_a ... ln_out_beta), in the parameters' own shapes."""
    _need(z, torch.bfloat16, "z", h.device)
    _need(dout, torch.bfloat16, "dout", h.device)
    if mask is not None:
        _need(mask, torch.bfloat16, "mask", h.device)
    B, N = z.shape[0], z.shape[1]
    D, C = h.D, h.C
    shapes = {"W_a": (C, D), "W_ga": (C, D), "W_b": (C, D), "W_gb": (C, D), "W_o": (D, C), "W_g": (D, D),
              "ln_in_gamma": (D,), "ln_in_beta": (D,), "ln_out_gamma": (C,), "ln_out_beta": (C,)}
    if dz is None:
        dz = torch.empty_like(z)
    _need(dz, torch.bfloat16, "dz", h.device)
    if grads is None:
        grads = {k: torch.empty(shp, dtype=torch.float32, device=z.device) for k, shp in shapes.items()}
    g = _lib.TrimulGrads()
    for k, field in GRAD_NAMES.items():
        _need(grads[k], torch.float32, k, h.device)
        setattr(g, field, grads[k].data_ptr())
    _check(_lib.load().trimul_backward(h.ptr, _vp(z), _vp(mask), _vp(dout), B, N, _direction(direction), _vp(dz),
                                       ctypes.byref(g), _stream(stream, h.device), flags))
    return dz, grads


def trimul_backward_workspace_bytes(h: Handle, B: int, N: int) -> int:
    return int(_lib.load().trimul_backward_workspace_bytes(h.ptr, B, N))


def trimul_kernels_per_backward(h: Handle, B: int, N: int) -> int:
    n = int(_lib.load().trimul_kernels_per_backward(h.ptr, B, N))
    if n < 0:
        raise TrimulError(1, trimul_last_error())
    return n


def trimul_set_stage_events(h: Handle, events):
    """events: four torch.cuda.Event(enable_timing=True) (already recorded once,
    so that they exist), or None to switch per-stage recording off."""
    if events is None:
        _check(_lib.load().trimul_set_stage_events(h.ptr, None))
        return
    arr = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(_lib.load().trimul_set_stage_events(h.ptr, arr))


def trimul_destroy(h: Handle):
    if h is not None and h.ptr:
        _check(_lib.load().trimul_destroy(h.ptr))
        h.ptr = ctypes.c_void_p()


class TriMul:
    """construct -> prepare (optional) -> __call__ -> free, on one GPU."""

    def __init__(self, params: dict, direction="outgoing", eps: float = 1e-5, device=None):
        self.direction = _direction(direction)
        self.handle = trimul_create(params, eps=eps, device=device)

    def prepare(self, n_token: int, batch: int = 1, masked: bool = True):
        trimul_prepare(self.handle, batch, n_token, masked)

    def __call__(self, z, mask=None, out=None, stream=None, flags: int = 0):
        return trimul_forward(self.handle, z, mask, self.direction, out=out, stream=stream, flags=flags)

    def free(self):
        trimul_destroy(self.handle)

    def __del__(self):
        try:
            if getattr(self, "handle", None) is not None and self.handle.ptr:
                trimul_destroy(self.handle)
        except Exception:
            pass
