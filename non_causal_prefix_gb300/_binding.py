"""ctypes binding of the C ABI declared in include/ncp_attn.h.

Argument marshalling only: every step of the attention runs in the CUDA
kernels of ``_lib/libncp_attn.so``.  There is no fallback; if the library is
missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

ATTN_OK = 0
ATTN_ERR_NULL = -1
ATTN_ERR_SHAPE = -2
ATTN_ERR_HEADDIM = -3
ATTN_ERR_ALIGN = -4
ATTN_ERR_ALIAS = -5
ATTN_ERR_CUDA = -6
ATTN_ERR_TIMEOUT = -7

# Every function the header declares, with its ctypes signature.
_VP, _I, _UIP = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_uint)
SIGNATURES = {
    "attn_dense_fwd": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP]),
    "attn_prefix_fwd": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _VP]),
    "attn_status_string": (ctypes.c_char_p, [_I]),
    "attn_device_status": (_I, [_VP, _UIP]),
    "attn_debug_set_fault": (_I, [_I, ctypes.c_uint]),
    "attn_debug_exp2": (_I, [_VP, _VP, ctypes.c_longlong, _I, _VP]),
    "attn_debug_schedule": (_I, [_I, _I, _I, _I, _I, _I, _VP, _I, _VP, _I, _VP, _VP, _VP]),
    "attn_dense_fwd_noalloc": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP]),
    "attn_block_causal_fwd": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP]),
    "attn_dense_cross_fwd": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP]),
    "attn_masked_prefix_fwd": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_float, _VP, _I, _I,
                                    _I, _I, _I, _VP]),
}

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    """A nonzero attn_status returned by the library."""

    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def library_path() -> str:
    return _build.LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load the compiled library (it must exist: see ``build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is missing: run non_causal_prefix_gb300.build()")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, what: str):
    if rc != ATTN_OK:
        raise AttnError(rc, what)


def _bnhd(t, name):
    if t.dim() != 4:
        raise ValueError(f"{name} must be [B, N, H, D]")
    return t.shape


def attn_dense_fwd(q, k, v, out, stream=None) -> None:
    """Enqueue dense attention: q, k, v, out are CUDA bf16 [B, N, H, D] tensors."""
    B, N, H, D = _bnhd(q, "q")
    for t, n in ((k, "k"), (v, "v"), (out, "out")):
        if tuple(t.shape) != (B, N, H, D):
            raise ValueError(f"{n} must have q's shape {tuple(q.shape)}")
    _check_tensors(q, k, v, out)
    rc = load_library().attn_dense_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                       B, N, H, D, _stream_handle(stream))
    _check(rc, "attn_dense_fwd")


def attn_dense_fwd_noalloc(q, k, v, out, stream=None) -> None:
    """``attn_dense_fwd`` with its workspace in the library's static device
    scratch instead of a cudaMalloc'd one (see the C header: calls that
    overlap on the GPU race on that scratch)."""
    B, N, H, D = _bnhd(q, "q")
    for t, n in ((k, "k"), (v, "v"), (out, "out")):
        if tuple(t.shape) != (B, N, H, D):
            raise ValueError(f"{n} must have q's shape {tuple(q.shape)}")
    _check_tensors(q, k, v, out)
    rc = load_library().attn_dense_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                               out.data_ptr(), B, N, H, D, _stream_handle(stream))
    _check(rc, "attn_dense_fwd_noalloc")


def attn_dense_cross_fwd(q, k, v, out, stream=None) -> None:
    """Enqueue dense cross attention: q, out [B, Nq, H, D]; k, v [B, Nk, H, D]."""
    B, Nq, H, D = _bnhd(q, "q")
    Bk, Nk, Hk, Dk = _bnhd(k, "k")
    if (Bk, Hk, Dk) != (B, H, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k/v must be [B, Nk, H, D] with q's B, H, D")
    if tuple(out.shape) != (B, Nq, H, D):
        raise ValueError("out must have q's shape")
    _check_tensors(q, k, v, out)
    rc = load_library().attn_dense_cross_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                             out.data_ptr(), B, Nq, Nk, H, D,
                                             _stream_handle(stream))
    _check(rc, "attn_dense_cross_fwd")


def attn_prefix_fwd(q, kp, vp, kc, vc, out, stream=None) -> None:
    """Enqueue prefix-cached attention over cat(kp, kc) / cat(vp, vc).

    kp/vp may be None or have Np == 0 (then only the current keys are used).
    """
    B, Nq, H, D = _bnhd(q, "q")
    Bc, Nc, Hc, Dc = _bnhd(kc, "kc")
    if (Bc, Hc, Dc) != (B, H, D) or tuple(vc.shape) != tuple(kc.shape):
        raise ValueError("kc/vc must be [B, Nc, H, D] with q's B, H, D")
    Np = 0 if kp is None else kp.shape[1]
    if Np > 0 and (tuple(kp.shape) != (B, Np, H, D) or tuple(vp.shape) != tuple(kp.shape)):
        raise ValueError("kp/vp must be [B, Np, H, D] with q's B, H, D")
    if tuple(out.shape) != (B, Nq, H, D):
        raise ValueError("out must have q's shape")
    tensors = [q, kc, vc, out] + ([kp, vp] if Np > 0 else [])
    _check_tensors(*tensors)
    rc = load_library().attn_prefix_fwd(
        q.data_ptr(), kp.data_ptr() if Np > 0 else None, vp.data_ptr() if Np > 0 else None,
        kc.data_ptr(), vc.data_ptr(), out.data_ptr(), B, Nq, Np, Nc, H, D,
        _stream_handle(stream))
    _check(rc, "attn_prefix_fwd")


def attn_block_causal_fwd(q, k, v, image_ids, out, stream=None) -> None:
    """Enqueue block-causal attention: q, k, v, out CUDA bf16 [B, N, H, D];
    image_ids a CUDA int32 tensor [N] (-1 = text token, >= 0 = image id)."""
    import torch
    B, N, H, D = _bnhd(q, "q")
    for t, n in ((k, "k"), (v, "v"), (out, "out")):
        if tuple(t.shape) != (B, N, H, D):
            raise ValueError(f"{n} must have q's shape {tuple(q.shape)}")
    if image_ids.dtype != torch.int32 or not image_ids.is_cuda or not image_ids.is_contiguous():
        raise ValueError("image_ids must be a contiguous CUDA int32 tensor")
    if tuple(image_ids.shape) != (N,):
        raise ValueError("image_ids must be [N]")
    _check_tensors(q, k, v, out)
    rc = load_library().attn_block_causal_fwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), image_ids.data_ptr(), out.data_ptr(),
        B, N, H, D, _stream_handle(stream))
    _check(rc, "attn_block_causal_fwd")


def block_causal_attention(q, k, v, image_ids, stream=None):
    """Allocate ``out`` with torch and run ``attn_block_causal_fwd``."""
    import torch
    out = torch.empty_like(q)
    attn_block_causal_fwd(q, k, v, image_ids, out, stream)
    return out


def attn_masked_prefix_fwd(q, kc, vc, kp, vp, image_ids, key_valid, sm_scale, out,
                           stream=None) -> None:
    """Enqueue the masked prefix-cached form: q, kc, vc, out [B, Nq, H, D]; kp, vp
    [B, Np, H, D] (or None); image_ids int32 [Np + Nq]; key_valid bool/uint8
    [B, Np + Nq] (or None: all valid); sm_scale > 0."""
    import torch
    B, Nq, H, D = _bnhd(q, "q")
    for t, n in ((kc, "kc"), (vc, "vc"), (out, "out")):
        if tuple(t.shape) != (B, Nq, H, D):
            raise ValueError(f"{n} must have q's shape {tuple(q.shape)}")
    Np = 0 if kp is None else kp.shape[1]
    if Np > 0 and (tuple(kp.shape) != (B, Np, H, D) or tuple(vp.shape) != tuple(kp.shape)):
        raise ValueError("kp/vp must be [B, Np, H, D] with q's B, H, D")
    if image_ids.dtype != torch.int32 or not image_ids.is_cuda or not image_ids.is_contiguous():
        raise ValueError("image_ids must be a contiguous CUDA int32 tensor")
    if tuple(image_ids.shape) != (Np + Nq,):
        raise ValueError("image_ids must be [Np + Nq]")
    kv_ptr = None
    if key_valid is not None:
        if key_valid.dtype not in (torch.bool, torch.uint8) or not key_valid.is_cuda \
                or not key_valid.is_contiguous() or tuple(key_valid.shape) != (B, Np + Nq):
            raise ValueError("key_valid must be a contiguous CUDA bool/uint8 tensor [B, Np + Nq]")
        kv_ptr = key_valid.data_ptr()
    _check_tensors(*([q, kc, vc, out] + ([kp, vp] if Np > 0 else [])))
    rc = load_library().attn_masked_prefix_fwd(
        q.data_ptr(), kc.data_ptr(), vc.data_ptr(), kp.data_ptr() if Np > 0 else None,
        vp.data_ptr() if Np > 0 else None, image_ids.data_ptr(), kv_ptr, float(sm_scale),
        out.data_ptr(), B, Nq, Np, H, D, _stream_handle(stream))
    _check(rc, "attn_masked_prefix_fwd")


def _check_tensors(*ts):
    import torch
    for t in ts:
        if t.dtype != torch.bfloat16:
            raise TypeError("tensors must be bfloat16")
        if not t.is_cuda:
            raise ValueError("tensors must be CUDA tensors")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous [B, N, H, D]")


def dense_attention(q, k, v, stream=None):
    """Allocate ``out`` with torch and run ``attn_dense_fwd``."""
    import torch
    out = torch.empty_like(q)
    attn_dense_fwd(q, k, v, out, stream)
    return out


def prefix_attention(q, kp, vp, kc, vc, stream=None):
    """Allocate ``out`` with torch and run ``attn_prefix_fwd``."""
    import torch
    out = torch.empty_like(q)
    attn_prefix_fwd(q, kp, vp, kc, vc, out, stream)
    return out


def device_status(stream=None):
    """(status, info) of attn_device_status: synchronises the stream."""
    info = ctypes.c_uint(0)
    rc = load_library().attn_device_status(_stream_handle(stream), ctypes.byref(info))
    return rc, info.value


def debug_exp2(x, mode: int, stream=None):
    """2^x on the GPU through the softmax's polynomial (mode 0) or MUFU (mode 1)
    exponential; x is a CUDA float32 tensor, returns a new tensor."""
    import torch
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA float32 tensor")
    y = torch.empty_like(x)
    _check(load_library().attn_debug_exp2(x.data_ptr(), y.data_ptr(), x.numel(), int(mode),
                                          _stream_handle(stream)), "attn_debug_exp2")
    return y


def debug_set_fault(mode: int, wait_limit_us: int = 0) -> None:
    _check(load_library().attn_debug_set_fault(int(mode), int(wait_limit_us)),
           "attn_debug_set_fault")


def debug_schedule(B: int, Nq: int, H: int, n_key_tiles: int, sms: int, masked: bool = False,
                   image_ids=None, Np: int = 0):
    """The launch schedule for these sizes on a GPU with `sms` SMs, computed on
    the host: (rows, grid, slots) with rows an int32 array [items, 12] of
    (cta, n, b, h, q0, two, t_begin, t_end, tail, piece, pieces, slot0).
    Masked forms take image_ids (Np + Nq ints) and Np; n_key_tiles is then
    ignored."""
    import numpy as np
    lib = load_library()
    ids = None
    if masked:
        ids = np.ascontiguousarray(np.asarray(image_ids, dtype=np.int32))
        if ids.shape != (Np + Nq,):
            raise ValueError("image_ids must hold Np + Nq ids")
    ids_ptr = ids.ctypes.data if ids is not None else None
    n_rows, grid, slots = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    args = (int(B), int(Nq), int(H), int(n_key_tiles), int(sms), 1 if masked else 0, ids_ptr,
            int(Np))
    rc = lib.attn_debug_schedule(*args, None, 0, ctypes.byref(n_rows), ctypes.byref(grid),
                                 ctypes.byref(slots))
    if rc not in (0, -2) or (rc == -2 and n_rows.value == 0):
        _check(rc, "attn_debug_schedule")
    rows = np.zeros((max(n_rows.value, 1), 12), dtype=np.int32)
    _check(lib.attn_debug_schedule(*args, rows.ctypes.data, rows.shape[0], ctypes.byref(n_rows),
                                   ctypes.byref(grid), ctypes.byref(slots)), "attn_debug_schedule")
    return rows[:n_rows.value], grid.value, slots.value
