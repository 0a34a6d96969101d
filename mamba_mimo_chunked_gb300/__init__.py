"""GB300 (sm_103a) implementation of the backward stages of the Mamba-3 MIMO
chunked scan: ``mamba_mimo_bwd_fwd`` (first stage; ``mamba_mimo_bwd_fwd_with_y``
also writes the forward output y) and ``mamba_mimo_bwd_bwd`` (second stage,
the reverse scan and its 12 gradients).

This module is a thin binding over the C ABI in
``include/mamba_mimo_bwd_fwd.h`` and ``include/mamba_mimo_bwd_bwd.h``
(``libmmbf.so``): it checks shapes, dtypes and devices the way the PR #125
page's ``_validate_inputs`` does (same exception types), allocates outputs
and workspace with torch, and passes raw device pointers and the current
CUDA stream.  Every step of the computation
runs in the library's CUDA kernels; there is no fallback of any kind.  If the
library is missing or cannot load, calls raise.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import NamedTuple

import torch

from . import _build

__all__ = ["MambaMimoBwdFwdOutputs", "mamba_mimo_bwd_fwd", "mamba_mimo_bwd_fwd_with_y", "workspace_size",
           "load_library", "last_launch_count", "build", "mamba_mimo_bwd_bwd", "bwd_bwd_workspace_size",
           "BWD_BWD_OUTPUTS"]

build = _build.build

_lock = threading.Lock()
_lib = None

MMBF_ERRORS = {
    1: ValueError,          # shape
    2: ValueError,          # argument pattern
    3: NotImplementedError,  # outside this build's envelope
    4: ValueError,          # alignment
    5: ValueError,          # workspace
    6: RuntimeError,        # CUDA
    7: TimeoutError,        # a bounded wait inside a kernel ran out
}


class MambaMimoBwdFwdOutputs(NamedTuple):
    """The five outputs of the first Mamba-3 MIMO backward stage."""

    dmimo_o: torch.Tensor | None
    states: torch.Tensor
    dz: torch.Tensor | None
    dmimo_z: torch.Tensor | None
    qk_dot: torch.Tensor


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("B", "S", "H", "G", "R", "N", "P")]


def load_library():
    """Load ``libmmbf.so`` (built in-tree by ``build()``); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is missing; run mamba_mimo_chunked_gb300.build()")
        lib = ctypes.CDLL(path)
        vp, i64, f32p = ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p
        lib.mamba_mimo_bwd_fwd.restype = ctypes.c_int
        lib.mamba_mimo_bwd_fwd.argtypes = (
            [ctypes.POINTER(_Dims)] + [vp] * 17 + [i64, i64] + [vp] * 6 + [ctypes.c_size_t, vp])
        lib.mamba_mimo_bwd_fwd_y.restype = ctypes.c_int
        lib.mamba_mimo_bwd_fwd_y.argtypes = (
            [ctypes.POINTER(_Dims)] + [vp] * 17 + [i64, i64] + [vp] * 7 + [ctypes.c_size_t, vp])
        lib.mamba_mimo_bwd_fwd_workspace_size.restype = ctypes.c_int
        lib.mamba_mimo_bwd_fwd_workspace_size.argtypes = [
            ctypes.POINTER(_Dims), i64, i64, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]
        lib.mamba_mimo_last_error.restype = ctypes.c_char_p
        lib.mamba_mimo_abi_version.restype = ctypes.c_int
        lib.mamba_mimo_last_launch_count.restype = ctypes.c_int
        lib.mamba_mimo_set_stage_events.restype = None
        lib.mamba_mimo_set_stage_events.argtypes = [ctypes.c_void_p, ctypes.c_int]
        lib.mamba_mimo_last_kernel_variant.restype = ctypes.c_int
        lib.mamba_mimo_device_status.restype = ctypes.c_int
        lib.mamba_mimo_device_status.argtypes = [ctypes.c_void_p]
        lib.mamba_mimo_set_test_hooks.restype = None
        lib.mamba_mimo_set_test_hooks.argtypes = [ctypes.c_int]
        lib.mamba_mimo_last_plan.restype = ctypes.c_int
        lib.mamba_mimo_last_plan.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.c_int]
        lib.mamba_mimo_stage_name.restype = ctypes.c_char_p
        lib.mamba_mimo_stage_name.argtypes = [ctypes.c_int]
        lib.mamba_mimo_bwd_bwd.restype = ctypes.c_int
        lib.mamba_mimo_bwd_bwd.argtypes = (
            [ctypes.POINTER(_Dims)] + [vp] * 17 + [i64, i64, ctypes.c_int, ctypes.c_int] + [vp] * 12 + [vp, ctypes.c_size_t, vp])
        lib.mamba_mimo_bwd_bwd_workspace_size.restype = ctypes.c_int
        lib.mamba_mimo_bwd_bwd_workspace_size.argtypes = [
            ctypes.POINTER(_Dims), i64, i64, ctypes.POINTER(ctypes.c_size_t)]
        _lib = lib
        del f32p
    return _lib


def _raise(lib, status: int):
    msg = lib.mamba_mimo_last_error().decode(errors="replace")
    raise MMBF_ERRORS.get(status, RuntimeError)(f"mamba_mimo_bwd_fwd: {msg} (status {status})")


def last_kernel_variant() -> int:
    """-1 if the last call on this thread used the generic kernels, else the
    index of the shape-specialised kernel family it used."""
    return load_library().mamba_mimo_last_kernel_variant()


def device_status(stream=None) -> None:
    """Synchronise the stream and raise if a bounded wait inside a kernel of
    this thread's last call ran out (its outputs are then incomplete)."""
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    st = lib.mamba_mimo_device_status(ctypes.c_void_p(stream))
    if st:
        _raise(lib, st)


def last_plan() -> dict:
    """Launch plan of the last successful call on this thread."""
    buf = (ctypes.c_int * 7)()
    n = load_library().mamba_mimo_last_plan(buf, 7)
    keys = ("chunks_per_segment", "segments", "units_per_segment", "chunks_per_unit", "output_slots",
            "single_kernel", "single_kernel_refused")
    return dict(zip(keys, list(buf)[:n]))


def last_launch_count() -> int:
    """Kernel launches enqueued by the last successful call on this thread."""
    return load_library().mamba_mimo_last_launch_count()


def _check(name, t, shape, dtype, device):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {list(shape)}, got {list(t.shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


def _validate(dout, q, k, v, q_bias, k_bias, mimo_v, mimo_o, z, mimo_z, angles, da_cs, da_cs_rev,
              dt, trap, d, segsum, chunk_size, rotary_dim_divisor):
    """Input checks in the order of the PR #125 API's _validate_inputs."""
    if q.dim() != 5:
        raise ValueError("q must have shape [B, S, R, G, N]")
    B, S, R, G, N = q.shape
    if B < 1 or S < 1 or R < 1 or G < 1:
        raise ValueError("B, S, R and G must be positive")
    if q.dtype != torch.bfloat16:
        raise TypeError("q, k, v, dout and trap must use torch.bfloat16")
    if q.device.type != "cuda":
        raise ValueError("mamba_mimo_bwd_fwd requires CUDA tensors")
    if chunk_size < 1 or chunk_size * R > 128:
        raise ValueError("chunk_size * R must be in [1, 128]")
    if rotary_dim_divisor not in (2, 4):
        raise ValueError("rotary_dim_divisor must be 2 or 4")
    if N % rotary_dim_divisor or N % 2:
        raise ValueError("N must be even and divisible by rotary_dim_divisor")
    if N > 128:
        raise ValueError("N greater than 128 is not supported")
    if k.shape != q.shape:
        raise ValueError("k must have the same shape as q")
    if v.dim() != 4 or tuple(v.shape[:2]) != (B, S):
        raise ValueError("v must have shape [B, S, H, P]")
    H, P = v.shape[2:]
    if H % G:
        raise ValueError("H must be divisible by G")
    if P > 128:
        raise ValueError("P greater than 128 is not supported")
    dev = q.device
    bf16, f32 = torch.bfloat16, torch.float32
    _check("k", k, q.shape, bf16, dev)
    _check("v", v, (B, S, H, P), bf16, dev)
    _check("q_bias", q_bias, (H, R, N), f32, dev)
    _check("k_bias", k_bias, (H, R, N), f32, dev)
    _check("mimo_v", mimo_v, (H, R, P), f32, dev)
    _check("angles", angles, (B, S, H, N // rotary_dim_divisor), f32, dev)
    for name, t in (("da_cs", da_cs), ("da_cs_rev", da_cs_rev), ("dt", dt)):
        _check(name, t, (B, H, S), f32, dev)
    _check("trap", trap, (B, H, S), bf16, dev)
    nc = (S + chunk_size - 1) // chunk_size
    _check("segsum", segsum, (B, H, nc, chunk_size, chunk_size), f32, dev)
    if d is not None:
        _check("d", d, (H,), f32, dev)
    if mimo_o is not None:
        _check("mimo_o", mimo_o, (H, R, P), f32, dev)
        _check("dout", dout, (B, S, H, P), bf16, dev)
    else:
        _check("dout", dout, (B, S, R, H, P), bf16, dev)
    if z is None:
        if mimo_z is not None:
            raise ValueError("mimo_z must be None when z is None")
    else:
        _check("z", z, (B, S, H, P), bf16, dev)
        if mimo_z is None:
            raise ValueError("mimo_z is required when z is present")
        _check("mimo_z", mimo_z, (H, R, P), f32, dev)
    return B, S, H, G, R, N, P


def workspace_size(B, S, H, G, R, N, P, chunk_size=16, rotary_dim_divisor=4, reduced=True,
                   has_z=True) -> int:
    """Device workspace bytes for a problem (a query; no GPU needed)."""
    lib = load_library()
    nbytes = ctypes.c_size_t(0)
    st = lib.mamba_mimo_bwd_fwd_workspace_size(
        ctypes.byref(_Dims(B, S, H, G, R, N, P)), chunk_size, rotary_dim_divisor, int(reduced),
        int(has_z), ctypes.byref(nbytes))
    if st:
        _raise(lib, st)
    return nbytes.value


_ws_cache: dict = {}


def _workspace(device, nbytes: int) -> torch.Tensor:
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def mamba_mimo_bwd_fwd(dout, q, k, v, q_bias, k_bias, mimo_v, mimo_o, z, mimo_z, angles, da_cs,
                       da_cs_rev, dt, trap, d, segsum, chunk_size: int = 16,
                       rotary_dim_divisor: int = 4, *, out: MambaMimoBwdFwdOutputs | None = None,
                       workspace: torch.Tensor | None = None) -> MambaMimoBwdFwdOutputs:
    """First Mamba-3 MIMO backward stage on the current CUDA stream.

    Arguments follow the pages' positional order.  ``mimo_o`` selects reduced
    ``dout`` ([B,S,H,P]) and produces ``dmimo_o``; ``z`` (with ``mimo_z``)
    produces ``dz`` and ``dmimo_z``; ``d`` adds the skip term.  ``out`` may
    pass preallocated outputs (same shapes/dtypes as returned); ``workspace``
    a uint8 device buffer of at least ``workspace_size(...)`` bytes.
    """
    return _run(dout, q, k, v, q_bias, k_bias, mimo_v, mimo_o, z, mimo_z, angles, da_cs, da_cs_rev,
                dt, trap, d, segsum, chunk_size, rotary_dim_divisor, out, workspace, None)


def mamba_mimo_bwd_fwd_with_y(dout, q, k, v, q_bias, k_bias, mimo_v, mimo_o, z, mimo_z, angles,
                              da_cs, da_cs_rev, dt, trap, d, segsum, chunk_size: int = 16,
                              rotary_dim_divisor: int = 4, *,
                              out: MambaMimoBwdFwdOutputs | None = None,
                              workspace: torch.Tensor | None = None, y: torch.Tensor | None = None):
    """mamba_mimo_bwd_fwd plus the layer's forward output ``y`` (BF16, shaped
    like ``dout``): sum over ranks of mimo_o * out * silu(z * mimo_z), or per
    rank without ``mimo_o`` (no gate without ``z``).  Returns (outputs, y)."""
    if y is None:
        y = torch.empty(dout.shape, dtype=torch.bfloat16, device=q.device)
    res = _run(dout, q, k, v, q_bias, k_bias, mimo_v, mimo_o, z, mimo_z, angles, da_cs, da_cs_rev,
               dt, trap, d, segsum, chunk_size, rotary_dim_divisor, out, workspace, y)
    return res, y


def _run(dout, q, k, v, q_bias, k_bias, mimo_v, mimo_o, z, mimo_z, angles, da_cs, da_cs_rev, dt,
         trap, d, segsum, chunk_size, rotary_dim_divisor, out, workspace, y):
    args = (dout, q, k, v, q_bias, k_bias, mimo_v, mimo_o, z, mimo_z, angles, da_cs, da_cs_rev,
            dt, trap, d, segsum)
    B, S, H, G, R, N, P = _validate(*args, chunk_size, rotary_dim_divisor)
    lib = load_library()
    dev = q.device
    args = tuple(None if a is None else a.contiguous() for a in args)
    nc = (S + chunk_size - 1) // chunk_size
    if out is None:
        out = MambaMimoBwdFwdOutputs(
            torch.empty((B, H, R, P), dtype=torch.float32, device=dev) if mimo_o is not None else None,
            torch.empty((B, H, nc, N, P), dtype=torch.bfloat16, device=dev),
            torch.empty((B, S, H, P), dtype=torch.bfloat16, device=dev) if z is not None else None,
            torch.empty((B, H, R, P), dtype=torch.float32, device=dev) if z is not None else None,
            torch.empty((B, H, S, R, R), dtype=torch.bfloat16, device=dev))
    nbytes = workspace_size(B, S, H, G, R, N, P, chunk_size, rotary_dim_divisor, mimo_o is not None,
                            z is not None)
    if workspace is None:
        workspace = _workspace(dev, nbytes)
    stream = torch.cuda.current_stream(dev).cuda_stream
    if y is not None:
        if y.dtype != torch.bfloat16 or tuple(y.shape) != tuple(dout.shape) or not y.is_contiguous() \
                or y.device != dev:
            raise ValueError("y must be a contiguous bf16 tensor shaped like dout on the inputs' device")
    with torch.cuda.device(dev):
        if y is None:
            st = lib.mamba_mimo_bwd_fwd(
                ctypes.byref(_Dims(B, S, H, G, R, N, P)), *[_ptr(a) for a in args], chunk_size,
                rotary_dim_divisor, *[_ptr(o) for o in out], _ptr(workspace),
                workspace.numel() * workspace.element_size(), ctypes.c_void_p(stream))
        else:
            st = lib.mamba_mimo_bwd_fwd_y(
                ctypes.byref(_Dims(B, S, H, G, R, N, P)), *[_ptr(a) for a in args], chunk_size,
                rotary_dim_divisor, *[_ptr(o) for o in out], _ptr(y), _ptr(workspace),
                workspace.numel() * workspace.element_size(), ctypes.c_void_p(stream))
    if st:
        _raise(lib, st)
    return out


# ---------------------------------------------------------------------------
# Second backward stage (include/mamba_mimo_bwd_bwd.h)

BWD_BWD_OUTPUTS = ("DQ", "DK", "DV", "DMIMO_V", "DANGLES", "DFACTOR", "DGAMMA", "DDA", "DSSDA",
                   "DDA_CS_REV", "DDA_CS", "DD")


def bwd_bwd_workspace_size(B, S, H, G, R, N, P, chunk_size=16, rotary_dim_divisor=4) -> int:
    """Device workspace bytes of mamba_mimo_bwd_bwd (a query; no GPU needed)."""
    lib = load_library()
    nbytes = ctypes.c_size_t(0)
    st = lib.mamba_mimo_bwd_bwd_workspace_size(ctypes.byref(_Dims(B, S, H, G, R, N, P)), chunk_size,
                                               rotary_dim_divisor, ctypes.byref(nbytes))
    if st:
        _raise(lib, st)
    return nbytes.value


# dtype codes of the second stage's C ABI (act_dtype, dqkv_dtype)
_BB_DTYPE_CODES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}


def mamba_mimo_bwd_bwd(dout, q, k, v, q_bias, k_bias, mimo_v, states, qk_dot, da_cs, da_cs_rev, dt,
                       trap, segsum, angles, mimo_o=None, d=None, chunk_size: int = 16,
                       rotary_dim_divisor: int = 4, output_dtype=None, *,
                       workspace: torch.Tensor | None = None) -> dict:
    """Second Mamba-3 MIMO backward stage on the current CUDA stream.

    Arguments in the pages' order (the first stage's ``states`` and
    ``qk_dot`` caches among them); ``mimo_o`` selects reduce-O ``dout``
    ([B,S,H,P]), ``d`` adds the D-skip gradient.  dout, q, k, v, states,
    qk_dot and trap share one dtype (float16, bfloat16 or float32, as on the
    pages); the other inputs are float32.  ``output_dtype`` sets the dtype
    of DQ, DK and DV (None: the inputs' dtype, as on the pages); the other
    nine gradients are FP32.  Returns a dict of the 12 gradients (``DD`` is
    None without ``d``)."""
    if q.dim() != 5:
        raise ValueError("q must have shape [B, S, R, G, N]")
    B, S, R, G, N = q.shape
    if q.dtype not in _BB_DTYPE_CODES:
        raise TypeError("q, k, v, dout, states, qk_dot and trap must use torch.float16, torch.bfloat16 "
                        "or torch.float32")
    if q.device.type != "cuda":
        raise ValueError("mamba_mimo_bwd_bwd requires CUDA tensors")
    if rotary_dim_divisor not in (2, 4):
        raise ValueError("rotary_dim_divisor must be 2 or 4")
    if N % 2 or N % rotary_dim_divisor:
        raise ValueError("N must be even and divisible by rotary_dim_divisor")
    if v.dim() != 4 or tuple(v.shape[:2]) != (B, S):
        raise ValueError("v must have shape [B, S, H, P]")
    H, P = v.shape[2:]
    if H % G:
        raise ValueError("H must be divisible by G")
    dev = q.device
    act, f32 = q.dtype, torch.float32
    nc = (S + chunk_size - 1) // chunk_size
    _check("k", k, q.shape, act, dev)
    _check("v", v, (B, S, H, P), act, dev)
    _check("q_bias", q_bias, (H, R, N), f32, dev)
    _check("k_bias", k_bias, (H, R, N), f32, dev)
    _check("mimo_v", mimo_v, (H, R, P), f32, dev)
    _check("states", states, (B, H, nc, N, P), act, dev)
    _check("qk_dot", qk_dot, (B, H, S, R, R), act, dev)
    for name, t in (("da_cs", da_cs), ("da_cs_rev", da_cs_rev), ("dt", dt)):
        _check(name, t, (B, H, S), f32, dev)
    _check("trap", trap, (B, H, S), act, dev)
    _check("segsum", segsum, (B, H, nc, chunk_size, chunk_size), f32, dev)
    _check("angles", angles, (B, S, H, N // rotary_dim_divisor), f32, dev)
    if mimo_o is not None:
        _check("mimo_o", mimo_o, (H, R, P), f32, dev)
        _check("dout", dout, (B, S, H, P), act, dev)
    else:
        _check("dout", dout, (B, S, R, H, P), act, dev)
    if d is not None:
        _check("d", d, (H,), f32, dev)
    if output_dtype is None:
        output_dtype = q.dtype
    if output_dtype not in _BB_DTYPE_CODES:
        raise TypeError("output_dtype must be None, torch.float16, torch.bfloat16 or torch.float32")
    args = tuple(None if a is None else a.contiguous() for a in (
        dout, q, k, v, q_bias, k_bias, mimo_v, states, qk_dot, da_cs, da_cs_rev, dt, trap, segsum,
        angles, mimo_o, d))
    lib = load_library()
    outs = {
        "DQ": torch.empty((B, S * R, H, N), dtype=output_dtype, device=dev),
        "DK": torch.empty((B, S * R, H, N), dtype=output_dtype, device=dev),
        "DV": torch.empty((B, S, H, P), dtype=output_dtype, device=dev),
        "DMIMO_V": torch.empty((B, H, R, P), dtype=f32, device=dev),
        "DANGLES": torch.empty((B, S, H, N // rotary_dim_divisor), dtype=f32, device=dev),
        "DFACTOR": torch.empty((B, H, S), dtype=f32, device=dev),
        "DGAMMA": torch.empty((B, H, S), dtype=f32, device=dev),
        "DDA": torch.empty((B, H, S), dtype=f32, device=dev),
        "DSSDA": torch.empty((B, H, nc, chunk_size, chunk_size), dtype=f32, device=dev),
        "DDA_CS_REV": torch.empty((B, H, S), dtype=f32, device=dev),
        "DDA_CS": torch.empty((B, H, S), dtype=f32, device=dev),
        "DD": torch.empty((B, H), dtype=f32, device=dev) if d is not None else None,
    }
    nbytes = bwd_bwd_workspace_size(B, S, H, G, R, N, P, chunk_size, rotary_dim_divisor)
    if workspace is None:
        workspace = _workspace(dev, nbytes)
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        st = lib.mamba_mimo_bwd_bwd(
            ctypes.byref(_Dims(B, S, H, G, R, N, P)), *[_ptr(a) for a in args], chunk_size,
            rotary_dim_divisor, _BB_DTYPE_CODES[act], _BB_DTYPE_CODES[output_dtype],
            *[_ptr(outs[n]) for n in BWD_BWD_OUTPUTS], _ptr(workspace),
            workspace.numel() * workspace.element_size(), ctypes.c_void_p(stream))
    if st:
        _raise(lib, st)
    return outs
