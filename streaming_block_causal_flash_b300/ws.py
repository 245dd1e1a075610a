"""Thin Python binding of the C ABI in ``include/ws.h`` (ctypes).

Same names as the C entry points.  Argument marshalling only: tensors are
checked for device, dtype, shape and contiguity, then their addresses, the
sizes and the current CUDA stream go to the native library, which does all
the work in its own kernels.  There is no other execution path: if the
native library is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# WS_DEBUG=1 selects the debug build (bounds-checked kernel indices; see
# build.py), built with `python -m streaming_block_causal_flash_b300.build --debug`.
LIB_PATH = os.path.join(_HERE, "libws_b300_debug.so" if os.environ.get("WS_DEBUG") == "1"
                        else "libws_b300.so")

WS_OK = 0
WS_ERR_INVALID_ARGUMENT = 1
WS_ERR_UNSUPPORTED = 2
WS_ERR_CAPACITY = 3
WS_ERR_CUDA = 4
WS_ERR_TIMEOUT = 5

WS_F32 = 0
WS_BF16 = 1

# Every symbol the header declares, with (restype, argtypes).
_c_i64, _c_int, _c_f32, _c_size, _c_u64 = (ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                           ctypes.c_size_t, ctypes.c_uint64)
_vp = ctypes.c_void_p
_i32p = ctypes.POINTER(ctypes.c_int32)
SIGNATURES = {
    "ws_kv_append": (_c_int, [_vp, _vp, _vp, _vp, _c_i64, _c_i64, _c_i64, _c_int, _c_int, _c_int, _vp]),
    "ws_block_causal_attn": (_c_int, [_vp, _vp, _vp, _vp, _vp, _i32p, _vp, _c_int, _c_i64, _c_int,
                                      _c_int, _c_f32, _c_int, _vp, _c_size, _vp]),
    "ws_block_causal_prefill": (_c_int, [_vp, _vp, _vp, _vp, _vp, _i32p, _vp, _c_int, _c_i64, _c_int,
                                         _c_int, _c_f32, _c_int, _vp, _c_size, _vp]),
    "ws_block_causal_attn_side": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _vp, _vp, _i32p, _vp, _c_int,
                                           _c_i64, _c_int, _c_int, _c_f32, _c_int, _vp, _c_size, _vp]),
    "ws_block_causal_attn_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _vp, _i32p, _vp, _c_int, _c_i64,
                                              _c_int, _c_int, _c_f32, _c_int, _vp]),
    "ws_fm_euler_step": (_c_int, [_vp, _c_int, _vp, _c_int, _vp, _c_i64, _c_f32, _vp]),
    "ws_fm_euler_cfg_step": (_c_int, [_vp, _c_int, _vp, _vp, _c_int, _vp, _c_i64, _c_f32, _c_f32, _vp]),
    "ws_block_causal_attn_workspace_size": (_c_size, [_c_i64, _c_i64, _c_int, _c_int]),
    "ws_kv_append_dev": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_i64, _c_i64, _c_int, _c_int, _c_int, _vp]),
    "ws_block_causal_attn_dev": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_i64, _c_i64, _c_int, _c_int,
                                          _c_f32, _c_int, _vp, _c_size, _vp]),
    "ws_block_causal_attn_dev_workspace_size": (_c_size, [_c_i64, _c_i64, _c_int, _c_int]),
    "ws_unit_state_advance": (_c_int, [_vp, _vp, _c_i64, _vp]),
    "ws_status_string": (ctypes.c_char_p, [_c_int]),
    "ws_last_error": (ctypes.c_char_p, []),
    "ws_get_device_error": (_c_int, [ctypes.POINTER(_c_int), ctypes.POINTER(_c_int)]),
    "ws_clear_device_error": (_c_int, []),
    "ws_set_wait_timeout_ns": (_c_int, [_c_u64]),
    "ws_debug_force_wait_timeout": (_c_int, [_c_int]),
    "ws_abi_version": (_c_int, []),
}

_lib = None


class WsError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_name(status)}: {message}")
        self.status = status


def load() -> ctypes.CDLL:
    """Load the in-tree native library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"native library {LIB_PATH} is missing; build it with "
                               "`python -m streaming_block_causal_flash_b300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_name(status: int) -> str:
    try:
        return load().ws_status_string(status).decode()
    except Exception:           # library not loadable: plain number
        return f"status {status}"


def _check(status: int):
    if status != WS_OK:
        raise WsError(status, load().ws_last_error().decode())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return WS_BF16
    if t.dtype == torch.float32:
        return WS_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: Optional[torch.Tensor], name: str, dtype=None) -> int:
    if t is None:
        return 0
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}")
    return t.data_ptr()


def _host_offsets(offsets) -> np.ndarray:
    arr = np.ascontiguousarray(np.asarray(offsets), dtype=np.int32)
    if arr.ndim != 1 or arr.size < 2:
        raise ValueError("offsets must be 1-D with at least two entries")
    return arr


def ws_kv_append(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                 v_cache: torch.Tensor, cache_len: int, stream=None) -> None:
    """cache[h, cache_len + t] = slice[t, h] for K and V ([n,H,D] -> [H,cap,D])."""
    n, H, D = k_new.shape
    if tuple(v_new.shape) != (n, H, D):
        raise ValueError("K and V slices differ in shape")
    if k_cache.dim() != 3 or k_cache.shape[0] != H or k_cache.shape[2] != D or \
            tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shape must be [H, capacity, D] and match the slice")
    dt = k_new.dtype
    _check(load().ws_kv_append(_dev(k_new, "k_new"), _dev(v_new, "v_new", dt),
                               _dev(k_cache, "k_cache", dt), _dev(v_cache, "v_cache", dt),
                               int(cache_len), int(n), int(k_cache.shape[1]), int(H), int(D),
                               _dtype_code(k_new), _stream_ptr(stream)))


def _attn_shapes(q, k_cache, v_cache, out, offsets_host, offsets_dev, lse, prefill: bool):
    """Shape checks the C ABI cannot make (it sees only pointers): the caches
    are [H, capacity, D] and equal in shape, and q/out hold exactly the rows
    the offsets give -- the newest block (offsets[-1] - offsets[-2] rows), or
    every token for prefill (offsets[-1] rows).  Returns (H, cap, D, offs)."""
    if k_cache.dim() != 3 or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache must both be [H, capacity, D]")
    H, cap, D = k_cache.shape
    offs = _host_offsets(offsets_host)
    if offsets_dev.dtype != torch.int32 or offsets_dev.numel() != offs.size:
        raise ValueError("device offsets must be int32 with the same length as host offsets")
    if q.dim() != 3 or q.shape[1] != H or q.shape[2] != D or tuple(out.shape) != tuple(q.shape):
        raise ValueError("q/out must be [rows, H, D]")
    rows = int(offs[-1]) if prefill else int(offs[-1]) - int(offs[-2])
    if q.shape[0] != rows:
        raise ValueError(f"q has {q.shape[0]} rows; the offsets give {rows}")
    if lse is not None and (lse.dtype != torch.float32 or lse.numel() != H * q.shape[0]):
        raise ValueError("lse must be float32 [H, rows]")
    return H, cap, D, offs


def _attn(fn_name, q, k_cache, v_cache, out, offsets_host, offsets_dev, lse, softmax_scale,
          workspace, stream):
    H, cap, D, offs = _attn_shapes(q, k_cache, v_cache, out, offsets_host, offsets_dev, lse,
                                   fn_name == "ws_block_causal_prefill")
    dt = q.dtype
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    fn = getattr(load(), fn_name)
    _check(fn(_dev(q, "q"), _dev(k_cache, "k_cache", dt), _dev(v_cache, "v_cache", dt),
              _dev(out, "out", dt), _dev(lse, "lse", torch.float32),
              offs.ctypes.data_as(_i32p), _dev(offsets_dev, "offsets_dev", torch.int32),
              int(offs.size - 1), int(cap), int(H), int(D), float(softmax_scale),
              _dtype_code(q), ws_ptr, ws_bytes, _stream_ptr(stream)))


def ws_block_causal_attn(q, k_cache, v_cache, out, offsets_host: Sequence[int],
                         offsets_dev: torch.Tensor, lse: Optional[torch.Tensor] = None,
                         softmax_scale: float = 0.0, workspace: Optional[torch.Tensor] = None,
                         stream=None) -> None:
    """Newest unit's queries (the last block) against the whole cache."""
    _attn("ws_block_causal_attn", q, k_cache, v_cache, out, offsets_host, offsets_dev, lse,
          softmax_scale, workspace, stream)


def ws_block_causal_attn_side(q, k_cache, v_cache, k_side, v_side, out,
                              offsets_host: Sequence[int], offsets_dev: torch.Tensor,
                              lse: Optional[torch.Tensor] = None, softmax_scale: float = 0.0,
                              workspace: Optional[torch.Tensor] = None, commit: bool = False,
                              stream=None) -> None:
    """Newest unit's queries against the cache (blocks before the last) plus
    the unit's own K/V from token-major side buffers [q_len, H, D]; with
    commit=True the kernel also writes those K/V into the cache rows of the
    last block (the append fused into the attention)."""
    H, cap, D, offs = _attn_shapes(q, k_cache, v_cache, out, offsets_host, offsets_dev, lse, False)
    dt = q.dtype
    if tuple(k_side.shape) != tuple(q.shape) or tuple(v_side.shape) != tuple(q.shape):
        raise ValueError("k_side/v_side must be [rows, H, D] like q")
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    _check(load().ws_block_causal_attn_side(
        _dev(q, "q"), _dev(k_cache, "k_cache", dt), _dev(v_cache, "v_cache", dt),
        _dev(k_side, "k_side", dt), _dev(v_side, "v_side", dt), 1 if commit else 0, _dev(out, "out", dt),
        _dev(lse, "lse", torch.float32), offs.ctypes.data_as(_i32p),
        _dev(offsets_dev, "offsets_dev", torch.int32), int(offs.size - 1), int(cap), int(H), int(D),
        float(softmax_scale), _dtype_code(q), ws_ptr, ws_bytes, _stream_ptr(stream)))


def ws_block_causal_attn_noalloc(q, k_cache, v_cache, out, offsets_host: Sequence[int],
                                 offsets_dev: torch.Tensor, lse: Optional[torch.Tensor] = None,
                                 softmax_scale: float = 0.0, stream=None) -> None:
    """ws_block_causal_attn without a caller workspace, for callers that may
    not allocate device memory: the library's static device scratch stands in
    for it.  Calls that can overlap on the GPU race on that scratch."""
    H, cap, D, offs = _attn_shapes(q, k_cache, v_cache, out, offsets_host, offsets_dev, lse, False)
    dt = q.dtype
    _check(load().ws_block_causal_attn_noalloc(
        _dev(q, "q"), _dev(k_cache, "k_cache", dt), _dev(v_cache, "v_cache", dt),
        _dev(out, "out", dt), _dev(lse, "lse", torch.float32), offs.ctypes.data_as(_i32p),
        _dev(offsets_dev, "offsets_dev", torch.int32), int(offs.size - 1), int(cap), int(H), int(D),
        float(softmax_scale), _dtype_code(q), _stream_ptr(stream)))


def ws_block_causal_prefill(q, k_cache, v_cache, out, offsets_host: Sequence[int],
                            offsets_dev: torch.Tensor, lse: Optional[torch.Tensor] = None,
                            softmax_scale: float = 0.0, stream=None) -> None:
    """Full-sequence block-causal attention over all offsets[-1] tokens."""
    _attn("ws_block_causal_prefill", q, k_cache, v_cache, out, offsets_host, offsets_dev, lse,
          softmax_scale, None, stream)


def ws_fm_euler_step(z: torch.Tensor, v: torch.Tensor, dtau: float,
                     z_bf16_out: Optional[torch.Tensor] = None, stream=None) -> None:
    """z <- z - dtau * v in place (z float32; v bf16 or float32)."""
    if z.numel() != v.numel():
        raise ValueError("z and v differ in size")
    if z_bf16_out is not None and z_bf16_out.numel() != z.numel():
        raise ValueError("z_bf16_out size mismatch")
    _check(load().ws_fm_euler_step(_dev(z, "z"), _dtype_code(z), _dev(v, "v"), _dtype_code(v),
                                   _dev(z_bf16_out, "z_bf16_out", torch.bfloat16), int(z.numel()),
                                   float(dtau), _stream_ptr(stream)))


def ws_fm_euler_cfg_step(z: torch.Tensor, v_uncond: torch.Tensor, v_cond: torch.Tensor,
                         guidance: float, dtau: float, z_bf16_out: Optional[torch.Tensor] = None,
                         stream=None) -> None:
    """z <- z - dtau * (v_u + guidance * (v_c - v_u)) in place (z float32)."""
    if not (z.numel() == v_uncond.numel() == v_cond.numel()):
        raise ValueError("z and the velocities differ in size")
    if v_uncond.dtype != v_cond.dtype:
        raise TypeError("v_uncond and v_cond must share a dtype")
    if z_bf16_out is not None and z_bf16_out.numel() != z.numel():
        raise ValueError("z_bf16_out size mismatch")
    _check(load().ws_fm_euler_cfg_step(_dev(z, "z"), _dtype_code(z), _dev(v_uncond, "v_uncond"),
                                       _dev(v_cond, "v_cond"), _dtype_code(v_uncond),
                                       _dev(z_bf16_out, "z_bf16_out", torch.bfloat16),
                                       int(z.numel()), float(guidance), float(dtau),
                                       _stream_ptr(stream)))


def ws_block_causal_attn_workspace_size(q_len: int, kv_len: int, num_heads: int,
                                        head_dim: int) -> int:
    n = load().ws_block_causal_attn_workspace_size(int(q_len), int(kv_len), int(num_heads),
                                                   int(head_dim))
    if n == ctypes.c_size_t(-1).value:
        raise WsError(WS_ERR_INVALID_ARGUMENT, "workspace size query failed")
    return int(n)


# ---------------------------------------------- device-resident unit sizes

def unit_state(cache_len: int, n_new: int, unit: int = 0, device="cuda") -> torch.Tensor:
    """A ws_unit_state {cache_len, n_new, unit} in device memory (int64 [3])."""
    return torch.tensor([int(cache_len), int(n_new), int(unit)], dtype=torch.int64, device=device)


def _state_ptr(state: torch.Tensor) -> int:
    if state.dtype != torch.int64 or state.numel() != 3:
        raise ValueError("state must be an int64 tensor of 3 values (ws_unit_state)")
    return _dev(state, "state")


def ws_kv_append_dev(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                     v_cache: torch.Tensor, state: torch.Tensor, stream=None) -> None:
    """ws_kv_append with cache_len / n_new read from the device state when the
    kernel runs; the slices are buffers of n_max = k_new.shape[0] rows."""
    n_max, H, D = k_new.shape
    if tuple(v_new.shape) != (n_max, H, D):
        raise ValueError("K and V slices differ in shape")
    if k_cache.dim() != 3 or k_cache.shape[0] != H or k_cache.shape[2] != D or \
            tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shape must be [H, capacity, D] and match the slice")
    dt = k_new.dtype
    _check(load().ws_kv_append_dev(_dev(k_new, "k_new"), _dev(v_new, "v_new", dt),
                                   _dev(k_cache, "k_cache", dt), _dev(v_cache, "v_cache", dt),
                                   _state_ptr(state), int(n_max), int(k_cache.shape[1]), int(H), int(D),
                                   _dtype_code(k_new), _stream_ptr(stream)))


def ws_block_causal_attn_dev_workspace_size(q_max: int, capacity: int, num_heads: int,
                                            head_dim: int) -> int:
    n = load().ws_block_causal_attn_dev_workspace_size(int(q_max), int(capacity), int(num_heads),
                                                       int(head_dim))
    if n == ctypes.c_size_t(-1).value:
        raise WsError(WS_ERR_INVALID_ARGUMENT, "workspace size query failed")
    return int(n)


def ws_block_causal_attn_dev(q, k_cache, v_cache, out, state: torch.Tensor,
                             lse: Optional[torch.Tensor] = None, softmax_scale: float = 0.0,
                             workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """The current unit's queries (rows < n_new of a q_max-row buffer) against
    the cache, sizes read from the device state when the kernels run."""
    if k_cache.dim() != 3 or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache must both be [H, capacity, D]")
    H, cap, D = k_cache.shape
    if q.dim() != 3 or q.shape[1] != H or q.shape[2] != D or tuple(out.shape) != tuple(q.shape):
        raise ValueError("q/out must be [q_max, H, D]")
    q_max = int(q.shape[0])
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (H, q_max)):
        raise ValueError("lse must be float32 [H, q_max]")
    if workspace is None:
        raise ValueError("ws_block_causal_attn_dev needs a workspace")
    dt = q.dtype
    _check(load().ws_block_causal_attn_dev(
        _dev(q, "q"), _dev(k_cache, "k_cache", dt), _dev(v_cache, "v_cache", dt), _dev(out, "out", dt),
        _dev(lse, "lse", torch.float32), _state_ptr(state), q_max, int(cap), int(H), int(D),
        float(softmax_scale), _dtype_code(q), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream)))


def ws_unit_state_advance(state: torch.Tensor, sizes_dev: torch.Tensor, stream=None) -> None:
    """cache_len += n_new; unit += 1; n_new = sizes[unit] (0 past the end)."""
    if sizes_dev.dtype != torch.int32 or sizes_dev.dim() != 1:
        raise ValueError("sizes must be a 1-D int32 device tensor")
    _check(load().ws_unit_state_advance(_state_ptr(state), _dev(sizes_dev, "sizes"),
                                        int(sizes_dev.numel()), _stream_ptr(stream)))


def ws_get_device_error():
    """(code, info) of the kernels' device error word (synchronises): code 1 a
    wait time-out, code 2 device-resident unit sizes out of range."""
    code, info = ctypes.c_int(0), ctypes.c_int(0)
    st = load().ws_get_device_error(ctypes.byref(code), ctypes.byref(info))
    if st not in (WS_OK, WS_ERR_TIMEOUT, WS_ERR_CAPACITY):
        _check(st)
    return code.value, info.value


def ws_clear_device_error() -> None:
    _check(load().ws_clear_device_error())


def ws_set_wait_timeout_ns(ns: int) -> None:
    _check(load().ws_set_wait_timeout_ns(int(ns)))


def ws_debug_force_wait_timeout(on: bool) -> None:
    """Test hook: make tensor-core attention launches give up on a wait."""
    _check(load().ws_debug_force_wait_timeout(1 if on else 0))


def ws_abi_version() -> int:
    return int(load().ws_abi_version())


def workspace_for(q_len: int, kv_len: int, num_heads: int, head_dim: int,
                  device="cuda") -> Optional[torch.Tensor]:
    """Allocate (with torch) the workspace ws_block_causal_attn needs, or None."""
    n = ws_block_causal_attn_workspace_size(q_len, kv_len, num_heads, head_dim)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device)
