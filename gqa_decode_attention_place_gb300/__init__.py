"""Python binding of libgqa_attn.so (include/gqa_attn.h).

Argument marshalling only: every function takes torch CUDA tensors, checks
their dtype, shape, contiguity and device, and passes raw device pointers and
the current CUDA stream to the C entry point of the same name.  All compute
runs in the library's CUDA kernels; there is no fallback path, and a missing
or unloadable library raises immediately.

With ``GQA_ATTN_DEBUG=1`` in the environment the range-checked build
(``lib/libgqa_attn_debug.so``, compiled with ``-DGQA_DEBUG``) is loaded
instead; ``attn_debug_build()`` says which one is in use.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

__all__ = [
    "AttnError", "load_library", "library_path",
    "attn_kv_append", "attn_decode_workspace_size", "attn_decode_step",
    "attn_prefill_causal", "attn_read_device_status", "attn_status_string",
    "attn_read_prefill_status", "attn_last_cuda_error", "decode_workspace", "attn_decode_step_noalloc",
    "attn_decode_step_append", "attn_decode_step_rope_append", "attn_decode_stream_step",
    "attn_decode_step_window", "attn_decode_multi", "attn_test_skip_tile",
    "attn_debug_build", "attn_read_prefill_skips", "debug_collect_range_bits",
    "attn_test_force_schedule",
]

ATTN_OK = 0
ATTN_DEV_BAD_POSITION = 0x1
ATTN_DEV_TIMEOUT = 0x2
ATTN_DEV_RANGE = 0x4

_LIB: Optional[ctypes.CDLL] = None
# Range-checked builds only: every workspace handed out by decode_workspace()
# (kept alive until debug_collect_range_bits() reads it), and any
# ATTN_DEV_RANGE bit a caller's own attn_read_device_status() saw.
_DEBUG_WORKSPACES: list = []
_DEBUG_RANGE_SEEN = 0


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {attn_status_string(code)} (status {code})"
        if code == 4:
            msg += f", CUDA error {attn_last_cuda_error()}"
        super().__init__(msg)


def _debug_requested() -> bool:
    return os.environ.get("GQA_ATTN_DEBUG", "0") not in ("", "0")


def library_path() -> str:
    return _build.lib_path(_debug_requested())


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libgqa_attn.so, or libgqa_attn_debug.so under GQA_ATTN_DEBUG=1
    (building it in-tree first if allowed and needed)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    debug = _debug_requested()
    path = _build.lib_path(debug)
    if not os.path.exists(path) or (build_if_missing and not _build.up_to_date(debug)):
        if not build_if_missing:
            raise RuntimeError(f"{path} is missing; run __graft_entry__.build()")
        _build.build(debug=debug)
    lib = ctypes.CDLL(path)
    vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    lib.attn_kv_append.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]
    lib.attn_kv_append.restype = i32
    lib.attn_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.attn_decode_workspace_size.restype = sz
    lib.attn_decode_step.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp, sz, vp]
    lib.attn_decode_step.restype = i32
    lib.attn_decode_step_append.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32,
                                            vp, vp, sz, vp]
    lib.attn_decode_step_append.restype = i32
    lib.attn_decode_step_rope_append.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                                 i32, i32, f32, vp, vp, sz, vp]
    lib.attn_decode_step_rope_append.restype = i32
    lib.attn_decode_stream_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                            i32, f32, vp, vp, sz, vp]
    lib.attn_decode_stream_step.restype = i32
    lib.attn_decode_step_window.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                            f32, vp, vp, sz, vp]
    lib.attn_decode_step_window.restype = i32
    lib.attn_decode_multi.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32,
                                      vp, vp, sz, vp]
    lib.attn_decode_multi.restype = i32
    lib.attn_test_skip_tile.argtypes = [i32]
    lib.attn_test_skip_tile.restype = i32
    lib.attn_test_force_schedule.argtypes = [i32]
    lib.attn_test_force_schedule.restype = i32
    lib.attn_decode_step_noalloc.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp]
    lib.attn_decode_step_noalloc.restype = i32
    lib.attn_prefill_causal.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp]
    lib.attn_prefill_causal.restype = i32
    lib.attn_read_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
    lib.attn_read_device_status.restype = i32
    lib.attn_read_prefill_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
    lib.attn_read_prefill_status.restype = i32
    lib.attn_status_string.argtypes = [i32]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_last_cuda_error.argtypes = []
    lib.attn_last_cuda_error.restype = i32
    lib.attn_debug_build.argtypes = []
    lib.attn_debug_build.restype = i32
    lib.attn_read_prefill_skips.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
    lib.attn_read_prefill_skips.restype = i32
    _LIB = lib
    return lib


def attn_status_string(code: int) -> str:
    return load_library().attn_status_string(int(code)).decode()


def attn_last_cuda_error() -> int:
    return int(load_library().attn_last_cuda_error())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _raise(code: int, where: str):
    if code != ATTN_OK:
        raise AttnError(code, where)


def attn_kv_append(k_new, v_new, positions, k_cache, v_cache, stream=None) -> None:
    """Write k_new/v_new [B,Hkv,D] into row positions[b] of k_cache/v_cache
    [B,Hkv,L,D] (bf16, in place)."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _check(t, n, torch.bfloat16, 3)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16, 4)
    _check(positions, "positions", torch.int32, 1)
    B, Hkv, L, D = k_cache.shape
    if tuple(v_cache.shape) != (B, Hkv, L, D) or tuple(k_new.shape) != (B, Hkv, D) \
            or tuple(v_new.shape) != (B, Hkv, D) or positions.shape[0] != B:
        raise ValueError("attn_kv_append: inconsistent shapes")
    code = load_library().attn_kv_append(
        k_new.data_ptr(), v_new.data_ptr(), positions.data_ptr(), k_cache.data_ptr(),
        v_cache.data_ptr(), B, Hkv, L, D, _stream(stream))
    _raise(code, "attn_kv_append")


def attn_decode_workspace_size(B: int, Hq: int, Hkv: int, L: int, D: int) -> int:
    return int(load_library().attn_decode_workspace_size(B, Hq, Hkv, L, D))


def decode_workspace(B: int, Hq: int, Hkv: int, L: int, D: int, device=None) -> torch.Tensor:
    """A zero-filled workspace tensor of the size attn_decode_step needs."""
    n = attn_decode_workspace_size(B, Hq, Hkv, L, D)
    if n == 0:
        raise AttnError(2, "attn_decode_workspace_size")
    ws = torch.zeros(n, dtype=torch.uint8, device=device or "cuda")
    if attn_debug_build():
        _DEBUG_WORKSPACES.append(ws)
    return ws


def debug_collect_range_bits() -> int:
    """Range-checked builds: synchronise, then return ATTN_DEV_RANGE if any
    decode launch since the last call skipped an access (read from every
    workspace decode_workspace() handed out, and from the status reads callers
    made themselves) or if a prefill launch did; clears all of it.  Always 0
    in release builds."""
    global _DEBUG_RANGE_SEEN
    if not attn_debug_build():
        return 0
    bits = _DEBUG_RANGE_SEEN
    for ws in _DEBUG_WORKSPACES:
        bits |= attn_read_device_status(ws)
    _DEBUG_WORKSPACES.clear()
    _DEBUG_RANGE_SEEN = 0
    if attn_read_prefill_skips():
        bits |= ATTN_DEV_RANGE
    return bits & ATTN_DEV_RANGE


def attn_decode_step(q, positions, k_cache, v_cache, scale: float, out=None, workspace=None,
                     stream=None) -> torch.Tensor:
    """out[b,h] = softmax(scale q[b,h].K[b,h//g,0..pos_b]) V[b,h//g,0..pos_b]."""
    _check(q, "q", torch.bfloat16, 3)
    _check(positions, "positions", torch.int32, 1)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16, 4)
    B, Hq, D = q.shape
    Hkv, L = k_cache.shape[1], k_cache.shape[2]
    if tuple(k_cache.shape) != (B, Hkv, L, D) or tuple(v_cache.shape) != (B, Hkv, L, D) \
            or positions.shape[0] != B:
        raise ValueError("attn_decode_step: inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", torch.bfloat16, 3)
        if tuple(out.shape) != (B, Hq, D):
            raise ValueError("attn_decode_step: out has the wrong shape")
    if workspace is None:
        workspace = decode_workspace(B, Hq, Hkv, L, D, device=q.device)
    code = load_library().attn_decode_step(
        q.data_ptr(), positions.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        B, Hq, Hkv, L, D, float(scale), out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _raise(code, "attn_decode_step")
    return out


def _decode_append(name, q, k_new, v_new, rope, positions, k_cache, v_cache, scale, out,
                   workspace, stream) -> torch.Tensor:
    _check(q, "q", torch.bfloat16, 3)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _check(t, n, torch.bfloat16, 3)
    _check(positions, "positions", torch.int32, 1)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16, 4)
    B, Hq, D = q.shape
    Hkv, L = k_cache.shape[1], k_cache.shape[2]
    if tuple(k_cache.shape) != (B, Hkv, L, D) or tuple(v_cache.shape) != (B, Hkv, L, D) \
            or tuple(k_new.shape) != (B, Hkv, D) or tuple(v_new.shape) != (B, Hkv, D) \
            or positions.shape[0] != B:
        raise ValueError(f"{name}: inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", torch.bfloat16, 3)
        if tuple(out.shape) != (B, Hq, D):
            raise ValueError(f"{name}: out has the wrong shape")
    if workspace is None:
        workspace = decode_workspace(B, Hq, Hkv, L, D, device=q.device)
    lib = load_library()
    head = (q.data_ptr(), k_new.data_ptr(), v_new.data_ptr())
    if rope is not None:
        head += tuple(t.data_ptr() if t is not None else None for t in rope)
    code = getattr(lib, name)(
        *head, positions.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), B, Hq, Hkv, L, D,
        float(scale), out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _raise(code, name)
    return out


def attn_decode_step_append(q, k_new, v_new, positions, k_cache, v_cache, scale: float,
                            out=None, workspace=None, stream=None) -> torch.Tensor:
    """attn_kv_append followed by attn_decode_step, in one launch."""
    return _decode_append("attn_decode_step_append", q, k_new, v_new, None, positions, k_cache,
                          v_cache, scale, out, workspace, stream)


def attn_decode_step_rope_append(q, k_new, v_new, cos, sin, positions, k_cache, v_cache,
                                 scale: float, out=None, workspace=None,
                                 stream=None) -> torch.Tensor:
    """attn_decode_step_append with the rotary embedding applied first: q and
    k_new are rotated by row b of ``cos``/``sin`` ([B, D] float32, the
    rotation at positions[b]); the cache receives the rotated key."""
    _check(q, "q", torch.bfloat16, 3)
    for t, n in ((cos, "cos"), (sin, "sin")):
        _check(t, n, torch.float32, 2)
    B, _, D = q.shape
    if tuple(cos.shape) != (B, D) or tuple(sin.shape) != (B, D):
        raise ValueError("attn_decode_step_rope_append: cos and sin must be [B, D]")
    return _decode_append("attn_decode_step_rope_append", q, k_new, v_new, (cos, sin), positions,
                          k_cache, v_cache, scale, out, workspace, stream)


def attn_decode_stream_step(q, k_new, v_new, positions, k_cache, v_cache, scale: float,
                            cos_table=None, sin_table=None, out=None, workspace=None,
                            stream=None) -> torch.Tensor:
    """One streaming step that a CUDA graph can replay unchanged: the fused
    append + decode (after the rotary embedding when ``cos_table``/``sin_table``,
    [L, D] float32 indexed by position, are given), then ``positions += 1`` on
    the device."""
    if (cos_table is None) != (sin_table is None):
        raise ValueError("attn_decode_stream_step: give both cos_table and sin_table, or neither")
    if cos_table is not None:
        L, D = k_cache.shape[2], q.shape[2]
        for t, n in ((cos_table, "cos_table"), (sin_table, "sin_table")):
            _check(t, n, torch.float32, 2)
            if tuple(t.shape) != (L, D):
                raise ValueError(f"attn_decode_stream_step: {n} must be [L, D]")
    return _decode_append("attn_decode_stream_step", q, k_new, v_new, (cos_table, sin_table),
                          positions, k_cache, v_cache, scale, out, workspace, stream)


def attn_decode_step_window(q, positions, k_cache, v_cache, scale: float, window: int,
                            k_new=None, v_new=None, out=None, workspace=None,
                            stream=None) -> torch.Tensor:
    """Decode over the last ``window`` rows up to each position (rows
    max(0, pos - window + 1) .. pos), appending k_new/v_new first if given."""
    _check(q, "q", torch.bfloat16, 3)
    _check(positions, "positions", torch.int32, 1)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16, 4)
    if (k_new is None) != (v_new is None):
        raise ValueError("attn_decode_step_window: give both k_new and v_new, or neither")
    B, Hq, D = q.shape
    Hkv, L = k_cache.shape[1], k_cache.shape[2]
    if tuple(v_cache.shape) != tuple(k_cache.shape) or k_cache.shape[0] != B or \
            k_cache.shape[3] != D or positions.shape[0] != B:
        raise ValueError("attn_decode_step_window: inconsistent shapes")
    if k_new is not None:
        for t, n in ((k_new, "k_new"), (v_new, "v_new")):
            _check(t, n, torch.bfloat16, 3)
            if tuple(t.shape) != (B, Hkv, D):
                raise ValueError(f"attn_decode_step_window: {n} must be [B, Hkv, D]")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", torch.bfloat16, 3)
        if tuple(out.shape) != (B, Hq, D):
            raise ValueError("attn_decode_step_window: out has the wrong shape")
    if workspace is None:
        workspace = decode_workspace(B, Hq, Hkv, L, D, device=q.device)
    ptr = lambda t: t.data_ptr() if t is not None else None
    code = load_library().attn_decode_step_window(
        q.data_ptr(), ptr(k_new), ptr(v_new), positions.data_ptr(), k_cache.data_ptr(),
        v_cache.data_ptr(), B, Hq, Hkv, L, D, int(window), float(scale), out.data_ptr(),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream))
    _raise(code, "attn_decode_step_window")
    return out


def attn_decode_multi(q, positions, k_cache, v_cache, scale: float, k_new=None, v_new=None,
                      out=None, workspace=None, stream=None) -> torch.Tensor:
    """S new tokens per sequence: q [B, S, Hq, D]; token t at positions[b] + t
    attends rows 0 .. positions[b] + t.  k_new/v_new [B, S, Hkv, D], if given,
    are appended first.  Returns out [B, S, Hq, D]."""
    _check(q, "q", torch.bfloat16, 4)
    _check(positions, "positions", torch.int32, 1)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16, 4)
    if (k_new is None) != (v_new is None):
        raise ValueError("attn_decode_multi: give both k_new and v_new, or neither")
    B, S, Hq, D = q.shape
    Hkv, L = k_cache.shape[1], k_cache.shape[2]
    if tuple(v_cache.shape) != tuple(k_cache.shape) or k_cache.shape[0] != B or \
            k_cache.shape[3] != D or positions.shape[0] != B:
        raise ValueError("attn_decode_multi: inconsistent shapes")
    if k_new is not None:
        for t, n in ((k_new, "k_new"), (v_new, "v_new")):
            _check(t, n, torch.bfloat16, 4)
            if tuple(t.shape) != (B, S, Hkv, D):
                raise ValueError(f"attn_decode_multi: {n} must be [B, S, Hkv, D]")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", torch.bfloat16, 4)
        if tuple(out.shape) != (B, S, Hq, D):
            raise ValueError("attn_decode_multi: out has the wrong shape")
    if workspace is None:
        workspace = decode_workspace(B, S * Hq, Hkv, L, D, device=q.device)
    ptr = lambda t: t.data_ptr() if t is not None else None
    code = load_library().attn_decode_multi(
        q.data_ptr(), ptr(k_new), ptr(v_new), positions.data_ptr(), k_cache.data_ptr(),
        v_cache.data_ptr(), B, S, Hq, Hkv, L, D, float(scale), out.data_ptr(),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream))
    _raise(code, "attn_decode_multi")
    return out


def attn_decode_step_noalloc(q, positions, k_cache, v_cache, scale: float, out=None,
                             stream=None) -> torch.Tensor:
    """attn_decode_step using the library's built-in scratch instead of a
    workspace, so the call allocates no device memory."""
    _check(q, "q", torch.bfloat16, 3)
    _check(positions, "positions", torch.int32, 1)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16, 4)
    B, Hq, D = q.shape
    Hkv, L = k_cache.shape[1], k_cache.shape[2]
    if tuple(k_cache.shape) != (B, Hkv, L, D) or tuple(v_cache.shape) != (B, Hkv, L, D) \
            or positions.shape[0] != B:
        raise ValueError("attn_decode_step_noalloc: inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", torch.bfloat16, 3)
        if tuple(out.shape) != (B, Hq, D):
            raise ValueError("attn_decode_step_noalloc: out has the wrong shape")
    code = load_library().attn_decode_step_noalloc(
        q.data_ptr(), positions.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        B, Hq, Hkv, L, D, float(scale), out.data_ptr(), _stream(stream))
    _raise(code, "attn_decode_step_noalloc")
    return out


def attn_prefill_causal(q, k, v, start_pos: int, scale: float, out=None,
                        stream=None) -> torch.Tensor:
    """Causal prefill: q [S,Hq,d] new tokens, k/v [start_pos+S,Hkv,d]."""
    _check(q, "q", torch.bfloat16, 3)
    _check(k, "k", torch.bfloat16, 3)
    _check(v, "v", torch.bfloat16, 3)
    S, Hq, d = q.shape
    T, Hkv = k.shape[0], k.shape[1]
    if T != start_pos + S or tuple(v.shape) != tuple(k.shape) or k.shape[2] != d:
        raise ValueError("attn_prefill_causal: inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out", torch.bfloat16, 3)
    code = load_library().attn_prefill_causal(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), S, int(start_pos), Hq, Hkv, d, float(scale),
        out.data_ptr(), _stream(stream))
    _raise(code, "attn_prefill_causal")
    return out


def attn_test_skip_tile(tile: int) -> None:
    """Failure-path tests only: the next decode launches never issue tile
    ``tile`` of the first segment, so the waits for it run out (-1: off)."""
    _raise(load_library().attn_test_skip_tile(int(tile)), "attn_test_skip_tile")


def attn_test_force_schedule(cluster: int) -> None:
    """Schedule tests only: split every segment by stream-K (0) or in
    clusters of `cluster` CTAs (1..16) from the next decode launch on; -1
    restores the automatic choice."""
    _raise(load_library().attn_test_force_schedule(int(cluster)), "attn_test_force_schedule")


def attn_read_prefill_status(stream=None) -> int:
    """Synchronise, read and clear the count of prefill waits that gave up."""
    n = ctypes.c_uint32(0)
    code = load_library().attn_read_prefill_status(ctypes.byref(n), _stream(stream))
    if code not in (0, 5):
        raise AttnError(code, "attn_read_prefill_status")
    return int(n.value)


def attn_debug_build() -> bool:
    """True if the loaded library has the device range checks."""
    return bool(load_library().attn_debug_build())


def attn_read_prefill_skips(stream=None) -> int:
    """Synchronise, read and clear the count of prefill accesses that failed
    a range check (range-checked builds; always 0 otherwise)."""
    n = ctypes.c_uint32(0)
    code = load_library().attn_read_prefill_skips(ctypes.byref(n), _stream(stream))
    if code not in (0, 5):
        raise AttnError(code, "attn_read_prefill_skips")
    return int(n.value)


def attn_read_device_status(workspace, stream=None) -> int:
    """Synchronise, read and clear the decode workspace's device status bits."""
    global _DEBUG_RANGE_SEEN
    bits = ctypes.c_uint32(0)
    code = load_library().attn_read_device_status(workspace.data_ptr(), ctypes.byref(bits),
                                                  _stream(stream))
    if code not in (0, 5):
        raise AttnError(code, "attn_read_device_status")
    _DEBUG_RANGE_SEEN |= int(bits.value) & ATTN_DEV_RANGE
    return int(bits.value)
