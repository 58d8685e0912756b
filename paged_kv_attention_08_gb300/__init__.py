"""Paged-attention decode for GB300 (sm_103a): thin Python binding.

Every call marshals torch tensors into the C ABI of ``libpa_decode.so``
(declared in ``include/pa_decode.h``) and launches on the current torch CUDA
stream.  Torch supplies device memory and streams only; all arithmetic runs in
the library's CUDA kernels.  There is no fallback: if the library is not built
or a call is rejected, an exception is raised.

    decode(out, q, k_cache, v_cache, block_tables, context_lens, scale)
    decode_splitkv(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                   max_context_len, partition_tokens=0, workspace=None)
    decode_splitkv_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                           max_context_len, partition_tokens=0)
    decode_multi(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                 max_context_len, partition_tokens=0, workspace=None)
    append_kv(k_cache, v_cache, k_new, v_new, block_tables, positions)
    workspace_size(q, k_cache, block_tables, out_dtype, max_context_len, partition_tokens=0)
    workspace_size_multi(q, k_cache, block_tables, out_dtype, max_context_len, partition_tokens=0)
    plan_info(q, k_cache, block_tables, max_context_len, partition_tokens=0)
    choose_partition_tokens(q, k_cache, block_tables, max_context_len, num_sms)
    resolve_blocks(out_phys, block_tables, context_lens, block_size, num_blocks)
    selftest_wait_timeout(timeout_ns)
    device_error()
    set_switch(which, value) / get_switch(which)     (test and tuning switches)

Every launching call also takes ``stream=`` (default: the current torch stream).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["PaError", "decode", "decode_splitkv", "decode_splitkv_noalloc", "decode_multi",
           "append_kv", "workspace_size", "workspace_size_multi", "plan_info", "choose_partition_tokens",
           "resolve_blocks", "selftest_wait_timeout", "device_error", "library_path", "F16",
           "BF16", "F32", "PARTITION_BALANCED", "set_switch", "get_switch", "SWITCH_MULTI_KERNEL",
           "SWITCH_TILE_COMPACT_Q", "KERNEL_AUTO", "KERNEL_MMA", "KERNEL_TILE"]

F16, BF16, F32 = 0, 1, 2
PARTITION_BALANCED = -1   # partition_tokens value requesting the balanced split
SWITCH_MULTI_KERNEL, SWITCH_TILE_COMPACT_Q = 0, 1      # pa_set_switch switches
KERNEL_AUTO, KERNEL_MMA, KERNEL_TILE = 0, 1, 2         # values of SWITCH_MULTI_KERNEL
_STATUS = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_WORKSPACE",
           4: "PA_ERR_CUDA", 5: "PA_ERR_TIMEOUT"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libpa_decode.so")
_lock = threading.Lock()
_lib = None


class PaError(RuntimeError):
    """A non-OK pa_status returned by the library."""

    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {_STATUS.get(code, code)}")


class _Shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("num_blocks", ctypes.c_int64), ("kv_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32)]


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it with "
                    "`python -m paged_kv_attention_08_gb300.build` (there is no fallback path)")
            lib = ctypes.CDLL(_LIB_PATH)
            P, S = ctypes.c_void_p, ctypes.POINTER(_Shape)
            i32, f32, sz = ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
            lib.pa_decode.argtypes = [P, P, P, P, P, P, S, f32, P]
            lib.pa_decode.restype = ctypes.c_int
            lib.pa_decode_splitkv.argtypes = [P, P, P, P, P, P, S, f32, i32, i32, P, sz, P]
            lib.pa_decode_splitkv.restype = ctypes.c_int
            lib.pa_decode_splitkv_noalloc.argtypes = [P, P, P, P, P, P, S, f32, i32, i32, P]
            lib.pa_decode_splitkv_noalloc.restype = ctypes.c_int
            lib.pa_decode_multi.argtypes = [P, P, P, P, P, P, S, i32, f32, i32, i32, P, sz, P]
            lib.pa_decode_multi.restype = ctypes.c_int
            lib.pa_plan_info.argtypes = [S, i32, i32, i32, P]
            lib.pa_plan_info.restype = ctypes.c_int
            lib.pa_workspace_size_multi.argtypes = [S, i32, i32, i32]
            lib.pa_workspace_size_multi.restype = sz
            lib.pa_workspace_size.argtypes = [S, i32, i32]
            lib.pa_workspace_size.restype = sz
            lib.pa_choose_partition_tokens.argtypes = [S, i32, i32]
            lib.pa_choose_partition_tokens.restype = i32
            lib.pa_resolve_blocks.argtypes = [P, P, P, S, P]
            lib.pa_resolve_blocks.restype = ctypes.c_int
            lib.pa_append_kv.argtypes = [P, P, P, P, P, P, S, P]
            lib.pa_append_kv.restype = ctypes.c_int
            lib.pa_selftest_wait_timeout.argtypes = [ctypes.c_uint64, P]
            lib.pa_selftest_wait_timeout.restype = ctypes.c_int
            lib.pa_device_error.argtypes = [ctypes.POINTER(i32), P]
            lib.pa_device_error.restype = ctypes.c_int
            lib.pa_set_switch.argtypes = [i32, i32]
            lib.pa_set_switch.restype = ctypes.c_int
            lib.pa_get_switch.argtypes = [i32]
            lib.pa_get_switch.restype = i32
            lib.pa_status_string.argtypes = [ctypes.c_int]
            lib.pa_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float16:
        return F16
    if dt == torch.bfloat16:
        return BF16
    if dt == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {dt}")


def make_shape(q: torch.Tensor, k_cache: torch.Tensor, block_tables: torch.Tensor,
               out_dtype: torch.dtype | None = None) -> _Shape:
    """pa_shape from tensor shapes: q [B,H,D], k_cache [NB,bs,Hkv,D], block_tables [B,max_blocks]."""
    if q.dim() != 3 or k_cache.dim() != 4 or block_tables.dim() != 2:
        raise ValueError("expected q [B,H,D], k_cache [NB,bs,Hkv,D], block_tables [B,max_blocks]")
    B, H, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    return _Shape(B, H, Hkv, D, bs, block_tables.shape[1], NB, _dtype_code(k_cache.dtype),
                  _dtype_code(out_dtype if out_dtype is not None else q.dtype))


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(code: int, what: str):
    if code != 0:
        raise PaError(code, what)


def _dev_tensors(*ts):
    dev = None
    for t in ts:
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors")
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("all tensors must be on one device")


def _ints(block_tables, context_lens):
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")


def _check_args(out, q, k_cache, v_cache, block_tables, context_lens, multi=False):
    """Shapes and dtypes that the library takes on trust: it reads the problem
    shape from q, k_cache and block_tables alone, so a v_cache, out, table or
    length tensor of another shape or dtype would be read or written past its
    memory.  Raises ValueError / TypeError before anything reaches the device."""
    if q.dim() != (4 if multi else 3):
        raise ValueError("q must be [batch, q_len, num_heads, head_dim]" if multi
                         else "q must be [batch, num_heads, head_dim]")
    if k_cache.dim() != 4:
        raise ValueError("k_cache must be [num_blocks, block_size, num_kv_heads, head_dim]")
    if tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError(f"v_cache {tuple(v_cache.shape)} must be shaped like k_cache "
                         f"{tuple(k_cache.shape)}")
    if v_cache.dtype != k_cache.dtype:
        raise TypeError("v_cache must have k_cache's dtype")
    if q.dtype != k_cache.dtype:
        raise TypeError("q must have the cache's dtype")
    if q.shape[-1] != k_cache.shape[3]:
        raise ValueError(f"q's head_dim {q.shape[-1]} differs from the cache's {k_cache.shape[3]}")
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError(f"out {tuple(out.shape)} must be shaped like q {tuple(q.shape)}")
    if out.dtype not in (torch.float32, q.dtype):
        raise TypeError("out must be float32 or q's dtype")
    if block_tables.dim() != 2 or block_tables.shape[0] != q.shape[0]:
        raise ValueError("block_tables must be [batch, max_blocks_per_seq]")
    if context_lens.dim() != 1 or context_lens.numel() != q.shape[0]:
        raise ValueError("context_lens must be [batch]")
    _ints(block_tables, context_lens)


def decode(out, q, k_cache, v_cache, block_tables, context_lens, scale: float, stream=None):
    """Single-pass paged decode into ``out`` ([B,H,D], fp32 or q's dtype)."""
    _check_args(out, q, k_cache, v_cache, block_tables, context_lens)
    _dev_tensors(out, q, k_cache, v_cache, block_tables, context_lens)
    shape = make_shape(q, k_cache, block_tables, out.dtype)
    _check(_load().pa_decode(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                             block_tables.data_ptr(), context_lens.data_ptr(),
                             ctypes.byref(shape), float(scale), _stream_ptr(stream)), "pa_decode")
    return out


def workspace_size(q, k_cache, block_tables, out_dtype, max_context_len: int,
                   partition_tokens: int = 0) -> int:
    shape = make_shape(q, k_cache, block_tables, out_dtype)
    return int(_load().pa_workspace_size(ctypes.byref(shape), int(max_context_len),
                                         int(partition_tokens)))


def choose_partition_tokens(q, k_cache, block_tables, max_context_len: int, num_sms: int) -> int:
    shape = make_shape(q, k_cache, block_tables, None)
    return int(_load().pa_choose_partition_tokens(ctypes.byref(shape), int(max_context_len),
                                                  int(num_sms)))


def decode_splitkv(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                   max_context_len: int, partition_tokens: int = 0, workspace=None, stream=None):
    """Flash-Decoding split-KV decode.  ``workspace`` is a CUDA byte tensor of at
    least ``workspace_size(...)`` bytes; when omitted one is taken from torch's
    allocator for this call."""
    _check_args(out, q, k_cache, v_cache, block_tables, context_lens)
    _dev_tensors(out, q, k_cache, v_cache, block_tables, context_lens)
    shape = make_shape(q, k_cache, block_tables, out.dtype)
    lib = _load()
    if workspace is None:
        need = lib.pa_workspace_size(ctypes.byref(shape), int(max_context_len), int(partition_tokens))
        workspace = torch.empty(max(int(need), 16), dtype=torch.uint8, device=q.device)
    else:
        _dev_tensors(workspace)
    _check(lib.pa_decode_splitkv(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(),
                                 v_cache.data_ptr(), block_tables.data_ptr(),
                                 context_lens.data_ptr(), ctypes.byref(shape), float(scale),
                                 int(max_context_len), int(partition_tokens),
                                 workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                 _stream_ptr(stream)), "pa_decode_splitkv")
    return out


def decode_splitkv_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                           max_context_len: int, partition_tokens: int = 0, stream=None):
    """Split-KV decode whose partials live in the library's fixed 16 MiB
    scratch instead of a caller workspace, for callers that cannot allocate
    device memory.  Calls that may overlap on the GPU race on that scratch;
    the first call on a device should come before any stream capture.
    Raises PaError (PA_ERR_WORKSPACE) when the partials would not fit."""
    _check_args(out, q, k_cache, v_cache, block_tables, context_lens)
    _dev_tensors(out, q, k_cache, v_cache, block_tables, context_lens)
    shape = make_shape(q, k_cache, block_tables, out.dtype)
    _check(_load().pa_decode_splitkv_noalloc(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_tables.data_ptr(), context_lens.data_ptr(), ctypes.byref(shape), float(scale),
        int(max_context_len), int(partition_tokens), _stream_ptr(stream)),
        "pa_decode_splitkv_noalloc")
    return out


def _multi_shape(q, k_cache, block_tables, out_dtype):
    if q.dim() != 4:
        raise ValueError("q must be [batch, q_len, num_heads, head_dim]")
    return make_shape(q[:, 0], k_cache, block_tables, out_dtype), int(q.shape[1])


class _PlanDesc(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("partitions", ctypes.c_int32),
                ("partition_tokens", ctypes.c_int32), ("reduce", ctypes.c_int32),
                ("ctas", ctypes.c_int32), ("threads", ctypes.c_int32)]


_KERNELS = {0: "mma.sync m16n8k16", 1: "tcgen05 tile"}
_REDUCE = {0: "none", 1: "cluster DSMEM", 2: "workspace+combine kernel", 3: "balanced split"}


def plan_info(q, k_cache, block_tables, max_context_len: int, partition_tokens: int = 0,
              out_dtype=None) -> dict:
    """The plan a split-KV call with these arguments uses on the current device
    (q [B, H, D] for one query token, [B, Q, H, D] for several)."""
    if q.dim() == 4:
        shape, q_len = _multi_shape(q, k_cache, block_tables, out_dtype or torch.float32)
    else:
        shape, q_len = make_shape(q, k_cache, block_tables, out_dtype or torch.float32), 1
    d = _PlanDesc()
    _check(_load().pa_plan_info(ctypes.byref(shape), q_len, int(max_context_len),
                                int(partition_tokens), ctypes.byref(d)), "pa_plan_info")
    return {"kernel": _KERNELS[d.kernel], "partitions": d.partitions,
            "partition_tokens": d.partition_tokens, "reduce": _REDUCE[d.reduce],
            "ctas": d.ctas, "threads": d.threads}


def workspace_size_multi(q, k_cache, block_tables, out_dtype, max_context_len: int,
                         partition_tokens: int = 0) -> int:
    shape, q_len = _multi_shape(q, k_cache, block_tables, out_dtype)
    return int(_load().pa_workspace_size_multi(ctypes.byref(shape), q_len, int(max_context_len),
                                               int(partition_tokens)))


def decode_multi(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                 max_context_len: int, partition_tokens: int = 0, workspace=None, stream=None):
    """Several query tokens per sequence (q, out: [B, Q, H, D]); query token i
    of sequence b attends causally to the cached tokens t <= context_lens[b] - Q + i."""
    _check_args(out, q, k_cache, v_cache, block_tables, context_lens, multi=True)
    _dev_tensors(out, q, k_cache, v_cache, block_tables, context_lens)
    shape, q_len = _multi_shape(q, k_cache, block_tables, out.dtype)
    lib = _load()
    if workspace is None:
        need = lib.pa_workspace_size_multi(ctypes.byref(shape), q_len, int(max_context_len),
                                           int(partition_tokens))
        workspace = torch.empty(max(int(need), 16), dtype=torch.uint8, device=q.device)
    else:
        _dev_tensors(workspace)
    _check(lib.pa_decode_multi(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(),
                               v_cache.data_ptr(), block_tables.data_ptr(),
                               context_lens.data_ptr(), ctypes.byref(shape), q_len, float(scale),
                               int(max_context_len), int(partition_tokens), workspace.data_ptr(),
                               workspace.numel() * workspace.element_size(), _stream_ptr(stream)),
           "pa_decode_multi")
    return out


def append_kv(k_cache, v_cache, k_new, v_new, block_tables, positions, stream=None):
    """Write each sequence's new token ([B, Hkv, D] k_new / v_new) into its
    cache slot at ``positions[b]``; negative positions and masked entries
    write nothing."""
    if k_cache.dim() != 4 or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache must both be [num_blocks, block_size, "
                         "num_kv_heads, head_dim]")
    if v_cache.dtype != k_cache.dtype or k_new.dtype != k_cache.dtype or v_new.dtype != k_cache.dtype:
        raise TypeError("new keys/values and both caches must have one dtype")
    if block_tables.dim() != 2 or positions.dim() != 1 or positions.numel() != block_tables.shape[0]:
        raise ValueError("block_tables must be [batch, max_blocks_per_seq], positions [batch]")
    _ints(block_tables, positions)
    B = block_tables.shape[0]
    NB, bs, Hkv, D = k_cache.shape
    if tuple(k_new.shape) != (B, Hkv, D) or tuple(v_new.shape) != (B, Hkv, D):
        raise ValueError("k_new/v_new must be [batch, num_kv_heads, head_dim]")
    _dev_tensors(k_cache, v_cache, k_new, v_new, block_tables, positions)
    shape = _Shape(B, Hkv, Hkv, D, bs, block_tables.shape[1], NB, _dtype_code(k_cache.dtype), F32)
    _check(_load().pa_append_kv(k_cache.data_ptr(), v_cache.data_ptr(), k_new.data_ptr(),
                                v_new.data_ptr(), block_tables.data_ptr(), positions.data_ptr(),
                                ctypes.byref(shape), _stream_ptr(stream)), "pa_append_kv")


def resolve_blocks(out_phys, block_tables, context_lens, block_size: int, num_blocks: int,
                   stream=None):
    """Physical block the kernels read for each (sequence, logical page); -1 if none."""
    if out_phys.dtype != torch.int32 or out_phys.shape != block_tables.shape:
        raise ValueError("out_phys must be int32 shaped like block_tables")
    if block_tables.dim() != 2 or context_lens.dim() != 1 or \
            context_lens.numel() != block_tables.shape[0]:
        raise ValueError("block_tables must be [batch, max_blocks_per_seq], context_lens [batch]")
    _ints(block_tables, context_lens)
    _dev_tensors(out_phys, block_tables, context_lens)
    B, mb = block_tables.shape
    shape = _Shape(B, 1, 1, 64, int(block_size), mb, int(num_blocks), F16, F32)
    _check(_load().pa_resolve_blocks(out_phys.data_ptr(), block_tables.data_ptr(),
                                     context_lens.data_ptr(), ctypes.byref(shape),
                                     _stream_ptr(stream)), "pa_resolve_blocks")
    return out_phys


def selftest_wait_timeout(timeout_ns: int, stream=None):
    """Run the bounded-wait self-test kernel (it records PA_ERR_TIMEOUT)."""
    _check(_load().pa_selftest_wait_timeout(int(timeout_ns), _stream_ptr(stream)),
           "pa_selftest_wait_timeout")


def device_error(stream=None) -> int:
    """Read and clear the device error word (synchronises the stream)."""
    code = ctypes.c_int32(0)
    _check(_load().pa_device_error(ctypes.byref(code), _stream_ptr(stream)), "pa_device_error")
    return int(code.value)


def set_switch(which: int, value: int):
    """Set a test / tuning switch (SWITCH_MULTI_KERNEL: KERNEL_AUTO, KERNEL_MMA or
    KERNEL_TILE; SWITCH_TILE_COMPACT_Q: 1 or 0) for every later call."""
    _check(_load().pa_set_switch(int(which), int(value)), "pa_set_switch")


def get_switch(which: int) -> int:
    return int(_load().pa_get_switch(int(which)))
