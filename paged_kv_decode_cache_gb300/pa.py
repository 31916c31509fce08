"""Thin ctypes binding of libpagedattn (include/pa.h), same entry-point names.

Argument marshalling only: every function checks dtypes, shapes and
contiguity of the torch tensors it is given, passes their device pointers to
the C entry point of the same name, and raises ``PAError`` on a negative
return code.  All compute happens in the CUDA kernels; there is no fallback.
Outputs are caller-allocated, as in the C ABI.  Work is enqueued on
``stream`` (default: torch's current stream) and nothing synchronises.
"""
from __future__ import annotations

import ctypes
import functools
import itertools
import os
import re
import threading
from typing import Optional

import torch

from . import build as _build

PA_OK, PA_EINVAL, PA_EUNSUPPORTED, PA_EWORKSPACE, PA_ECUDA = 0, -1, -2, -3, -4
PA_STATUS_BAD_BLOCK, PA_STATUS_BAD_SLOT, PA_STATUS_BAD_SEQLEN, PA_STATUS_TIMEOUT = 1, 2, 4, 8
PA_OPT_DECODE_KERNEL, PA_OPT_SPLIT_MERGE, PA_OPT_PDL, PA_OPT_CASCADE = 0, 1, 2, 3
PA_CASCADE_AUTO, PA_CASCADE_ALWAYS, PA_CASCADE_NEVER = 0, 1, 2
PA_KERNEL_AUTO, PA_KERNEL_CUDA_CORE, PA_KERNEL_TENSOR_CORE = 0, 1, 2
PA_MERGE_AUTO, PA_MERGE_GRID = 0, 1

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pa.h")


class PAError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn}: {msg} (code {code})")
        self.code = code


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None

_P, _I32, _I64, _F32, _SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                             ctypes.c_size_t)
_SIGNATURES = {
    "pa_cache_write": ([_P, _P, _P, _I64, _P, _P, CacheDesc, _P, _P], ctypes.c_int),
    "pa_decode": ([_P, _P, _P, _P, _P, CacheDesc, _P, _I32, _P, _I32, _I32, _F32, _P, _P],
                  ctypes.c_int),
    "pa_choose_num_splits": ([_I32, _I32, _I32, _I32, _I32, _I32, _I32], ctypes.c_int),
    "pa_partition_tokens": ([_I32, _I32, _I32], ctypes.c_int),
    "pa_splitkv_workspace_bytes": ([_I32, _I32, _I32, _I32], _SZ),
    "pa_decode_partial": ([_P, _P, _P, _P, _P, CacheDesc, _P, _I32, _P, _I32, _I32, _F32, _I32,
                           _P, _P], ctypes.c_int),
    "pa_combine": ([_P, _P, _P, _P, _I32, _I32, _I32, _I32, _P], ctypes.c_int),
    "pa_decode_splitkv": ([_P, _P, _P, _P, _P, CacheDesc, _P, _I32, _P, _I32, _I32, _F32, _I32,
                           _P, _SZ, _P, _P], ctypes.c_int),
    "pa_decode_step": ([_P, _P, _P, _P, _P, _P, _P, _P, CacheDesc, _P, _I32, _P, _I32, _I32, _F32,
                        _I32, _P, _SZ, _P, _P], ctypes.c_int),
    "pa_decode_splitkv_noalloc": ([_P, _P, _P, _P, _P, CacheDesc, _P, _I32, _P, _I32, _I32, _F32,
                                   _I32, _P, _P], ctypes.c_int),
    "pa_auto_num_splits": ([_I32, _I32, _I32, _I32, _I32, _I32], ctypes.c_int),
    "pa_decode_mq": ([_P, _P, _P, _I32, _P, _P, CacheDesc, _P, _I32, _P, _I32, _I32, _F32, _I32,
                      _P, _SZ, _P, _P], ctypes.c_int),
    "pa_choose_num_splits_mq": ([_I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32], ctypes.c_int),
    "pa_decode_launches": ([_I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32], ctypes.c_int),
    "pa_decode_cascade": ([_P, _P, _P, _P, _P, CacheDesc, _I32, _P, _I32, _P, _I32, _I32, _F32, _P,
                           _SZ, _P, _P], ctypes.c_int),
    "pa_cascade_workspace_bytes": ([_I32, _I32, _I32, _I32, _I32, _I32, _I32], _SZ),
    "pa_cascade_pays": ([_I32, _I32, _I32, _I32, _I32], ctypes.c_int),
    "pa_cascade_launches": ([_I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32], ctypes.c_int),
    "pa_cache_write_fp8": ([_P, _P, _P, _I64, _P, _P, CacheDesc, _F32, _F32, _P, _P], ctypes.c_int),
    "pa_decode_splitkv_fp8": ([_P, _P, _P, _P, _P, CacheDesc, _F32, _F32, _P, _I32, _P, _I32, _I32,
                               _F32, _I32, _P, _SZ, _P, _P], ctypes.c_int),
    "pa_decode_step_fp8": ([_P, _P, _P, _P, _P, _P, _P, _P, CacheDesc, _F32, _F32, _P, _I32, _P, _I32,
                            _I32, _F32, _I32, _P, _SZ, _P, _P], ctypes.c_int),
    "pa_set_option": ([_I32, _I32], ctypes.c_int),
    "pa_get_option": ([_I32], ctypes.c_int),
    "pa_strerror": ([ctypes.c_int], ctypes.c_char_p),
    "pa_version": ([], ctypes.c_int),
}


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libpagedattn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with paged_kv_decode_cache_gb300.build.build() "
                    "(needs nvcc); there is no CPU fallback")
            L = ctypes.CDLL(path)
            for name, (args, res) in _SIGNATURES.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def header_functions(path: str = HEADER) -> list[str]:
    """Names of the functions include/pa.h declares."""
    with open(path) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def _check(name: str, rc: int):
    if rc != PA_OK:
        raise PAError(name, rc, pa_strerror(rc))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _one_cuda_device(devices, fn: str) -> Optional[torch.device]:
    """The one CUDA device among `devices` (None when there is none: the
    per-tensor checks then reject the call); several raise ValueError."""
    cuda = {d for d in devices if d.type == "cuda"}
    if len(cuda) > 1:
        raise ValueError(f"{fn}: tensors on several devices ({', '.join(sorted(map(str, cuda)))})")
    return next(iter(cuda)) if cuda else None


def _on_tensors_device(fn):
    """Run a wrapper on the device its tensors live on (and that device's
    current stream when none is given): the C library launches on the current
    device.  A call whose device is already current runs unchanged."""
    @functools.wraps(fn)
    def call(*args, **kwargs):
        dev = _one_cuda_device([a.device for a in itertools.chain(args, kwargs.values())
                                if isinstance(a, torch.Tensor)], fn.__name__)
        stream = kwargs.get("stream")
        if dev is not None and stream is not None and stream.device != dev:
            raise ValueError(f"{fn.__name__}: stream on {stream.device}, tensors on {dev}")
        if dev is None or dev.index == torch.cuda.current_device():
            return fn(*args, **kwargs)
        with torch.cuda.device(dev):
            return fn(*args, **kwargs)
    return call


def cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    nb, bs, hkv, d = k_cache.shape
    return CacheDesc(nb, bs, hkv, d)


def pa_strerror(code: int) -> str:
    return lib().pa_strerror(code).decode()


def pa_version() -> int:
    return lib().pa_version()


def pa_set_option(option: int, value: int) -> None:
    """Set a process-wide switch (PA_OPT_*): raises PAError on an unknown switch or value."""
    _check("pa_set_option", lib().pa_set_option(option, value))


def pa_get_option(option: int) -> int:
    v = lib().pa_get_option(option)
    if v < 0:
        _check("pa_get_option", v)
    return v


def pa_choose_num_splits(B: int, Hq: int, Hkv: int, D: int, max_blocks_per_seq: int,
                         block_size: int, sm_count: int) -> int:
    r = lib().pa_choose_num_splits(B, Hq, Hkv, D, max_blocks_per_seq, block_size, sm_count)
    _check("pa_choose_num_splits", min(r, 0))
    return r


def pa_choose_num_splits_mq(B: int, q_len: int, Hq: int, Hkv: int, D: int,
                            max_blocks_per_seq: int, block_size: int, sm_count: int) -> int:
    r = lib().pa_choose_num_splits_mq(B, q_len, Hq, Hkv, D, max_blocks_per_seq, block_size,
                                      sm_count)
    _check("pa_choose_num_splits_mq", min(r, 0))
    return r


def pa_decode_launches(B: int, q_len: int, Hq: int, Hkv: int, D: int, max_blocks_per_seq: int,
                       block_size: int, num_splits: int, sm_count: int) -> int:
    r = lib().pa_decode_launches(B, q_len, Hq, Hkv, D, max_blocks_per_seq, block_size, num_splits,
                                 sm_count)
    _check("pa_decode_launches", min(r, 0))
    return r


def pa_partition_tokens(max_blocks_per_seq: int, block_size: int, num_splits: int) -> int:
    r = lib().pa_partition_tokens(max_blocks_per_seq, block_size, num_splits)
    _check("pa_partition_tokens", min(r, 0))
    return r


def pa_splitkv_workspace_bytes(B: int, Hq: int, D: int, num_splits: int) -> int:
    return int(lib().pa_splitkv_workspace_bytes(B, Hq, D, num_splits))


def pa_auto_num_splits(B: int, Hq: int, Hkv: int, D: int, max_blocks_per_seq: int,
                       block_size: int) -> int:
    r = lib().pa_auto_num_splits(B, Hq, Hkv, D, max_blocks_per_seq, block_size)
    _check("pa_auto_num_splits", min(r, 0))
    return r


@_on_tensors_device
def pa_cache_write(k_new, v_new, slot_mapping, k_cache, v_cache, status=None, stream=None):
    _need(k_new, "k_new", torch.bfloat16, 3)
    _need(v_new, "v_new", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    if v_cache.shape != k_cache.shape or v_new.shape != k_new.shape:
        raise ValueError("K/V shape mismatch")
    if k_new.shape[0] != slot_mapping.shape[0] or tuple(k_new.shape[1:]) != tuple(k_cache.shape[2:]):
        raise ValueError("k_new must be [N, Hkv, D] matching the pool")
    rc = lib().pa_cache_write(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), slot_mapping.shape[0],
                              _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache), _ptr(status),
                              _stream(stream))
    _check("pa_cache_write", rc)


def _decode_inputs(q, k_cache, v_cache, block_tables, seq_lens):
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache differ in shape")
    B, Hq, D = q.shape
    if k_cache.shape[3] != D or block_tables.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("inconsistent q / cache / table shapes")
    return B, Hq, D


@_on_tensors_device
def pa_decode(out, lse, q, k_cache, v_cache, block_tables, seq_lens, scale, status=None,
              stream=None):
    B, Hq, D = _decode_inputs(q, k_cache, v_cache, block_tables, seq_lens)
    _need(out, "out", torch.bfloat16, 3)
    if tuple(out.shape) != (B, Hq, D):
        raise ValueError("out must be [B, Hq, D]")
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    rc = lib().pa_decode(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                         cache_desc(k_cache), _ptr(block_tables), block_tables.shape[1],
                         _ptr(seq_lens), B, Hq, float(scale), _ptr(status), _stream(stream))
    _check("pa_decode", rc)


@_on_tensors_device
def pa_decode_partial(part_o, part_lse, q, k_cache, v_cache, block_tables, seq_lens, scale,
                      num_splits, status=None, stream=None):
    B, Hq, D = _decode_inputs(q, k_cache, v_cache, block_tables, seq_lens)
    _need(part_o, "part_o", torch.float32, 4)
    _need(part_lse, "part_lse", torch.float32, 3)
    if tuple(part_o.shape) != (B, Hq, num_splits, D) or tuple(part_lse.shape) != (B, Hq, num_splits):
        raise ValueError("partials must be [B, Hq, P, D] and [B, Hq, P]")
    rc = lib().pa_decode_partial(_ptr(part_o), _ptr(part_lse), _ptr(q), _ptr(k_cache),
                                 _ptr(v_cache), cache_desc(k_cache), _ptr(block_tables),
                                 block_tables.shape[1], _ptr(seq_lens), B, Hq, float(scale),
                                 num_splits, _ptr(status), _stream(stream))
    _check("pa_decode_partial", rc)


@_on_tensors_device
def pa_combine(out, lse, part_o, part_lse, stream=None):
    _need(part_o, "part_o", torch.float32, 4)
    _need(part_lse, "part_lse", torch.float32, 3)
    _need(out, "out", torch.bfloat16, 3)
    B, Hq, P, D = part_o.shape
    if tuple(out.shape) != (B, Hq, D) or tuple(part_lse.shape) != (B, Hq, P):
        raise ValueError("inconsistent combine shapes")
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    rc = lib().pa_combine(_ptr(out), _ptr(lse), _ptr(part_o), _ptr(part_lse), B, Hq, P, D,
                          _stream(stream))
    _check("pa_combine", rc)


@_on_tensors_device
def pa_decode_splitkv(out, lse, q, k_cache, v_cache, block_tables, seq_lens, scale,
                      num_splits=0, workspace=None, status=None, stream=None):
    B, Hq, D = _decode_inputs(q, k_cache, v_cache, block_tables, seq_lens)
    _need(out, "out", torch.bfloat16, 3)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    ws_bytes = 0
    if workspace is not None:
        if not (workspace.is_cuda and workspace.is_contiguous()):
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_bytes = workspace.numel() * workspace.element_size()
    rc = lib().pa_decode_splitkv(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                 cache_desc(k_cache), _ptr(block_tables), block_tables.shape[1],
                                 _ptr(seq_lens), B, Hq, float(scale), num_splits,
                                 _ptr(workspace), ws_bytes, _ptr(status), _stream(stream))
    _check("pa_decode_splitkv", rc)


@_on_tensors_device
def pa_decode_step(out, lse, q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                   seq_lens, scale, num_splits=0, workspace=None, status=None, stream=None):
    """Fused step: write this step's new K/V through slot_mapping and run split-KV decode."""
    B, Hq, D = _decode_inputs(q, k_cache, v_cache, block_tables, seq_lens)
    _need(out, "out", torch.bfloat16, 3)
    _need(k_new, "k_new", torch.bfloat16, 3)
    _need(v_new, "v_new", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    if tuple(k_new.shape) != (B, k_cache.shape[2], D) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [B, Hkv, D]")
    if slot_mapping.shape[0] != B:
        raise ValueError("slot_mapping must be [B]")
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    ws_bytes = 0
    if workspace is not None:
        if not (workspace.is_cuda and workspace.is_contiguous()):
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_bytes = workspace.numel() * workspace.element_size()
    rc = lib().pa_decode_step(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_new), _ptr(v_new),
                              _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache),
                              _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B, Hq,
                              float(scale), num_splits, _ptr(workspace), ws_bytes, _ptr(status),
                              _stream(stream))
    _check("pa_decode_step", rc)


PA_NOALLOC_SCRATCH_BYTES = 4 << 20


@_on_tensors_device
def pa_decode_mq(out, lse, q, k_cache, v_cache, block_tables, seq_lens, scale, num_splits=0,
                 workspace=None, status=None, stream=None):
    """Causal multi-query decode: q and out are [B, q_len, Hq, D], lse [B, q_len, Hq]."""
    _need(q, "q", torch.bfloat16, 4)
    B, q_len, Hq, D = q.shape
    _decode_inputs(q.view(B, q_len * Hq, D), k_cache, v_cache, block_tables, seq_lens)
    _need(out, "out", torch.bfloat16, 4)
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError("out must be [B, q_len, Hq, D]")
    if lse is not None:
        _need(lse, "lse", torch.float32, 3)
    ws_bytes = 0
    if workspace is not None:
        if not (workspace.is_cuda and workspace.is_contiguous()):
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_bytes = workspace.numel() * workspace.element_size()
    rc = lib().pa_decode_mq(_ptr(out), _ptr(lse), _ptr(q), q_len, _ptr(k_cache), _ptr(v_cache),
                            cache_desc(k_cache), _ptr(block_tables), block_tables.shape[1],
                            _ptr(seq_lens), B, Hq, float(scale), num_splits, _ptr(workspace),
                            ws_bytes, _ptr(status), _stream(stream))
    _check("pa_decode_mq", rc)


def pa_cascade_workspace_bytes(B: int, Hq: int, Hkv: int, D: int, n_prefix_blocks: int,
                               max_blocks_per_seq: int, block_size: int) -> int:
    return int(lib().pa_cascade_workspace_bytes(B, Hq, Hkv, D, n_prefix_blocks, max_blocks_per_seq,
                                                block_size))


def pa_cascade_launches(B: int, Hq: int, Hkv: int, D: int, n_prefix_blocks: int,
                        max_blocks_per_seq: int, block_size: int, sm_count: int) -> int:
    r = lib().pa_cascade_launches(B, Hq, Hkv, D, n_prefix_blocks, max_blocks_per_seq, block_size,
                                  sm_count)
    _check("pa_cascade_launches", min(r, 0))
    return r


def pa_cascade_pays(B: int, Hkv: int, D: int, n_prefix_blocks: int, block_size: int) -> bool:
    """Whether pa_decode_cascade runs the cascade (True) or plain split decode."""
    r = lib().pa_cascade_pays(B, Hkv, D, n_prefix_blocks, block_size)
    _check("pa_cascade_pays", min(r, 0))
    return r == 1


@_on_tensors_device
def pa_decode_cascade(out, lse, q, k_cache, v_cache, n_prefix_blocks, block_tables, seq_lens, scale,
                      workspace=None, status=None, stream=None):
    """Decode with the first n_prefix_blocks table entries shared by every sequence:
    the prefix is attended once for the whole batch, then each suffix, then merged."""
    B, Hq, D = _decode_inputs(q, k_cache, v_cache, block_tables, seq_lens)
    _need(out, "out", torch.bfloat16, 3)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    ws_bytes = 0
    if workspace is not None:
        if not (workspace.is_cuda and workspace.is_contiguous()):
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_bytes = workspace.numel() * workspace.element_size()
    rc = lib().pa_decode_cascade(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                 cache_desc(k_cache), n_prefix_blocks, _ptr(block_tables),
                                 block_tables.shape[1], _ptr(seq_lens), B, Hq, float(scale),
                                 _ptr(workspace), ws_bytes, _ptr(status), _stream(stream))
    _check("pa_decode_cascade", rc)


def _need_pool8(t, name):
    _need(t, name, torch.uint8, 4)


@_on_tensors_device
def pa_cache_write_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                       status=None, stream=None):
    """Quantising slot-mapping write into uint8 e4m3 pools [num_blocks, bs, Hkv, D]."""
    _need(k_new, "k_new", torch.bfloat16, 3)
    _need(v_new, "v_new", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need_pool8(k_cache, "k_cache")
    _need_pool8(v_cache, "v_cache")
    if v_cache.shape != k_cache.shape or v_new.shape != k_new.shape:
        raise ValueError("K/V shape mismatch")
    if k_new.shape[0] != slot_mapping.shape[0] or tuple(k_new.shape[1:]) != tuple(k_cache.shape[2:]):
        raise ValueError("k_new must be [N, Hkv, D] matching the pool")
    rc = lib().pa_cache_write_fp8(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), k_new.shape[0],
                                  _ptr(k_cache), _ptr(v_cache), cache_desc(k_cache),
                                  float(k_scale), float(v_scale), _ptr(status), _stream(stream))
    _check("pa_cache_write_fp8", rc)


@_on_tensors_device
def pa_decode_splitkv_fp8(out, lse, q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens,
                          scale, num_splits=0, workspace=None, status=None, stream=None):
    """Split-KV decode over uint8 e4m3 pools with per-pool scales."""
    _need(q, "q", torch.bfloat16, 3)
    _need_pool8(k_cache, "k_cache")
    _need_pool8(v_cache, "v_cache")
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, Hq, D = q.shape
    if v_cache.shape != k_cache.shape or k_cache.shape[3] != D or block_tables.shape[0] != B:
        raise ValueError("inconsistent q / cache / table shapes")
    _need(out, "out", torch.bfloat16, 3)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    ws_bytes = 0
    if workspace is not None:
        if not (workspace.is_cuda and workspace.is_contiguous()):
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_bytes = workspace.numel() * workspace.element_size()
    rc = lib().pa_decode_splitkv_fp8(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                     cache_desc(k_cache), float(k_scale), float(v_scale),
                                     _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B,
                                     Hq, float(scale), num_splits, _ptr(workspace), ws_bytes,
                                     _ptr(status), _stream(stream))
    _check("pa_decode_splitkv_fp8", rc)


@_on_tensors_device
def pa_decode_step_fp8(out, lse, q, k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                       block_tables, seq_lens, scale, num_splits=0, workspace=None, status=None,
                       stream=None):
    """Fused step over uint8 e4m3 pools: quantise and write this step's new K/V
    through slot_mapping, then split-KV decode."""
    _need(q, "q", torch.bfloat16, 3)
    _need_pool8(k_cache, "k_cache")
    _need_pool8(v_cache, "v_cache")
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, Hq, D = q.shape
    if v_cache.shape != k_cache.shape or k_cache.shape[3] != D or block_tables.shape[0] != B:
        raise ValueError("inconsistent q / cache / table shapes")
    _need(out, "out", torch.bfloat16, 3)
    _need(k_new, "k_new", torch.bfloat16, 3)
    _need(v_new, "v_new", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    if tuple(k_new.shape) != (B, k_cache.shape[2], D) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [B, Hkv, D]")
    if slot_mapping.shape[0] != B:
        raise ValueError("slot_mapping must be [B]")
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    ws_bytes = 0
    if workspace is not None:
        if not (workspace.is_cuda and workspace.is_contiguous()):
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_bytes = workspace.numel() * workspace.element_size()
    rc = lib().pa_decode_step_fp8(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_new), _ptr(v_new),
                                  _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
                                  cache_desc(k_cache), float(k_scale), float(v_scale),
                                  _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B, Hq,
                                  float(scale), num_splits, _ptr(workspace), ws_bytes, _ptr(status),
                                  _stream(stream))
    _check("pa_decode_step_fp8", rc)


@_on_tensors_device
def pa_decode_splitkv_noalloc(out, lse, q, k_cache, v_cache, block_tables, seq_lens, scale,
                              num_splits=0, status=None, stream=None):
    """Split-KV decode with the partials in the library's built-in device array
    (no workspace argument, no allocation).  Calls that overlap on the GPU race
    on that array; the first call on a device should precede stream capture."""
    B, Hq, D = _decode_inputs(q, k_cache, v_cache, block_tables, seq_lens)
    _need(out, "out", torch.bfloat16, 3)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    rc = lib().pa_decode_splitkv_noalloc(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache),
                                         _ptr(v_cache), cache_desc(k_cache), _ptr(block_tables),
                                         block_tables.shape[1], _ptr(seq_lens), B, Hq,
                                         float(scale), num_splits, _ptr(status), _stream(stream))
    _check("pa_decode_splitkv_noalloc", rc)
