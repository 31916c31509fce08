"""fp64 CPU oracle for paged-KV decode attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use this package.  The product path (the CUDA
library and its Python binding) never imports it, and it imports nothing from
the product.  The arithmetic lives in ``pa_oracle.c`` (plain C, double
precision, OpenMP over query rows); this module builds it with gcc and
marshals numpy arrays into it.

bf16 tensors are passed as ``numpy.uint16`` arrays holding the bit patterns.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")

_lock = threading.Lock()
_lib = None

ORACLE_OK = 0
ORACLE_EBADARG = -1
ORACLE_EBLOCK = -2
ORACLE_ESLOT = -3


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into _build/liboracle.so (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _bind(lib):
    P = ctypes.c_void_p
    i32, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
    lib.oracle_cache_write.argtypes = [P, P, P, i64, P, P, i32, i32, i32, i32]
    f64 = ctypes.c_double
    lib.oracle_decode_rows.argtypes = [P, P, P, P, i32, P, P, P, i32, i32, i32, i32,
                                       P, i32, P, i32, i32, f64, P, i32]
    lib.oracle_decode_partial.argtypes = [P, P, P, P, P, i32, i32, i32, i32,
                                          P, i32, P, i32, i32, f64, i32, i32, P, i32]
    lib.oracle_combine.argtypes = [P, P, P, P, i64, i32, i32]
    lib.oracle_e4m3_to_bf16.argtypes = [P, P, i64]
    lib.oracle_bf16_to_e4m3.argtypes = [P, P, i64, f32]
    lib.oracle_cache_write_fp8.argtypes = [P, P, P, i64, P, P, i32, i32, i32, i32, f32, f32]
    lib.oracle_decode_mq.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32, P, i32, P, i32, i32,
                                     f64, P, i32]
    lib.oracle_max_threads.argtypes = []
    for fn in (lib.oracle_cache_write, lib.oracle_decode_rows,
               lib.oracle_decode_partial, lib.oracle_combine, lib.oracle_max_threads):
        fn.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def use_library(path: str):
    """Temporarily route every oracle call through another build of pa_oracle.c.

    The pin tests use this to run deliberately broken copies of the oracle
    (mutants compiled from edited source) and check that some pin fails.
    """
    global _lib
    prev = _load()
    with _lock:
        _lib = _bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        with _lock:
            _lib = prev


def compile_variant(src_text: str, out_path: str) -> str:
    """Compile an edited copy of the oracle source (same flags as build())."""
    c_path = out_path + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                    "-fno-fast-math", "-ffp-contract=off", c_path, "-o", out_path, "-lm"],
                   check=True)
    return out_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _req(a, dtype):
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return np.ascontiguousarray(a)


def _f32(x) -> float:
    """The fp32 value of a scale, as the library receives it, widened to a Python float."""
    return float(np.float32(x))


def _check(rc, what):
    if rc != ORACLE_OK:
        raise OracleError(f"{what} failed with code {rc}")


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def cache_write(k_new, v_new, slot_mapping, k_cache, v_cache):
    """In-place slot-mapping scatter into the (uint16) pools."""
    k_new = _req(k_new, np.uint16)
    v_new = _req(v_new, np.uint16)
    slot_mapping = _req(slot_mapping, np.int64)
    if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
        raise ValueError("pools must be C-contiguous")
    nb, bs, hkv, d = k_cache.shape
    if k_new.shape != (slot_mapping.shape[0], hkv, d) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [N, Hkv, D]")
    rc = _load().oracle_cache_write(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                    slot_mapping.shape[0], _ptr(k_cache), _ptr(v_cache),
                                    nb, bs, hkv, d)
    _check(rc, "oracle_cache_write")


def _common(q, k_cache, v_cache, block_tables, seq_lens):
    q = _req(q, np.uint16)
    k_cache = _req(k_cache, np.uint16)
    v_cache = _req(v_cache, np.uint16)
    block_tables = _req(block_tables, np.int32)
    seq_lens = _req(seq_lens, np.int32)
    B, Hq, D = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("cache shape mismatch")
    if block_tables.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("block_tables/seq_lens shape mismatch")
    return q, k_cache, v_cache, block_tables, seq_lens, B, Hq, D, nb, bs, hkv


def decode_rows(q, k_cache, v_cache, block_tables, seq_lens, scale, rows_b, rows_h,
                nthreads: int = 0):
    """Exact attention for the listed (b, h) rows: returns (out[n, D], lse[n]) in fp64.
    ``scale`` is taken as the fp32 value the library's callers pass."""
    return _decode_rows_exact(q, k_cache, v_cache, block_tables, seq_lens, _f32(scale), rows_b,
                              rows_h, nthreads)


def _decode_rows_exact(q, k_cache, v_cache, block_tables, seq_lens, scale, rows_b, rows_h,
                       nthreads: int = 0):
    """decode_rows with ``scale`` used as given, in double precision."""
    q, k_cache, v_cache, block_tables, seq_lens, B, Hq, D, nb, bs, hkv = _common(
        q, k_cache, v_cache, block_tables, seq_lens)
    rows_b = _req(rows_b, np.int32)
    rows_h = _req(rows_h, np.int32)
    n = rows_b.shape[0]
    out = np.empty((n, D), np.float64)
    lse = np.empty((n,), np.float64)
    nthr = nthreads if nthreads > 0 else max_threads()
    scores = np.empty((max(nthr, max_threads()), block_tables.shape[1] * bs), np.float64)
    rc = _load().oracle_decode_rows(_ptr(out), _ptr(lse), _ptr(rows_b), _ptr(rows_h), n,
                                    _ptr(q), _ptr(k_cache), _ptr(v_cache), nb, bs, hkv, D,
                                    _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
                                    B, Hq, float(scale), _ptr(scores), nthreads)
    _check(rc, "oracle_decode_rows")
    return out, lse


def decode(q, k_cache, v_cache, block_tables, seq_lens, scale, nthreads: int = 0):
    """Exact attention for every (b, h): returns (out[B, Hq, D], lse[B, Hq]) in fp64."""
    return _decode_exact(q, k_cache, v_cache, block_tables, seq_lens, _f32(scale), nthreads)


def _decode_exact(q, k_cache, v_cache, block_tables, seq_lens, scale, nthreads: int = 0):
    B, Hq, D = np.asarray(q).shape
    bb, hh = np.meshgrid(np.arange(B, dtype=np.int32), np.arange(Hq, dtype=np.int32),
                         indexing="ij")
    out, lse = _decode_rows_exact(q, k_cache, v_cache, block_tables, seq_lens, scale,
                                  bb.ravel(), hh.ravel(), nthreads)
    return out.reshape(B, Hq, D), lse.reshape(B, Hq)


# ------------------------------------------------------------------ FP8 KV
def e4m3_to_bf16(codes):
    """Exact widening of e4m3 codes (uint8) to bf16 bit patterns (uint16)."""
    codes = _req(codes, np.uint8)
    out = np.empty(codes.shape, np.uint16)
    _check(_load().oracle_e4m3_to_bf16(_ptr(out), _ptr(codes), codes.size), "oracle_e4m3_to_bf16")
    return out


def bf16_to_e4m3(x, scale):
    """Quantise bf16 bit patterns to e4m3 codes: RNE of fp32(x) / scale, saturating at +-448."""
    x = _req(x, np.uint16)
    out = np.empty(x.shape, np.uint8)
    _check(_load().oracle_bf16_to_e4m3(_ptr(out), _ptr(x), x.size, float(scale)),
           "oracle_bf16_to_e4m3")
    return out


def cache_write_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale):
    """In-place slot-mapping scatter of quantised rows into uint8 e4m3 pools."""
    k_new = _req(k_new, np.uint16)
    v_new = _req(v_new, np.uint16)
    slot_mapping = _req(slot_mapping, np.int64)
    if k_cache.dtype != np.uint8 or v_cache.dtype != np.uint8:
        raise TypeError("fp8 pools must be uint8")
    if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
        raise ValueError("pools must be C-contiguous")
    nb, bs, hkv, d = k_cache.shape
    rc = _load().oracle_cache_write_fp8(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                        slot_mapping.shape[0], _ptr(k_cache), _ptr(v_cache),
                                        nb, bs, hkv, d, float(k_scale), float(v_scale))
    _check(rc, "oracle_cache_write_fp8")


def decode_fp8(q, k_cache, v_cache, block_tables, seq_lens, scale, k_scale, v_scale,
               nthreads: int = 0):
    """Exact attention over e4m3 pools whose code c stands for e4m3(c) * k_scale
    (K) and e4m3(c) * v_scale (V), the scales being the fp32 values the library
    receives.  A per-pool scale factors out of the attention exactly: the
    scores are (scale * k_scale) times the dot products with the widened codes,
    that product formed in double precision, and the output is multiplied by
    v_scale.  Returns (out[B, Hq, D], lse[B, Hq]) in fp64."""
    kw = e4m3_to_bf16(k_cache)
    vw = e4m3_to_bf16(v_cache)
    out, lse = _decode_exact(q, kw, vw, block_tables, seq_lens, _f32(scale) * _f32(k_scale),
                             nthreads)
    return out * _f32(v_scale), lse


def decode_mq(q, k_cache, v_cache, block_tables, seq_lens, scale, nthreads: int = 0):
    """Causal multi-query attention: q is [B, q_len, Hq, D] (the last q_len
    positions of each sequence); returns (out[B, q_len, Hq, D], lse[B, q_len, Hq])."""
    q = _req(q, np.uint16)
    B, q_len, Hq, D = q.shape
    _, k_cache, v_cache, block_tables, seq_lens, _, _, _, nb, bs, hkv = _common(
        q[:, 0], k_cache, v_cache, block_tables, seq_lens)
    out = np.empty((B, q_len, Hq, D), np.float64)
    lse = np.empty((B, q_len, Hq), np.float64)
    nthr = nthreads if nthreads > 0 else max_threads()
    scores = np.empty((max(nthr, max_threads()), block_tables.shape[1] * bs), np.float64)
    rc = _load().oracle_decode_mq(_ptr(out), _ptr(lse), _ptr(q), q_len, _ptr(k_cache),
                                  _ptr(v_cache), nb, bs, hkv, D, _ptr(block_tables),
                                  block_tables.shape[1], _ptr(seq_lens), B, Hq, _f32(scale),
                                  _ptr(scores), nthreads)
    _check(rc, "oracle_decode_mq")
    return out, lse


def decode_partial(q, k_cache, v_cache, block_tables, seq_lens, scale, num_parts, chunk,
                   nthreads: int = 0):
    """Per-partition partials: (part_o[B, Hq, P, D], part_lse[B, Hq, P]) in fp64."""
    q, k_cache, v_cache, block_tables, seq_lens, B, Hq, D, nb, bs, hkv = _common(
        q, k_cache, v_cache, block_tables, seq_lens)
    part_o = np.empty((B, Hq, num_parts, D), np.float64)
    part_lse = np.empty((B, Hq, num_parts), np.float64)
    nthr = nthreads if nthreads > 0 else max_threads()
    scores = np.empty((max(nthr, max_threads()), block_tables.shape[1] * bs), np.float64)
    rc = _load().oracle_decode_partial(_ptr(part_o), _ptr(part_lse), _ptr(q), _ptr(k_cache),
                                       _ptr(v_cache), nb, bs, hkv, D, _ptr(block_tables),
                                       block_tables.shape[1], _ptr(seq_lens), B, Hq,
                                       _f32(scale), num_parts, chunk, _ptr(scores), nthreads)
    _check(rc, "oracle_decode_partial")
    return part_o, part_lse


def combine(part_o, part_lse):
    """Log-sum-exp merge over the partition axis: returns (out[..., D], lse[...])."""
    part_o = _req(part_o, np.float64)
    part_lse = _req(part_lse, np.float64)
    *lead, P, D = part_o.shape
    if tuple(part_lse.shape) != tuple(lead) + (P,):
        raise ValueError("part_lse shape mismatch")
    rows = int(np.prod(lead)) if lead else 1
    out = np.empty(tuple(lead) + (D,), np.float64)
    lse = np.empty(tuple(lead), np.float64)
    rc = _load().oracle_combine(_ptr(out), _ptr(lse), _ptr(part_o), _ptr(part_lse), rows, P, D)
    _check(rc, "oracle_combine")
    return out, lse
