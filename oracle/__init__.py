"""CPU oracle for the GQA decode step and the read-only attend over a KV
cache (float64 loops, plain C).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package. The CUDA
library shares no code with it and never calls it.

The arithmetic lives in ``gqa_oracle.c`` (see its header for the definition
and the passages it follows). This module only builds that file with gcc,
marshals numpy arrays to it and returns float64 outputs.

bfloat16 data is passed as ``numpy.uint16`` arrays holding the raw bits (the
upper half of an IEEE binary32); float32 data as ``numpy.float32``; an E4M3
(OCP FP8) cache as ``numpy.uint8`` bytes with ``k_scale`` / ``v_scale``
float32 arrays of one scale per cache head.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB = os.path.join(_HERE, "libgqa_oracle.so")

F32, BF16, E4M3 = 0, 1, 2
OK, INVALID_ARGUMENT = 0, 1

_lock = threading.Lock()
_lib = None


class _Mods(ctypes.Structure):
    _fields_ = [("head_sink", ctypes.c_void_p), ("window", ctypes.c_int),
                ("kept_prefix", ctypes.c_int), ("kept_prefix_rows", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p), ("new_dtype", ctypes.c_int)]


def _mods(sink, window, kept_prefix, keep, scales=None):
    """The orc_mods argument (None when no modifier is given). Arrays that
    back it are appended to ``keep`` so they outlive the call. ``scales`` =
    (k_scale, v_scale, new_dtype) for an E4M3 cache."""
    if sink is None and not window and scales is None and \
            (kept_prefix is None or np.isscalar(kept_prefix) and kept_prefix == 0):
        return None
    m = _Mods()
    if scales is not None:
        ks = np.ascontiguousarray(scales[0], dtype=np.float32)
        vs = np.ascontiguousarray(scales[1], dtype=np.float32)
        keep += [ks, vs]
        m.k_scale, m.v_scale, m.new_dtype = ks.ctypes.data, vs.ctypes.data, int(scales[2])
    if sink is not None:
        a = np.ascontiguousarray(sink, dtype=np.float32)
        keep.append(a)
        m.head_sink = a.ctypes.data
    m.window = int(window or 0)
    if kept_prefix is None or np.isscalar(kept_prefix):
        m.kept_prefix = int(kept_prefix or 0)
    else:
        a = np.ascontiguousarray(kept_prefix, dtype=np.int32)
        keep.append(a)
        m.kept_prefix_rows = a.ctypes.data
    return ctypes.byref(m), m


def build(force: bool = False) -> str:
    """Compile the oracle into ``libgqa_oracle.so`` beside its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
             "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # GQA_ORACLE_LIB lets the mutation tests load a deliberately
            # broken copy of the oracle to prove the pins catch it.
            lib = ctypes.CDLL(os.environ.get("GQA_ORACLE_LIB") or build())
            P, I = ctypes.c_void_p, ctypes.c_int
            lib.orc_decode_dense.argtypes = [I, P, P, P, P, P, P, P, I, I, I, I, I, I,
                                             P, I, I, P, P, I, P]
            lib.orc_decode_dense.restype = I
            lib.orc_decode_paged.argtypes = [I, P, P, P, P, P, P, P, I, I, I, I, I, I, I,
                                             P, I, I, P, P, I, P]
            lib.orc_decode_paged.restype = I
            lib.orc_validate_dense.argtypes = [P, P, I, I, I]
            lib.orc_validate_dense.restype = I
            lib.orc_validate_paged.argtypes = [P, P, I, I, I, I]
            lib.orc_validate_paged.restype = I
            lib.orc_attend_dense.argtypes = [I, I, P, P, P, P, P, I, I, I, I, I, I,
                                             P, I, P, P, I, P]
            lib.orc_attend_dense.restype = I
            lib.orc_attend_paged.argtypes = [I, I, P, P, P, P, P, I, I, I, I, I, I, I,
                                             P, I, P, P, I, P]
            lib.orc_attend_paged.restype = I
            lib.orc_validate_attend_dense.argtypes = [P, P, I, I, I]
            lib.orc_validate_attend_dense.restype = I
            lib.orc_validate_attend_paged.argtypes = [P, P, I, I, I, I]
            lib.orc_validate_attend_paged.restype = I
            lib.orc_decode_multi_dense.argtypes = [I, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I,
                                                   I, P, P, I, P]
            lib.orc_decode_multi_dense.restype = I
            lib.orc_decode_multi_paged.argtypes = [I, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I,
                                                   I, P, P, I, P]
            lib.orc_decode_multi_paged.restype = I
            lib.orc_validate_multi_dense.argtypes = [P, P, P, I, I, I, I]
            lib.orc_validate_multi_dense.restype = I
            lib.orc_validate_multi_paged.argtypes = [P, P, P, I, I, I, I, I]
            lib.orc_validate_multi_paged.restype = I
            lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
            lib.orc_e4m3_encode.restype = ctypes.c_uint8
            lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_decode.restype = ctypes.c_double
            lib.orc_default_threads.argtypes = []
            lib.orc_default_threads.restype = I
            _lib = lib
    return _lib


def default_threads() -> int:
    return _load().orc_default_threads()


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.uint8:
        return E4M3
    raise TypeError(f"oracle takes float32, uint16 (bfloat16 bits) or uint8 (E4M3 bytes), not {a.dtype}")


def e4m3_encode(x: float) -> int:
    """E4M3 code of float32 x (round to nearest even, saturating)."""
    return int(_load().orc_e4m3_encode(float(np.float32(x))))


def e4m3_decode(c: int) -> float:
    return float(_load().orc_e4m3_decode(int(c)))


def _cache_dtypes(q, news, caches, k_scale, v_scale):
    """(dtype code passed to the oracle, scales tuple or None): q and the new
    keys / values share one dtype; the caches that one too, or E4M3 bytes with
    per-head scales."""
    for a in news:
        if a is not None and a.dtype != q.dtype:
            raise TypeError("q, k_new and v_new share one dtype")
    for a in caches:
        if not a.flags.c_contiguous:
            raise ValueError("arrays must be C-contiguous (the caches are written in place)")
        if a.dtype != caches[0].dtype:
            raise TypeError("the two caches share one dtype")
    if caches[0].dtype == np.uint8:
        if k_scale is None or v_scale is None:
            raise ValueError("an E4M3 cache needs k_scale and v_scale")
        return E4M3, (k_scale, v_scale, _dtype_code(q))
    if caches[0].dtype != q.dtype:
        raise TypeError("q, k_new, v_new and the caches share one dtype")
    return _dtype_code(q), None


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))
    return a


class OracleResult:
    def __init__(self, status, out, threads):
        self.status = status
        self.out = out
        self.threads = threads


def decode_dense(q, k_new, v_new, k_cache, v_cache, lengths, slot_ids=None, *,
                 rows=None, append=True, threads=None, sink=None, window=0,
                 kept_prefix=0, k_scale=None, v_scale=None) -> OracleResult:
    """One decode step on a dense (R, Hkv, Smax, D) cache, in place.

    ``q`` (B, Hq, D); ``k_new``/``v_new`` (B, Hkv, D); ``lengths`` (B,) int32;
    ``slot_ids`` (B,) int32 or None. With ``append`` the caches (numpy arrays,
    modified in place) receive the new key/value at slot ``lengths[b]``.
    ``rows`` restricts the work to those batch rows (others stay NaN in out).
    Softmax modifiers: ``sink`` (Hq,) float32 logits, ``window`` W (0: none),
    ``kept_prefix`` an int or a (B,) int32 array.
    Returns an OracleResult with ``out`` (B, Hq, D) float64.
    """
    dt, scales = _cache_dtypes(q, (k_new, v_new), (k_cache, v_cache), k_scale, v_scale)
    B, Hq, D = q.shape
    R, Hkv, Smax, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape and k_new.shape == (B, Hkv, D)
    q, k_new, v_new = _c(q), _c(k_new), _c(v_new)
    lengths = _c(lengths, np.int32)
    slot_ids = _c(slot_ids, np.int32)
    rows_a = None if rows is None else _c(np.asarray(rows), np.int32)
    out = np.full((B, Hq, D), np.nan, dtype=np.float64)
    used = ctypes.c_int(0)
    nthr = default_threads() if threads is None else int(threads)
    keep = []
    mods = _mods(sink, window, kept_prefix, keep, scales)
    st = _load().orc_decode_dense(dt, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                  _ptr(v_cache), _ptr(lengths), _ptr(slot_ids),
                                  B, Hq, Hkv, D, R, Smax, _ptr(rows_a),
                                  0 if rows_a is None else len(rows_a), int(bool(append)),
                                  _ptr(out), mods and mods[0], nthr, ctypes.addressof(used))
    return OracleResult(st, out, used.value)


def decode_paged(q, k_new, v_new, k_blocks, v_blocks, block_table, lengths, *,
                 rows=None, append=True, threads=None, sink=None, window=0,
                 kept_prefix=0, k_scale=None, v_scale=None) -> OracleResult:
    """One decode step on a paged cache (num_blocks, Hkv, block_size, D) with a
    (B, max_blocks) int32 block table (-1 = unused). Same contract as
    :func:`decode_dense` otherwise."""
    dt, scales = _cache_dtypes(q, (k_new, v_new), (k_blocks, v_blocks), k_scale, v_scale)
    B, Hq, D = q.shape
    NB, Hkv, BS, D2 = k_blocks.shape
    assert D2 == D and v_blocks.shape == k_blocks.shape and k_new.shape == (B, Hkv, D)
    MB = block_table.shape[1]
    q, k_new, v_new = _c(q), _c(k_new), _c(v_new)
    block_table = _c(block_table, np.int32)
    lengths = _c(lengths, np.int32)
    rows_a = None if rows is None else _c(np.asarray(rows), np.int32)
    out = np.full((B, Hq, D), np.nan, dtype=np.float64)
    used = ctypes.c_int(0)
    nthr = default_threads() if threads is None else int(threads)
    keep = []
    mods = _mods(sink, window, kept_prefix, keep, scales)
    st = _load().orc_decode_paged(dt, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_blocks),
                                  _ptr(v_blocks), _ptr(block_table), _ptr(lengths),
                                  B, Hq, Hkv, D, NB, BS, MB, _ptr(rows_a),
                                  0 if rows_a is None else len(rows_a), int(bool(append)),
                                  _ptr(out), mods and mods[0], nthr, ctypes.addressof(used))
    return OracleResult(st, out, used.value)


def attend_dense(q, k_cache, v_cache, lengths, slot_ids=None, *, rows=None,
                 threads=None, sink=None, window=0, kept_prefix=0, k_scale=None,
                 v_scale=None) -> OracleResult:
    """Read-only attend on a dense (R, Hkv, Smax, D) cache: every query head
    attends slots ``0 .. lengths[b]-1`` of its cache head; nothing is written.
    ``q`` may be float32 over a bfloat16 cache. Returns ``out`` (B, Hq, D)
    float64."""
    qt = _dtype_code(q)
    kt = _dtype_code(k_cache)
    if v_cache.dtype != k_cache.dtype:
        raise TypeError("k_cache and v_cache share one dtype")
    B, Hq, D = q.shape
    R, Hkv, Smax, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape
    q, k_cache, v_cache = _c(q), _c(k_cache), _c(v_cache)
    lengths = _c(lengths, np.int32)
    slot_ids = _c(slot_ids, np.int32)
    rows_a = None if rows is None else _c(np.asarray(rows), np.int32)
    out = np.full((B, Hq, D), np.nan, dtype=np.float64)
    used = ctypes.c_int(0)
    nthr = default_threads() if threads is None else int(threads)
    keep = []
    mods = _mods(sink, window, kept_prefix, keep,
                 (k_scale, v_scale, qt) if kt == E4M3 else None)
    st = _load().orc_attend_dense(qt, kt, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(lengths),
                                  _ptr(slot_ids), B, Hq, Hkv, D, R, Smax, _ptr(rows_a),
                                  0 if rows_a is None else len(rows_a), _ptr(out),
                                  mods and mods[0], nthr, ctypes.addressof(used))
    return OracleResult(st, out, used.value)


def attend_paged(q, k_blocks, v_blocks, block_table, lengths, *, rows=None,
                 threads=None, sink=None, window=0, kept_prefix=0, k_scale=None,
                 v_scale=None) -> OracleResult:
    """Read-only attend on a paged cache; same contract as :func:`attend_dense`."""
    qt = _dtype_code(q)
    kt = _dtype_code(k_blocks)
    if v_blocks.dtype != k_blocks.dtype:
        raise TypeError("k_blocks and v_blocks share one dtype")
    B, Hq, D = q.shape
    NB, Hkv, BS, D2 = k_blocks.shape
    assert D2 == D and v_blocks.shape == k_blocks.shape
    MB = block_table.shape[1]
    q, k_blocks, v_blocks = _c(q), _c(k_blocks), _c(v_blocks)
    block_table = _c(block_table, np.int32)
    lengths = _c(lengths, np.int32)
    rows_a = None if rows is None else _c(np.asarray(rows), np.int32)
    out = np.full((B, Hq, D), np.nan, dtype=np.float64)
    used = ctypes.c_int(0)
    nthr = default_threads() if threads is None else int(threads)
    keep = []
    mods = _mods(sink, window, kept_prefix, keep,
                 (k_scale, v_scale, qt) if kt == E4M3 else None)
    st = _load().orc_attend_paged(qt, kt, _ptr(q), _ptr(k_blocks), _ptr(v_blocks),
                                  _ptr(block_table), _ptr(lengths), B, Hq, Hkv, D, NB, BS, MB,
                                  _ptr(rows_a), 0 if rows_a is None else len(rows_a), _ptr(out),
                                  mods and mods[0], nthr, ctypes.addressof(used))
    return OracleResult(st, out, used.value)


def decode_multi_dense(q, k_new, v_new, k_cache, v_cache, lengths, cu_q, slot_ids=None, *,
                       append=True, threads=None, sink=None, window=0, kept_prefix=0,
                       k_scale=None, v_scale=None) -> OracleResult:
    """Multi-token step on a dense (R, Hkv, Smax, D) cache: the q_len[b] =
    cu_q[b+1] - cu_q[b] new tokens of row b (rows cu_q[b].. of the packed
    q (T, Hq, D), k_new / v_new (T, Hkv, D)) are appended in place at slots
    lengths[b] + i, and token i attends slots 0 .. lengths[b] + i. Returns
    ``out`` (T, Hq, D) float64."""
    dt, scales = _cache_dtypes(q, (k_new, v_new), (k_cache, v_cache), k_scale, v_scale)
    T, Hq, D = q.shape
    R, Hkv, Smax, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape and k_new.shape == (T, Hkv, D)
    q, k_new, v_new = _c(q), _c(k_new), _c(v_new)
    lengths, cu_q, slot_ids = _c(lengths, np.int32), _c(cu_q, np.int32), _c(slot_ids, np.int32)
    B = len(lengths)
    out = np.full((T, Hq, D), np.nan, dtype=np.float64)
    used = ctypes.c_int(0)
    nthr = default_threads() if threads is None else int(threads)
    keep = []
    mods = _mods(sink, window, kept_prefix, keep, scales)
    st = _load().orc_decode_multi_dense(dt, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                        _ptr(v_cache), _ptr(lengths), _ptr(cu_q), _ptr(slot_ids), B, T,
                                        Hq, Hkv, D, R, Smax, int(bool(append)), _ptr(out),
                                        mods and mods[0], nthr, ctypes.addressof(used))
    return OracleResult(st, out, used.value)


def decode_multi_paged(q, k_new, v_new, k_blocks, v_blocks, block_table, lengths, cu_q, *,
                       append=True, threads=None, sink=None, window=0, kept_prefix=0,
                       k_scale=None, v_scale=None) -> OracleResult:
    """Multi-token step on a paged cache; same contract as
    :func:`decode_multi_dense`."""
    dt, scales = _cache_dtypes(q, (k_new, v_new), (k_blocks, v_blocks), k_scale, v_scale)
    T, Hq, D = q.shape
    NB, Hkv, BS, D2 = k_blocks.shape
    assert D2 == D and v_blocks.shape == k_blocks.shape and k_new.shape == (T, Hkv, D)
    MB = block_table.shape[1]
    q, k_new, v_new = _c(q), _c(k_new), _c(v_new)
    block_table, lengths, cu_q = _c(block_table, np.int32), _c(lengths, np.int32), _c(cu_q, np.int32)
    B = len(lengths)
    out = np.full((T, Hq, D), np.nan, dtype=np.float64)
    used = ctypes.c_int(0)
    nthr = default_threads() if threads is None else int(threads)
    keep = []
    mods = _mods(sink, window, kept_prefix, keep, scales)
    st = _load().orc_decode_multi_paged(dt, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_blocks),
                                        _ptr(v_blocks), _ptr(block_table), _ptr(lengths), _ptr(cu_q), B,
                                        T, Hq, Hkv, D, NB, BS, MB, int(bool(append)), _ptr(out),
                                        mods and mods[0], nthr, ctypes.addressof(used))
    return OracleResult(st, out, used.value)


def validate_multi_dense(lengths, cu_q, slot_ids, T, R, Smax) -> int:
    lengths, cu_q, slot_ids = _c(lengths, np.int32), _c(cu_q, np.int32), _c(slot_ids, np.int32)
    return _load().orc_validate_multi_dense(_ptr(lengths), _ptr(cu_q), _ptr(slot_ids), len(lengths), T,
                                            R, Smax)


def validate_multi_paged(lengths, cu_q, block_table, T, num_blocks, block_size) -> int:
    lengths, cu_q, bt = _c(lengths, np.int32), _c(cu_q, np.int32), _c(block_table, np.int32)
    return _load().orc_validate_multi_paged(_ptr(lengths), _ptr(cu_q), _ptr(bt), len(lengths), T,
                                            num_blocks, block_size, bt.shape[1])


def validate_attend_dense(lengths, slot_ids, R, Smax) -> int:
    lengths = _c(lengths, np.int32)
    slot_ids = _c(slot_ids, np.int32)
    return _load().orc_validate_attend_dense(_ptr(lengths), _ptr(slot_ids), len(lengths), R, Smax)


def validate_attend_paged(lengths, block_table, num_blocks, block_size) -> int:
    lengths = _c(lengths, np.int32)
    block_table = _c(block_table, np.int32)
    return _load().orc_validate_attend_paged(_ptr(lengths), _ptr(block_table), len(lengths),
                                             num_blocks, block_size, block_table.shape[1])


def validate_dense(lengths, slot_ids, R, Smax) -> int:
    lengths = _c(lengths, np.int32)
    slot_ids = _c(slot_ids, np.int32)
    return _load().orc_validate_dense(_ptr(lengths), _ptr(slot_ids), len(lengths), R, Smax)


def validate_paged(lengths, block_table, num_blocks, block_size) -> int:
    lengths = _c(lengths, np.int32)
    block_table = _c(block_table, np.int32)
    return _load().orc_validate_paged(_ptr(lengths), _ptr(block_table), len(lengths),
                                      num_blocks, block_size, block_table.shape[1])
