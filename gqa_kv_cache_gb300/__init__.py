"""GQA decode step over a KV cache on GB300 (sm_103a).

Thin Python binding of ``libgqa.so``: it checks tensor shapes and dtypes,
passes device pointers and the current CUDA stream to the C ABI
(include/gqa_decode.h) and raises on error codes. Every step of the decode
runs in the library's CUDA kernels; PyTorch only provides device memory and
streams. There is no CPU fallback: without the built library or a GPU the
calls raise.

One decode step, per batch row b: the new key/value are appended in place at
slot ``lengths[b]`` of the row's cache, and every query head h attends over
slots ``0..lengths[b]`` of cache head ``h // (Hq // Hkv)`` with a float32
softmax of ``q.K/sqrt(D)``; the output is float32 (B, Hq, D).

The read-only attend (``attend``, ``attend_paged``) attends slots
``0..lengths[b]-1`` (lengths counts the valid slots) and writes nothing but
its output; its query may be float32 over a bfloat16 cache.

A cache of E4M3 (FP8) bytes (``torch.uint8`` or ``torch.float8_e4m3fn``
tensors) takes ``k_scale`` / ``v_scale`` float32 (Hkv,) tensors: K =
k_scale[kvh] * K8; the decode step then takes bfloat16 q, k_new and v_new and
quantises the appended token.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

__all__ = ["decode_step", "decode_step_paged", "attend", "attend_paged", "decode_multi",
           "decode_multi_paged", "workspace_bytes", "validate", "validate_attend", "validate_multi",
           "GqaError", "trace_enable", "trace_collect", "KERNELS", "library_path"]

OK, INVALID_ARGUMENT, UNSUPPORTED, CUDA_ERROR, WORKSPACE = 0, 1, 2, 3, 4
KERNELS = {"auto": 0, "simt": 1, "tc": 2, "unit": 3, "tc5": 4}
STATUS_BITS = {1: "bad length", 2: "bad slot id", 4: "bad block", 8: "timeout", 16: "bad kept prefix",
               32: "bad token offsets"}
_DTYPES = {torch.float32: 0, torch.bfloat16: 1}
E4M3 = 2
_BYTE_DTYPES = (torch.uint8,) + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ())


def _cache_code(t) -> int:
    """gqa_dtype of a cache tensor."""
    if t.dtype in _BYTE_DTYPES:
        return E4M3
    if t.dtype not in _DTYPES:
        raise TypeError("a cache must be float32, bfloat16 or E4M3 bytes")
    return _DTYPES[t.dtype]

library_path = _lib.LIB_PATH


class GqaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        msg = _lib.load().gqa_status_string(code).decode()
        super().__init__(f"{what}: {msg} (status {code})")


def _check(code: int, what: str):
    if code != OK:
        raise GqaError(code, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _opts(kernel, grid_ctas, sched_pad=None, sink=None, window=0, kept_prefix=0, device=None, B=None,
          Hq=None, k_scale=None, v_scale=None, Hkv=None, wait_limit_cycles=0, test_stall=False):
    """The gqa_options struct. Softmax modifiers: ``sink`` a float32 (Hq,)
    device tensor, ``window`` an int >= 0, ``kept_prefix`` an int >= 0 or an
    int32 (B,) device tensor. ``wait_limit_cycles`` > 0 shortens the
    tensor-core consumers' wait for a tile to that many SM clock cycles and
    ``test_stall`` makes each consumer's first wait one that runs out (both
    for tests of the timeout path)."""
    o = _lib.GqaOptions()
    o.wait_limit_cycles = int(wait_limit_cycles or 0)
    o.test_stall = 1 if test_stall else 0
    o.kernel = KERNELS[kernel] if isinstance(kernel, str) else int(kernel)
    o.grid_ctas = int(grid_ctas)
    o.sched_pad = 0 if sched_pad is None else int(sched_pad) + 1   # 0 = library default
    o.window = int(window or 0)
    if sink is not None:
        if sink.dtype != torch.float32 or sink.shape != (Hq,) or not sink.is_contiguous() \
                or sink.device != device:
            raise TypeError("sink must be a contiguous float32 (Hq,) tensor on q's device")
        o.head_sink = sink.data_ptr()
    if isinstance(kept_prefix, torch.Tensor):
        if kept_prefix.dtype != torch.int32 or kept_prefix.shape != (B,) \
                or not kept_prefix.is_contiguous() or kept_prefix.device != device:
            raise TypeError("kept_prefix must be an int or a contiguous int32 (B,) tensor on q's device")
        o.kept_prefix_rows = kept_prefix.data_ptr()
    else:
        o.kept_prefix = int(kept_prefix or 0)
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        if t is None:
            continue
        if t.dtype != torch.float32 or t.shape != (Hkv,) or not t.is_contiguous() or t.device != device:
            raise TypeError(f"{name} must be a contiguous float32 (Hkv,) tensor on q's device")
        setattr(o, name, t.data_ptr())
    return o


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


_ws_cache: dict = {}


def _workspace(device, nbytes):
    """A per-device workspace, zero-filled when allocated; the library leaves
    it zero-filled after every call, whatever the sizes."""
    buf = _ws_cache.get(device)
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _ws_cache[device] = buf
    return buf


def workspace_bytes(B, Hq, Hkv, D, dtype=torch.bfloat16, kernel="auto", grid_ctas=0) -> int:
    """Workspace bytes the library needs for one step of these sizes."""
    o = _opts(kernel, grid_ctas)
    code = E4M3 if dtype in _BYTE_DTYPES else _DTYPES[dtype]
    return int(_lib.load().gqa_workspace_bytes(B, Hq, Hkv, D, code, ctypes.byref(o)))


def _common_checks(q, k_new, v_new, caches, lengths, out, q_any_dtype=False):
    """Checks shared by the entry points; returns (cache gqa_dtype, out). The
    query and the new keys / values share the cache dtype, except over an E4M3
    cache (bfloat16 then; the attend's query is free)."""
    if not q.is_cuda:
        raise ValueError("tensors must be on a CUDA device")
    if q.dtype not in _DTYPES:
        raise TypeError("q must be float32 or bfloat16")
    code = _cache_code(caches[0][1])
    if code == E4M3:
        if not q_any_dtype and q.dtype != torch.bfloat16:
            raise TypeError("over an E4M3 cache q, k_new and v_new are bfloat16")
        new_dt = torch.bfloat16
    else:
        dt = caches[0][1].dtype if q_any_dtype else q.dtype
        if dt not in _DTYPES:
            raise TypeError("the cache must be float32 or bfloat16")
        new_dt = dt
    news = () if k_new is None else (("k_new", k_new), ("v_new", v_new))
    for name, t in news:
        if t.dtype != new_dt:
            raise TypeError(f"{name} must have dtype {new_dt}")
    for name, t in caches:
        if t.dtype != caches[0][1].dtype:
            raise TypeError(f"{name} must have dtype {caches[0][1].dtype}")
    for name, t in (*news, *caches):
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if not q.is_contiguous():
        raise ValueError("q must be contiguous")
    if lengths.dtype != torch.int32 or not lengths.is_contiguous() or lengths.device != q.device:
        raise TypeError("lengths must be a contiguous int32 tensor on q's device")
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    elif out.shape != (B, Hq, D) or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 (B, Hq, D) tensor")
    return code, out


def decode_step(q, k_new, v_new, k_cache, v_cache, lengths, slot_ids=None, *, out=None,
                status=None, kernel="auto", grid_ctas=0, workspace=None, stream=None, sched_pad=None,
                sink=None, window=0, kept_prefix=0, k_scale=None, v_scale=None,
                wait_limit_cycles=0, test_stall=False):
    """One decode step on a dense (R, Hkv, Smax, D) cache (continuous batch
    when ``slot_ids`` is given). Appends in place; returns ``out``. A
    ``workspace`` passed in must be zero-filled before its first use (the
    library leaves it zero-filled after every call). ``sink``, ``window`` and
    ``kept_prefix`` are the softmax modifiers of the C header's gqa_options."""
    dt, out = _common_checks(q, k_new, v_new, (("k_cache", k_cache), ("v_cache", v_cache)),
                             lengths, out)
    B, Hq, D = q.shape
    R, Hkv, Smax, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape or k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D):
        raise ValueError("shape mismatch between q, k_new, v_new and the caches")
    if slot_ids is not None and (slot_ids.dtype != torch.int32 or slot_ids.shape != (B,)):
        raise TypeError("slot_ids must be int32 of shape (B,)")
    o = _opts(kernel, grid_ctas, sched_pad, sink, window, kept_prefix, q.device, B, Hq, k_scale, v_scale, Hkv,
              wait_limit_cycles, test_stall)
    lib = _lib.load()
    need = lib.gqa_workspace_bytes(B, Hq, Hkv, D, dt, ctypes.byref(o))
    ws = _workspace(q.device, need) if workspace is None else workspace
    code = lib.gqa_decode_step_ex(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(lengths), _ptr(slot_ids), _ptr(out), B, Hq, Hkv, D, R, Smax,
                                  dt, _ptr(ws), ws.numel() * ws.element_size(),
                                  _ptr(status), _stream(stream), ctypes.byref(o))
    _check(code, "gqa_decode_step")
    return out


def decode_step_paged(q, k_new, v_new, k_blocks, v_blocks, block_table, lengths, *, out=None,
                      status=None, kernel="auto", grid_ctas=0, workspace=None, stream=None,
                      sched_pad=None, sink=None, window=0, kept_prefix=0, k_scale=None, v_scale=None,
                      wait_limit_cycles=0, test_stall=False):
    """One decode step on a paged cache (num_blocks, Hkv, block_size, D) with
    a (B, max_blocks) int32 block table (-1 = unused). Appends in place."""
    dt, out = _common_checks(q, k_new, v_new, (("k_blocks", k_blocks), ("v_blocks", v_blocks)),
                             lengths, out)
    B, Hq, D = q.shape
    NB, Hkv, BS, D2 = k_blocks.shape
    if D2 != D or v_blocks.shape != k_blocks.shape or k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D):
        raise ValueError("shape mismatch between q, k_new, v_new and the blocks")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B \
            or not block_table.is_contiguous():
        raise TypeError("block_table must be a contiguous int32 (B, max_blocks) tensor")
    MB = block_table.shape[1]
    o = _opts(kernel, grid_ctas, sched_pad, sink, window, kept_prefix, q.device, B, Hq, k_scale, v_scale, Hkv,
              wait_limit_cycles, test_stall)
    lib = _lib.load()
    need = lib.gqa_workspace_bytes(B, Hq, Hkv, D, dt, ctypes.byref(o))
    ws = _workspace(q.device, need) if workspace is None else workspace
    code = lib.gqa_decode_step_paged_ex(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_blocks),
                                        _ptr(v_blocks), _ptr(block_table), _ptr(lengths), _ptr(out),
                                        B, Hq, Hkv, D, NB, BS, MB, dt, _ptr(ws),
                                        ws.numel() * ws.element_size(), _ptr(status),
                                        _stream(stream), ctypes.byref(o))
    _check(code, "gqa_decode_step_paged")
    return out


def attend(q, k_cache, v_cache, lengths, slot_ids=None, *, out=None, status=None, kernel="auto",
           grid_ctas=0, workspace=None, stream=None, sched_pad=None, sink=None, window=0,
           kept_prefix=0, k_scale=None, v_scale=None, wait_limit_cycles=0, test_stall=False):
    """Read-only attend on a dense (R, Hkv, Smax, D) cache: slots
    ``0..lengths[b]-1`` (1 <= lengths[b] <= Smax), nothing written but ``out``.
    ``q`` (B, Hq, D) is float32 or bfloat16 whatever the cache dtype."""
    dt, out = _common_checks(q, None, None, (("k_cache", k_cache), ("v_cache", v_cache)),
                             lengths, out, q_any_dtype=True)
    B, Hq, D = q.shape
    R, Hkv, Smax, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape or Hq % Hkv:
        raise ValueError("shape mismatch between q and the caches")
    if slot_ids is not None and (slot_ids.dtype != torch.int32 or slot_ids.shape != (B,)):
        raise TypeError("slot_ids must be int32 of shape (B,)")
    o = _opts(kernel, grid_ctas, sched_pad, sink, window, kept_prefix, q.device, B, Hq, k_scale, v_scale, Hkv,
              wait_limit_cycles, test_stall)
    lib = _lib.load()
    need = lib.gqa_workspace_bytes(B, Hq, Hkv, D, dt, ctypes.byref(o))
    ws = _workspace(q.device, need) if workspace is None else workspace
    code = lib.gqa_attend(_ptr(q), _DTYPES[q.dtype], _ptr(k_cache), _ptr(v_cache), _ptr(lengths),
                          _ptr(slot_ids), _ptr(out), B, Hq, Hkv, D, R, Smax, dt, _ptr(ws),
                          ws.numel() * ws.element_size(), _ptr(status), _stream(stream),
                          ctypes.byref(o))
    _check(code, "gqa_attend")
    return out


def attend_paged(q, k_blocks, v_blocks, block_table, lengths, *, out=None, status=None,
                 kernel="auto", grid_ctas=0, workspace=None, stream=None, sched_pad=None,
                 sink=None, window=0, kept_prefix=0, k_scale=None, v_scale=None,
                wait_limit_cycles=0, test_stall=False):
    """Read-only attend on a paged cache (num_blocks, Hkv, block_size, D)."""
    dt, out = _common_checks(q, None, None, (("k_blocks", k_blocks), ("v_blocks", v_blocks)),
                             lengths, out, q_any_dtype=True)
    B, Hq, D = q.shape
    NB, Hkv, BS, D2 = k_blocks.shape
    if D2 != D or v_blocks.shape != k_blocks.shape or Hq % Hkv:
        raise ValueError("shape mismatch between q and the blocks")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B \
            or not block_table.is_contiguous():
        raise TypeError("block_table must be a contiguous int32 (B, max_blocks) tensor")
    o = _opts(kernel, grid_ctas, sched_pad, sink, window, kept_prefix, q.device, B, Hq, k_scale, v_scale, Hkv,
              wait_limit_cycles, test_stall)
    lib = _lib.load()
    need = lib.gqa_workspace_bytes(B, Hq, Hkv, D, dt, ctypes.byref(o))
    ws = _workspace(q.device, need) if workspace is None else workspace
    code = lib.gqa_attend_paged(_ptr(q), _DTYPES[q.dtype], _ptr(k_blocks), _ptr(v_blocks),
                                _ptr(block_table), _ptr(lengths), _ptr(out), B, Hq, Hkv, D, NB, BS,
                                block_table.shape[1], dt, _ptr(ws),
                                ws.numel() * ws.element_size(), _ptr(status), _stream(stream),
                                ctypes.byref(o))
    _check(code, "gqa_attend_paged")
    return out


def _multi_checks(q, k_new, v_new, caches, lengths, cu_q, out):
    dt, out = _common_checks(q, k_new, v_new, caches, lengths, out)
    if cu_q.dtype != torch.int32 or cu_q.dim() != 1 or cu_q.shape[0] != lengths.shape[0] + 1 \
            or not cu_q.is_contiguous() or cu_q.device != q.device:
        raise TypeError("cu_q must be a contiguous int32 (B + 1,) tensor on q's device")
    return dt, out


def decode_multi(q, k_new, v_new, k_cache, v_cache, lengths, cu_q, slot_ids=None, *, max_q_len,
                 out=None, status=None, kernel="auto", grid_ctas=0, workspace=None, stream=None,
                 sched_pad=None, sink=None, window=0, kept_prefix=0, k_scale=None,
                 v_scale=None, wait_limit_cycles=0, test_stall=False):
    """Multi-token step on a dense (R, Hkv, Smax, D) cache: the packed tokens
    cu_q[b] .. cu_q[b+1]-1 of row b (q (T, Hq, D), k_new / v_new (T, Hkv, D))
    are appended at slots lengths[b] + i and token i attends slots
    0 .. lengths[b] + i. ``max_q_len`` bounds every q_len. Over an E4M3
    cache q, k_new and v_new are bfloat16 and ``k_scale`` / ``v_scale`` are
    required, as in :func:`decode_step`. Returns out (T, Hq, D)."""
    dt, out = _multi_checks(q, k_new, v_new, (("k_cache", k_cache), ("v_cache", v_cache)), lengths,
                            cu_q, out)
    T, Hq, D = q.shape
    B = lengths.shape[0]
    R, Hkv, Smax, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape or k_new.shape != (T, Hkv, D) or v_new.shape != (T, Hkv, D):
        raise ValueError("shape mismatch between q, k_new, v_new and the caches")
    if slot_ids is not None and (slot_ids.dtype != torch.int32 or slot_ids.shape != (B,)):
        raise TypeError("slot_ids must be int32 of shape (B,)")
    o = _opts(kernel, grid_ctas, sched_pad, sink, window, kept_prefix, q.device, B, Hq, k_scale, v_scale, Hkv,
              wait_limit_cycles, test_stall)
    lib = _lib.load()
    need = lib.gqa_workspace_bytes_multi(B, Hq, Hkv, D, dt, int(max_q_len), ctypes.byref(o))
    ws = _workspace(q.device, need) if workspace is None else workspace
    code = lib.gqa_decode_multi(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                _ptr(lengths), _ptr(cu_q), _ptr(slot_ids), _ptr(out), B, T, int(max_q_len),
                                Hq, Hkv, D, R, Smax, dt, _ptr(ws), ws.numel() * ws.element_size(),
                                _ptr(status), _stream(stream), ctypes.byref(o))
    _check(code, "gqa_decode_multi")
    return out


def decode_multi_paged(q, k_new, v_new, k_blocks, v_blocks, block_table, lengths, cu_q, *, max_q_len,
                       out=None, status=None, kernel="auto", grid_ctas=0, workspace=None, stream=None,
                       sched_pad=None, sink=None, window=0, kept_prefix=0, k_scale=None,
                       v_scale=None, wait_limit_cycles=0, test_stall=False):
    """Multi-token step on a paged cache (num_blocks, Hkv, block_size, D)."""
    dt, out = _multi_checks(q, k_new, v_new, (("k_blocks", k_blocks), ("v_blocks", v_blocks)), lengths,
                            cu_q, out)
    T, Hq, D = q.shape
    B = lengths.shape[0]
    NB, Hkv, BS, D2 = k_blocks.shape
    if D2 != D or v_blocks.shape != k_blocks.shape or k_new.shape != (T, Hkv, D) or v_new.shape != (T, Hkv, D):
        raise ValueError("shape mismatch between q, k_new, v_new and the blocks")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B \
            or not block_table.is_contiguous():
        raise TypeError("block_table must be a contiguous int32 (B, max_blocks) tensor")
    o = _opts(kernel, grid_ctas, sched_pad, sink, window, kept_prefix, q.device, B, Hq, k_scale, v_scale, Hkv,
              wait_limit_cycles, test_stall)
    lib = _lib.load()
    need = lib.gqa_workspace_bytes_multi(B, Hq, Hkv, D, dt, int(max_q_len), ctypes.byref(o))
    ws = _workspace(q.device, need) if workspace is None else workspace
    code = lib.gqa_decode_multi_paged(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_blocks), _ptr(v_blocks),
                                      _ptr(block_table), _ptr(lengths), _ptr(cu_q), _ptr(out), B, T,
                                      int(max_q_len), Hq, Hkv, D, NB, BS, block_table.shape[1], dt,
                                      _ptr(ws), ws.numel() * ws.element_size(), _ptr(status),
                                      _stream(stream), ctypes.byref(o))
    _check(code, "gqa_decode_multi_paged")
    return out


def validate_multi(lengths, cu_q, T, *, slot_ids=None, R=None, Smax=None, block_table=None,
                   num_blocks=None, block_size=None, stream=None) -> bool:
    """Full content check on the GPU for a multi-token step (synchronous)."""
    B = lengths.shape[0]
    res = torch.empty(1, dtype=torch.int32, device=lengths.device)
    lib = _lib.load()
    if block_table is not None:
        code = lib.gqa_validate_multi(_ptr(lengths), _ptr(cu_q), None, _ptr(block_table), B, T, 0, 0,
                                      num_blocks, block_size, block_table.shape[1], _ptr(res), _stream(stream))
    else:
        code = lib.gqa_validate_multi(_ptr(lengths), _ptr(cu_q), _ptr(slot_ids), None, B, T, R, Smax, 0, 0, 0,
                                      _ptr(res), _stream(stream))
    if code == INVALID_ARGUMENT:
        return False
    _check(code, "gqa_validate_multi")
    return True


def _validate(fn, what, lengths, slot_ids, R, Smax, block_table, num_blocks, block_size, stream):
    B = lengths.shape[0]
    res = torch.empty(1, dtype=torch.int32, device=lengths.device)
    if block_table is not None:
        code = fn(_ptr(lengths), None, _ptr(block_table), B, 0, 0, num_blocks, block_size,
                  block_table.shape[1], _ptr(res), _stream(stream))
    else:
        code = fn(_ptr(lengths), _ptr(slot_ids), None, B, R, Smax, 0, 0, 0, _ptr(res),
                  _stream(stream))
    if code == INVALID_ARGUMENT:
        return False
    _check(code, what)
    return True


def validate(lengths, *, slot_ids=None, R=None, Smax=None, block_table=None, num_blocks=None,
             block_size=None, stream=None) -> bool:
    """Full content check on the GPU for the decode step (synchronous). True
    when valid."""
    return _validate(_lib.load().gqa_validate, "gqa_validate", lengths, slot_ids, R, Smax,
                     block_table, num_blocks, block_size, stream)


def validate_attend(lengths, *, slot_ids=None, R=None, Smax=None, block_table=None,
                    num_blocks=None, block_size=None, stream=None) -> bool:
    """Full content check on the GPU for the read-only attend (synchronous)."""
    return _validate(_lib.load().gqa_validate_attend, "gqa_validate_attend", lengths, slot_ids, R,
                     Smax, block_table, num_blocks, block_size, stream)


def trace_enable(on: bool = True) -> bool:
    return bool(_lib.load().gqa_trace_enable(int(on)))


def trace_collect() -> dict:
    """{kernel name: (launches, total ms)} since the previous collect."""
    lib = _lib.load()
    n = 4
    launches = (ctypes.c_int64 * n)()
    ms = (ctypes.c_double * n)()
    _check(lib.gqa_trace_collect(n, launches, ms), "gqa_trace_collect")
    return {lib.gqa_kernel_name(k).decode(): (launches[k], ms[k]) for k in range(n)}
