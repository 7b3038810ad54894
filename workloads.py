"""Seeded synthetic inputs for the GQA decode step.

This module only draws random numbers into tensors of the right shapes; it
holds none of the decode step's arithmetic. Both the CUDA path's tests and
benchmark and the CPU oracle's tests take their inputs from here.

Workloads (shapes and distributions of the five decode configurations the
library is measured on):

  pr1_fp32       fp32, B=2, Hq=8, Hkv=2 (G=4), D=64, cache (B,Hkv,256,D);
                 lengths ~ U{1..255}; q, new K/V and valid slots ~ N(0,1);
                 stale slots (index >= lengths[b]) ~ N(0, 100^2).
  llama3_8b      bf16, B=32, Hq=32, Hkv=8 (G=4), D=128, cache (B,Hkv,4096,D);
                 lengths ~ U{1024..4095}; every value ~ N(0,1) cast to bf16.
  long_context   bf16, B=4, Hq=64, Hkv=8 (G=8), D=128, Smax=131072;
                 lengths ~ U{32768..131071}; values ~ N(0,1); every key
                 (cache and new) scaled by 3 before the cast.
  ragged_slots   bf16, B=256, Hq=32, Hkv=4 (G=8), D=128, cache
                 (512,Hkv,8192,D); slot_ids = first B of a random permutation
                 of the 512 rows; lengths = floor(exp(U[ln 16, ln 8192)))
                 clipped to [16, 8191].
  paged          bf16, B=64, Hq=48, Hkv=8 (G=6), D=128, blocks
                 (65536,Hkv,16,D); block table = a random permutation of the
                 65536 blocks reshaped to (64,1024), entries at index
                 >= ceil((lengths[b]+1)/16) set to -1; lengths ~ U{512..16383}.

The read-only attend uses the same draws (``generate(w, attend=True)``):
lengths then count the valid slots (the decode draw + 1, so the slot the
decode step would append to is valid data), the stale region starts after
them, and there is no k_new / v_new; ``q_f32=True`` keeps the query in
float32 instead of casting it to the cache dtype.

The multi-token step uses ``generate(w, q_lens=...)``: row b brings
q_lens[b] new tokens, lengths are the decode draw clamped so the tokens fit
(lengths[b] + q_lens[b] <= capacity), q / k_new / v_new are packed over the
T = sum(q_lens) tokens, cu_q holds the offsets and a paged table covers
every touched slot.

``generate(w, kv_e4m3=True)`` stores the cache as E4M3 (OCP FP8) bytes:
the same draws, divided per cache head by a scale 4 * key_scale / 448 (so
N(0,1) data up to 4 sigma uses the whole E4M3 range), clamped to +-448 and
cast with torch's float8_e4m3fn; k_scale / v_scale hold the scales; q,
k_new and v_new stay bfloat16.

Random draws come from a ``torch.Generator`` on the target device seeded
with the workload's seed, in a fixed order, in chunks of ``_CHUNK`` elements
(so an 8 GB cache never needs a 17 GB float32 staging copy).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

_CHUNK = 1 << 26


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                 # "f32" | "bf16"
    B: int
    Hq: int
    Hkv: int
    D: int
    Smax: int = 0              # dense / slot_ids capacity per row
    R: int = 0                 # dense rows (0: same as B)
    slot_ids: bool = False
    paged: bool = False
    num_blocks: int = 0
    block_size: int = 16
    max_blocks: int = 0
    len_lo: int = 1
    len_hi: int = 1
    len_dist: str = "uniform"  # "uniform" | "loguniform"
    stale_std: float = 1.0     # std of slots beyond the valid range
    key_scale: float = 1.0
    seed: int = 0
    notes: dict = field(default_factory=dict, compare=False)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def rows(self) -> int:
        return self.R if self.R else self.B

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


WORKLOADS = {
    "pr1_fp32": Workload("pr1_fp32", "f32", B=2, Hq=8, Hkv=2, D=64, Smax=256,
                         len_lo=1, len_hi=255, stale_std=100.0, seed=0),
    "llama3_8b": Workload("llama3_8b", "bf16", B=32, Hq=32, Hkv=8, D=128, Smax=4096,
                          len_lo=1024, len_hi=4095, seed=1),
    "long_context": Workload("long_context", "bf16", B=4, Hq=64, Hkv=8, D=128,
                             Smax=131072, len_lo=32768, len_hi=131071, key_scale=3.0, seed=2),
    "ragged_slots": Workload("ragged_slots", "bf16", B=256, Hq=32, Hkv=4, D=128, Smax=8192,
                             R=512, slot_ids=True, len_lo=16, len_hi=8191,
                             len_dist="loguniform", seed=3),
    "paged": Workload("paged", "bf16", B=64, Hq=48, Hkv=8, D=128, paged=True,
                      num_blocks=65536, block_size=16, max_blocks=1024,
                      len_lo=512, len_hi=16383, seed=4),
}


def small(name: str, **kw) -> Workload:
    """A workload of the given shape family, resized by keyword overrides."""
    return replace(WORKLOADS[name], **kw) if name in WORKLOADS else Workload(name, **kw)


def _normal(shape, gen, device, std=1.0, scale=1.0):
    n = math.prod(shape)
    flat = torch.empty(n, dtype=torch.float32, device=device)
    for i in range(0, n, _CHUNK):
        m = min(_CHUNK, n - i)
        flat[i:i + m] = torch.randn(m, generator=gen, device=device)
    if std * scale != 1.0:
        flat.mul_(std * scale)
    return flat.view(shape)


def _cast(x, w):
    return x if w.dtype == "f32" else x.to(torch.bfloat16)


def _normal_cast(shape, gen, device, w, scale=1.0):
    """N(0, scale^2) drawn chunk by chunk and cast to the workload dtype, so
    the float32 staging copy stays at one chunk."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=w.torch_dtype, device=device)
    for i in range(0, n, _CHUNK):
        m = min(_CHUNK, n - i)
        x = torch.randn(m, generator=gen, device=device)
        if scale != 1.0:
            x.mul_(scale)
        out[i:i + m] = x.to(w.torch_dtype)
    return out.view(shape)


def _lengths(w, gen, device):
    if w.len_dist == "uniform":
        return torch.randint(w.len_lo, w.len_hi + 1, (w.B,), generator=gen,
                             device=device, dtype=torch.int64).to(torch.int32)
    u = torch.rand(w.B, generator=gen, device=device, dtype=torch.float64)
    lo = max(w.len_lo, 1)
    x = torch.exp(math.log(lo) + u * (math.log(w.len_hi + 1) - math.log(lo)))
    return torch.floor(x).clamp(w.len_lo, w.len_hi).to(torch.int32)


def generate(w: Workload, device="cpu", attend: bool = False, q_f32: bool = False,
             q_lens=None, kv_e4m3: bool = False) -> dict:
    """All inputs of one decode step of workload ``w`` on ``device``.

    Returns a dict with q (B,Hq,D), k_new/v_new (B,Hkv,D), lengths (B,) int32,
    and either k_cache/v_cache (R,Hkv,Smax,D) [+ slot_ids (B,) int32] or
    k_blocks/v_blocks (num_blocks,Hkv,block_size,D) + block_table (B,max_blocks).
    With ``attend`` the inputs of the read-only attend instead (see the module
    docstring): lengths count valid slots and there is no k_new / v_new.
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    t = {}
    t["lengths"] = _lengths(w, gen, device)
    if attend:
        t["lengths"] = t["lengths"] + 1
    ntok = w.B
    if q_lens is not None:
        ql = torch.as_tensor(q_lens, dtype=torch.int64).to(device)
        cap = w.max_blocks * w.block_size if w.paged else w.Smax
        t["lengths"] = torch.minimum(t["lengths"].to(torch.int64), cap - ql).clamp(min=0).to(torch.int32)
        t["cu_q"] = torch.cat([torch.zeros(1, dtype=torch.int64, device=device), torch.cumsum(ql, 0)]).to(torch.int32)
        ntok = int(ql.sum().item())
    if q_f32:
        t["q"] = _normal((ntok, w.Hq, w.D), gen, device)
    else:
        t["q"] = _normal_cast((ntok, w.Hq, w.D), gen, device, w)
    t["k_new"] = _normal_cast((ntok, w.Hkv, w.D), gen, device, w, w.key_scale)
    t["v_new"] = _normal_cast((ntok, w.Hkv, w.D), gen, device, w)
    if w.paged:
        shape = (w.num_blocks, w.Hkv, w.block_size, w.D)
        t["k_blocks"] = _normal_cast(shape, gen, device, w, w.key_scale)
        t["v_blocks"] = _normal_cast(shape, gen, device, w)
        need = w.B * w.max_blocks
        if w.num_blocks < need:
            raise ValueError("the block-table recipe needs num_blocks >= B * max_blocks")
        perm = torch.randperm(w.num_blocks, generator=gen, device=device)[:need]
        bt = perm.view(w.B, w.max_blocks).to(torch.int32)
        # blocks holding the slots the call touches: 0..lengths[b] (decode), 0..lengths[b]-1 (attend)
        if q_lens is not None:
            touched = t["lengths"].to(torch.int64) + torch.as_tensor(q_lens, dtype=torch.int64).to(device)
        else:
            touched = t["lengths"].to(torch.int64) + (0 if attend else 1)
        used = (touched + w.block_size - 1) // w.block_size
        idx = torch.arange(w.max_blocks, device=device)[None, :]
        t["block_table"] = torch.where(idx < used[:, None], bt, torch.full_like(bt, -1))
        return quantise_cache(w, _drop_new(t, attend)) if kv_e4m3 else _drop_new(t, attend)
    shape = (w.rows, w.Hkv, w.Smax, w.D)
    if w.stale_std == 1.0:
        t["k_cache"] = _normal_cast(shape, gen, device, w, w.key_scale)
        t["v_cache"] = _normal_cast(shape, gen, device, w)
    else:
        valid_k = _normal(shape, gen, device, scale=w.key_scale)
        valid_v = _normal(shape, gen, device)
        stale_k = _normal(shape, gen, device, std=w.stale_std, scale=w.key_scale)
        stale_v = _normal(shape, gen, device, std=w.stale_std)
    if w.slot_ids:
        t["slot_ids"] = torch.randperm(w.rows, generator=gen, device=device)[:w.B].to(torch.int32)
    if w.stale_std != 1.0:
        # slots at or beyond each row's length hold large stale numbers
        row_len = torch.zeros(w.rows, dtype=torch.int64, device=device)
        rows = t["slot_ids"].to(torch.int64) if w.slot_ids else torch.arange(w.B, device=device)
        row_len[rows] = t["lengths"].to(torch.int64)
        valid = (torch.arange(w.Smax, device=device)[None, :] < row_len[:, None])[:, None, :, None]
        t["k_cache"] = _cast(torch.where(valid, valid_k, stale_k), w)
        t["v_cache"] = _cast(torch.where(valid, valid_v, stale_v), w)
    return quantise_cache(w, _drop_new(t, attend)) if kv_e4m3 else _drop_new(t, attend)


def _drop_new(t: dict, attend: bool) -> dict:
    if attend:
        del t["k_new"], t["v_new"]
    return t


def _to_e4m3(x, scale):
    """(N, Hkv, S, D) values as E4M3 bytes of x / scale[kvh] (chunked over N)."""
    out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    s = scale.view(1, -1, 1, 1)
    step = max(1, _CHUNK // max(1, x[0].numel()))
    for i in range(0, x.shape[0], step):
        y = (x[i:i + step].float() / s).clamp_(-448.0, 448.0)
        out[i:i + step] = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return out


def quantise_cache(w: Workload, t: dict, key_range: float = 4.0) -> dict:
    """The cache of ``t`` as E4M3 bytes with per-head scales (see the module
    docstring; ``key_range`` * key_scale is the largest key the scale
    represents, 4 sigma by default); the other inputs unchanged."""
    dev = t["q"].device
    ks = torch.full((w.Hkv,), key_range * w.key_scale / 448.0, dtype=torch.float32, device=dev)
    vs = torch.full((w.Hkv,), 4.0 / 448.0, dtype=torch.float32, device=dev)
    names = ("k_blocks", "v_blocks") if w.paged else ("k_cache", "v_cache")
    t[names[0]] = _to_e4m3(t[names[0]], ks)
    t[names[1]] = _to_e4m3(t[names[1]], vs)
    t["k_scale"], t["v_scale"] = ks, vs
    return t


def kv_bytes_read(w: Workload, lengths) -> int:
    """Bytes of cached K and V one step must read: sum_b lengths[b]*Hkv*D*2*es
    (the new token's K/V come from the inputs, not from the cache)."""
    total = int(torch.as_tensor(lengths).to(torch.int64).sum().item())
    return total * w.Hkv * w.D * 2 * w.elem_bytes


def expected_kv_bytes(w: Workload) -> float:
    """The same count at the mean of the length distribution."""
    if w.len_dist == "uniform":
        mean = (w.len_lo + w.len_hi) / 2
    else:
        a, b = math.log(w.len_lo), math.log(w.len_hi + 1)
        mean = (math.exp(b) - math.exp(a)) / (b - a) - 0.5
    return w.B * mean * w.Hkv * w.D * 2 * w.elem_bytes
