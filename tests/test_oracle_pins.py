"""Pins for the CPU oracle: values the pages print, closed forms, invariants,
library special cases and brute force. None of these re-types the oracle's
own formula; each checks it against something fixed outside it.

Pages:
  [P1] tensortonic "KV cache decode step" (cs336-l10): statement, Examples 1-3.
  [P2] tensortonic "Grouped-Query Decode Step" (JAX): statement, formula,
       Examples 1-3, Hints 1-3, Requirements, Constraints.
  [P5] clika runtime "groupQueryAttention": slot_ids and block-table rules.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import to_np, oracle_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------- page values

@pytest.mark.parametrize("ex", _golden("kv_cache_decode_step_examples.json")["examples"],
                         ids=lambda e: e["name"])
def test_p1_examples(ex):
    """[P1] Examples 1-3: output and both extended caches. The page's cache
    holds S positions and the new token goes to position S, so our cache has
    S+1 slots and lengths = S."""
    f = lambda x: np.asarray(x, dtype=np.float32)
    q, kn, vn = f(ex["query"]), f(ex["new_key"]), f(ex["new_value"])
    kc0, vc0 = f(ex["key_cache"]), f(ex["value_cache"])
    B, Hkv, S, D = kc0.shape
    assert q.shape[1] == ex["num_query_heads"] and Hkv == ex["num_kv_heads"]
    kc = np.zeros((B, Hkv, S + 1, D), np.float32)
    vc = np.zeros_like(kc)
    kc[:, :, :S], vc[:, :, :S] = kc0, vc0
    r = oracle.decode_dense(q, kn, vn, kc, vc, np.full(B, S, np.int32))
    assert r.status == oracle.OK
    np.testing.assert_allclose(r.out, ex["output"], rtol=0, atol=5e-7)
    np.testing.assert_allclose(kc, ex["new_key_cache"], rtol=0, atol=5e-7)
    np.testing.assert_allclose(vc, ex["new_value_cache"], rtol=0, atol=5e-7)
    # the appended slot holds exactly the new key's bits
    assert kc[:, :, S].tobytes() == kn.tobytes() and vc[:, :, S].tobytes() == vn.tobytes()


@pytest.mark.parametrize("ex", _golden("grouped_query_decode_step_examples.json")["examples"],
                         ids=lambda e: e["name"])
def test_p2_examples(ex):
    """[P2] Examples 1-3. The page's cache is slot-major (B,S,Hkv,D) and its
    lengths count the new token, which is already stored. Mapped here: the
    cache is transposed to (B,Hkv,S,D), our append slot is lengths-1 and the
    new key/value are that slot's contents, so the append rewrites the same
    bits and the output must be the page's."""
    q = np.asarray(ex["query"], np.float32)
    kc = np.ascontiguousarray(np.asarray(ex["key_cache"], np.float32).transpose(0, 2, 1, 3))
    vc = np.ascontiguousarray(np.asarray(ex["value_cache"], np.float32).transpose(0, 2, 1, 3))
    lens = np.asarray(ex["lengths"], np.int32)
    B = q.shape[0]
    kn = np.stack([kc[b, :, lens[b] - 1] for b in range(B)])
    vn = np.stack([vc[b, :, lens[b] - 1] for b in range(B)])
    before_k, before_v = kc.copy(), vc.copy()
    r = oracle.decode_dense(q, kn, vn, kc, vc, lens - 1)
    assert r.status == oracle.OK
    np.testing.assert_allclose(r.out, ex["output"], rtol=0, atol=5e-7)
    assert kc.tobytes() == before_k.tobytes() and vc.tobytes() == before_v.tobytes()


def test_p2_example1_weights():
    """[P2] Example 1 explanation prints head 0's weights 0.669762/0.330238:
    with V = identity rows, the output is the weight vector itself."""
    q = np.array([[[1, 0]]], np.float32)
    kc = np.array([[[[1, 0], [0, 1], [5, 5]]]], np.float32)
    vc = np.array([[[[1, 0], [0, 1], [50, 50]]]], np.float32)
    r = oracle.decode_dense(q, kc[:, :, 1].copy(), vc[:, :, 1].copy(), kc, vc,
                            np.array([1], np.int32))
    np.testing.assert_allclose(r.out[0, 0], [0.669762, 0.330238], atol=5e-7)


# ---------------------------------------------------------------- bf16 format

def test_bf16_widening_matches_format():
    """bf16 is the top half of binary32: 0x3F80 = 1, 0xC000 = -2,
    0x3F81 = 1 + 2^-7, 0x0001 = 2^-133 (subnormal). A one-slot cache returns
    the new value exactly, so the oracle's widening shows through."""
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0001], np.uint16)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 2.0 ** -133]
    q = np.zeros((1, 1, 4), np.uint16)
    k = np.zeros((1, 1, 4), np.uint16)
    v = bits.reshape(1, 1, 4).copy()
    kc = np.zeros((1, 1, 1, 4), np.uint16)
    vc = np.zeros_like(kc)
    r = oracle.decode_dense(q, k, v, kc, vc, np.array([0], np.int32))
    assert list(r.out[0, 0]) == want


def test_bf16_agrees_with_f32_on_representable_values():
    """On values exactly representable in bf16, the bf16 and f32 branches of
    the oracle must give bit-identical float64 outputs."""
    w = W.small("llama3_8b", B=3, Hq=8, Hkv=2, D=16, Smax=24, len_lo=0, len_hi=23, seed=11)
    t = W.generate(w)
    tb = oracle_inputs(t)
    tf = {k: (to_np(v.float()) if v.dtype == torch.bfloat16 else to_np(v)) for k, v in t.items()}
    rb = oracle.decode_dense(tb["q"], tb["k_new"], tb["v_new"], tb["k_cache"], tb["v_cache"], tb["lengths"])
    rf = oracle.decode_dense(tf["q"], tf["k_new"], tf["v_new"], tf["k_cache"], tf["v_cache"], tf["lengths"])
    assert rb.out.tobytes() == rf.out.tobytes()


# --------------------------------------------------------------- brute force

def _brute_force(q, kc, vc, kn, vn, lens, slot_ids=None):
    """Direct softmax without max subtraction, pure Python, on tiny shapes:
    w_j = e^{s_j} / sum_m e^{s_m}  ([P2] formula, literally)."""
    B, Hq, D = q.shape
    Hkv = kc.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for b in range(B):
        r = b if slot_ids is None else int(slot_ids[b])
        L = int(lens[b])
        for h in range(Hq):
            g = h // G
            keys = [[float(x) for x in kc[r, g, j]] for j in range(L)] + [[float(x) for x in kn[b, g]]]
            vals = [[float(x) for x in vc[r, g, j]] for j in range(L)] + [[float(x) for x in vn[b, g]]]
            qs = [float(x) for x in q[b, h]]
            e = [math.exp(sum(a * c for a, c in zip(qs, k)) / math.sqrt(D)) for k in keys]
            z = sum(e)
            for d in range(D):
                out[b, h, d] = sum(e[j] * vals[j][d] for j in range(L + 1)) / z
    return out


@pytest.mark.parametrize("seed", range(12))
def test_brute_force_tiny(seed):
    """Random tiny cases within the [P2] Constraints (B 1-3, S 3-8, Hq 2-8,
    D 2-4, Hkv | Hq, lengths in range, stale slots much larger)."""
    rng = np.random.default_rng(seed)
    B, S, D = rng.integers(1, 4), rng.integers(3, 9), rng.integers(2, 5)
    Hq = int(rng.choice([2, 3, 4, 6, 8]))
    Hkv = int(rng.choice([d for d in range(1, Hq + 1) if Hq % d == 0]))
    lens = rng.integers(0, S, size=B).astype(np.int32)
    q = rng.normal(size=(B, Hq, D)).astype(np.float32)
    kc = (rng.normal(size=(B, Hkv, S, D)) * 50).astype(np.float32)
    vc = (rng.normal(size=(B, Hkv, S, D)) * 50).astype(np.float32)
    for b in range(B):
        kc[b, :, :lens[b]] /= 50
        vc[b, :, :lens[b]] /= 50
    kn = rng.normal(size=(B, Hkv, D)).astype(np.float32)
    vn = rng.normal(size=(B, Hkv, D)).astype(np.float32)
    want = _brute_force(q, kc, vc, kn, vn, lens)
    r = oracle.decode_dense(q, kn, vn, kc, vc, lens)
    np.testing.assert_allclose(r.out, want, rtol=1e-12, atol=1e-12)


def test_einsum_mask_formulation():
    """[P2] Hints 1-3 (reshape by cache head, einsum against a slot-major
    cache, fixed-shape mask) written in numpy float64, against the oracle."""
    rng = np.random.default_rng(5)
    B, S, Hq, Hkv, D = 3, 8, 8, 2, 4
    G = Hq // Hkv
    q = rng.normal(size=(B, Hq, D)).astype(np.float32)
    kc = rng.normal(size=(B, Hkv, S, D)).astype(np.float32)
    vc = rng.normal(size=(B, Hkv, S, D)).astype(np.float32)
    lens = np.array([0, 4, 7], np.int32)
    kn = rng.normal(size=(B, Hkv, D)).astype(np.float32)
    vn = rng.normal(size=(B, Hkv, D)).astype(np.float32)
    k_ext, v_ext = kc.astype(np.float64), vc.astype(np.float64)
    for b in range(B):
        k_ext[b, :, lens[b]] = kn[b]
        v_ext[b, :, lens[b]] = vn[b]
    keys = k_ext.transpose(0, 2, 1, 3)                      # (B,S,Hkv,D)
    vals = v_ext.transpose(0, 2, 1, 3)
    qg = q.astype(np.float64).reshape(B, Hkv, G, D)
    s = np.einsum("bkgd,bskd->bkgs", qg, keys) / np.sqrt(D)
    mask = np.arange(S)[None, :] < (lens + 1)[:, None]
    s = np.where(mask[:, None, None, :], s, -np.inf)
    w = np.exp(s - s.max(-1, keepdims=True))
    w /= w.sum(-1, keepdims=True)
    o = np.einsum("bkgs,bskd->bkgd", w, vals).reshape(B, Hq, D)
    r = oracle.decode_dense(q, kn, vn, kc.copy(), vc.copy(), lens)
    np.testing.assert_allclose(r.out, o, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (6, 1)])
def test_library_sdpa(Hq, Hkv):
    """torch's scaled_dot_product_attention in float64 on the valid prefix,
    with each cache head repeated for its G query heads: covers MHA (G=1),
    GQA and MQA (Hkv=1)."""
    w = W.small("llama3_8b", dtype="f32", B=3, Hq=Hq, Hkv=Hkv, D=32, Smax=40,
                len_lo=0, len_hi=39, seed=21)
    t = W.generate(w)
    a = oracle_inputs(t)
    r = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"], a["v_cache"], a["lengths"])
    G = Hq // Hkv
    for b in range(w.B):
        L = int(t["lengths"][b])
        k = torch.cat([t["k_cache"][b, :, :L], t["k_new"][b, :, None]], 1).double()
        v = torch.cat([t["v_cache"][b, :, :L], t["v_new"][b, :, None]], 1).double()
        k = k.repeat_interleave(G, 0)
        v = v.repeat_interleave(G, 0)
        o = torch.nn.functional.scaled_dot_product_attention(
            t["q"][b][:, None].double(), k, v)[:, 0]
        np.testing.assert_allclose(r.out[b], o.numpy(), rtol=1e-12, atol=1e-12)


# -------------------------------------------------------------- closed forms

def _rand_case(seed, dtype="f32", **kw):
    base = dict(B=3, Hq=8, Hkv=2, D=16, Smax=32, len_lo=0, len_hi=31, seed=seed)
    base.update(kw)
    w = W.small("llama3_8b", dtype=dtype, **base)
    return w, oracle_inputs(W.generate(w))


def test_identical_keys_give_mean_of_values():
    """[P1] Example 1's explanation, generalised: identical keys -> mean."""
    w, a = _rand_case(1)
    a["k_cache"][:] = a["k_cache"][:, :, :1]
    a["k_new"][:] = a["k_cache"][:, :, 0]
    r = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"], a["v_cache"], a["lengths"])
    for b in range(w.B):
        L = int(a["lengths"][b])
        mean = a["v_cache"][b, :, :L + 1].astype(np.float64).mean(1)   # after append
        np.testing.assert_allclose(r.out[b], np.repeat(mean, w.G, 0), rtol=1e-12, atol=1e-12)


def test_zero_query_uniform_weights():
    """[P1] Example 2 / [P2] Example 3 head 0: equal scores -> uniform."""
    w, a = _rand_case(2)
    a["q"][:] = 0
    r = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"], a["v_cache"], a["lengths"])
    for b in range(w.B):
        L = int(a["lengths"][b])
        mean = a["v_cache"][b, :, :L + 1].astype(np.float64).mean(1)
        np.testing.assert_allclose(r.out[b], np.repeat(mean, w.G, 0), rtol=1e-12, atol=1e-12)


def test_empty_cache_returns_new_value():
    """[P2] Example 2 row 1: one valid slot -> output is that value exactly."""
    w, a = _rand_case(3)
    a["lengths"][:] = 0
    r = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"], a["v_cache"], a["lengths"])
    want = np.repeat(a["v_new"].astype(np.float64), w.G, 1)
    assert np.array_equal(r.out, want)


def test_weights_sum_to_one():
    """sum_j w_j = 1: with every value vector all ones the output is 1."""
    w, a = _rand_case(4)
    a["v_cache"][:] = 1
    a["v_new"][:] = 1
    r = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"], a["v_cache"], a["lengths"])
    np.testing.assert_allclose(r.out, 1.0, rtol=0, atol=1e-14)


def test_value_shift():
    """o(V + c) = o(V) + c, because the weights sum to one."""
    w, a = _rand_case(5)
    r0 = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(), a["v_cache"].copy(), a["lengths"])
    c = np.float32(2.0)
    r1 = oracle.decode_dense(a["q"], a["k_new"], a["v_new"] + c, a["k_cache"].copy(), a["v_cache"] + c, a["lengths"])
    np.testing.assert_allclose(r1.out, r0.out + 2.0, rtol=0, atol=1e-6)


def test_key_query_rescale():
    """Scores use q.K only: K*alpha with q/alpha leaves the output unchanged
    (alpha a power of two, so the rescaled inputs are exact)."""
    w, a = _rand_case(6)
    r0 = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(), a["v_cache"].copy(), a["lengths"])
    r1 = oracle.decode_dense(a["q"] / 4, a["k_new"] * 4, a["v_new"], a["k_cache"] * 4, a["v_cache"].copy(), a["lengths"])
    assert np.array_equal(r0.out, r1.out)


def test_scale_is_inverse_sqrt_d():
    """s = q.K / sqrt(D): two slots, keys chosen so q.K = sqrt(D)*ln 3 and 0;
    weights 3/4 and 1/4 exactly (D = 16, sqrt(D) = 4)."""
    D = 16
    q = np.zeros((1, 1, D), np.float32); q[0, 0, 0] = 1
    kc = np.zeros((1, 1, 2, D), np.float32)
    kc[0, 0, 0, 0] = 4 * math.log(3)
    vc = np.zeros_like(kc); vc[0, 0, 0, 0] = 1
    kn = np.zeros((1, 1, D), np.float32)
    vn = np.zeros((1, 1, D), np.float32); vn[0, 0, 1] = 1
    r = oracle.decode_dense(q, kn, vn, kc, vc, np.array([1], np.int32))
    e = math.exp(float(np.float32(4 * math.log(3))) / 4)
    np.testing.assert_allclose(r.out[0, 0, :2], [e / (e + 1), 1 / (e + 1)], rtol=1e-15)
    np.testing.assert_allclose(r.out[0, 0, :2], [0.75, 0.25], atol=1e-7)


def test_group_mapping_is_contiguous():
    """Query head h reads cache head floor(h/G) ([P2] statement): give each
    cache head a distinct constant value and read it back per query head."""
    B, Hq, Hkv, D, S = 1, 8, 4, 4, 5
    q = np.random.default_rng(0).normal(size=(B, Hq, D)).astype(np.float32)
    kc = np.random.default_rng(1).normal(size=(B, Hkv, S, D)).astype(np.float32)
    vc = np.zeros((B, Hkv, S, D), np.float32)
    for g in range(Hkv):
        vc[:, g] = g + 1
    kn = np.zeros((B, Hkv, D), np.float32)
    vn = vc[:, :, 0].copy()
    r = oracle.decode_dense(q, kn, vn, kc, vc, np.array([3], np.int32))
    for h in range(Hq):
        np.testing.assert_allclose(r.out[0, h], h // (Hq // Hkv) + 1, atol=1e-14)


# ---------------------------------------------------------------- invariants

def test_stale_slots_cannot_matter():
    """[P2]: slots at or beyond the length get zero weight. Fill them with
    other numbers, Inf and NaN: the output must not change by a single bit."""
    w, a = _rand_case(7)
    r0 = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(), a["v_cache"].copy(), a["lengths"])
    for fill in (1e30, np.inf, np.nan):
        kc, vc = a["k_cache"].copy(), a["v_cache"].copy()
        for b in range(w.B):
            kc[b, :, a["lengths"][b]:] = fill
            vc[b, :, a["lengths"][b]:] = -fill
        r1 = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], kc, vc, a["lengths"])
        assert r1.out.tobytes() == r0.out.tobytes()


def test_slot_permutation():
    """The softmax is a sum over slots: reordering the cached slots changes
    the output by rounding only."""
    w, a = _rand_case(8)
    r0 = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(), a["v_cache"].copy(), a["lengths"])
    kc, vc = a["k_cache"].copy(), a["v_cache"].copy()
    rng = np.random.default_rng(0)
    for b in range(w.B):
        L = int(a["lengths"][b])
        p = rng.permutation(L)
        kc[b, :, :L] = kc[b][:, p]
        vc[b, :, :L] = vc[b][:, p]
    r1 = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], kc, vc, a["lengths"])
    np.testing.assert_allclose(r1.out, r0.out, rtol=1e-12, atol=1e-13)


def test_append_touches_one_slot_per_row_head():
    """In-place append ([P5] description): afterwards the cache equals the old
    cache with exactly slot lengths[b] of each (row, head) replaced by the new
    key/value bits; every other byte, and every unused row, is unchanged."""
    w = W.small("ragged_slots", dtype="bf16", B=4, R=7, Hq=8, Hkv=2, D=16, Smax=20,
                len_lo=1, len_hi=19, seed=9)
    a = oracle_inputs(W.generate(w))
    kc, vc = a["k_cache"].copy(), a["v_cache"].copy()
    oracle.decode_dense(a["q"], a["k_new"], a["v_new"], kc, vc, a["lengths"], a["slot_ids"])
    want_k, want_v = a["k_cache"].copy(), a["v_cache"].copy()
    for b in range(w.B):
        r, L = a["slot_ids"][b], a["lengths"][b]
        want_k[r, :, L] = a["k_new"][b]
        want_v[r, :, L] = a["v_new"][b]
    assert kc.tobytes() == want_k.tobytes() and vc.tobytes() == want_v.tobytes()


def test_slot_ids_is_a_row_map():
    """[P5] slot_ids names the cache row of each batch row: the same data laid
    out row b -> row slot_ids[b] gives the bit-identical output."""
    w = W.small("ragged_slots", dtype="f32", B=4, R=9, Hq=8, Hkv=4, D=8, Smax=16,
                len_lo=0, len_hi=15, seed=10)
    a = oracle_inputs(W.generate(w))
    sid = a["slot_ids"]
    dense_k = np.ascontiguousarray(a["k_cache"][sid])
    dense_v = np.ascontiguousarray(a["v_cache"][sid])
    r0 = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], dense_k, dense_v, a["lengths"])
    r1 = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"], a["v_cache"], a["lengths"], sid)
    assert r0.out.tobytes() == r1.out.tobytes()
    assert np.array_equal(dense_k, a["k_cache"][sid])


@pytest.mark.parametrize("block_size", [1, 4, 16])
def test_paged_equals_dense(block_size):
    """A paged cache with the same logical content as a dense one gives the
    bit-identical output, and the append lands in block bt[b][L/bs] at
    offset L%bs; unused blocks are never read (NaN-filled here)."""
    max_blocks = 20 // block_size + 1
    w = W.small("paged", dtype="bf16", B=3, Hq=6, Hkv=2, D=8, num_blocks=3 * max_blocks + 5,
                block_size=block_size, max_blocks=max_blocks, len_lo=0, len_hi=19, seed=12)
    a = oracle_inputs(W.generate(w))
    bt, lens, bs = a["block_table"], a["lengths"], block_size
    Smax = w.max_blocks * bs
    dense_k = np.zeros((w.B, w.Hkv, Smax, w.D), np.uint16)
    dense_v = np.zeros_like(dense_k)
    for b in range(w.B):
        for s in range(Smax):
            blk = bt[b, s // bs]
            if blk >= 0:
                dense_k[b, :, s] = a["k_blocks"][blk, :, s % bs]
                dense_v[b, :, s] = a["v_blocks"][blk, :, s % bs]
    used = set(bt[bt >= 0].tolist())
    kb, vb = a["k_blocks"].copy(), a["v_blocks"].copy()
    for blk in range(w.num_blocks):
        if blk not in used:
            kb[blk] = 0x7FC0   # bf16 NaN
            vb[blk] = 0x7FC0
    r0 = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], dense_k, dense_v, lens)
    kb0 = kb.copy()
    r1 = oracle.decode_paged(a["q"], a["k_new"], a["v_new"], kb, vb, bt, lens)
    assert r1.status == oracle.OK
    assert r0.out.tobytes() == r1.out.tobytes()
    for b in range(w.B):
        L = lens[b]
        blk = bt[b, L // bs]
        assert kb[blk, :, L % bs].tobytes() == a["k_new"][b].tobytes()
        kb[blk, :, L % bs] = kb0[blk, :, L % bs]
    assert kb.tobytes() == kb0.tobytes()


def test_rows_subset_matches_full():
    """Computing only some batch rows gives those rows' full-run values."""
    w, a = _rand_case(13, B=5)
    r_all = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(), a["v_cache"].copy(), a["lengths"])
    r_sub = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(), a["v_cache"].copy(), a["lengths"],
                                rows=[4, 1], append=False)
    assert r_sub.out[[1, 4]].tobytes() == r_all.out[[1, 4]].tobytes()
    assert np.isnan(r_sub.out[[0, 2, 3]]).all()


def test_threads_do_not_change_bits():
    w, a = _rand_case(14, B=4)
    r1 = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(), a["v_cache"].copy(), a["lengths"], threads=1)
    r8 = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(), a["v_cache"].copy(), a["lengths"], threads=8)
    assert r1.out.tobytes() == r8.out.tobytes()


# ----------------------------------------------------------------- validation

def test_validate_dense_rules():
    """[P5]: slot_ids entries in [0, max_seqs), no two rows sharing one; our
    reading: 0 <= lengths[b] <= Smax-1, and R >= B without slot_ids."""
    L = np.array([0, 5, 9], np.int32)
    assert oracle.validate_dense(L, None, 3, 10) == oracle.OK
    assert oracle.validate_dense(L, None, 2, 10) == oracle.INVALID_ARGUMENT     # R < B
    assert oracle.validate_dense(np.array([0, 5, 10], np.int32), None, 3, 10) == oracle.INVALID_ARGUMENT
    assert oracle.validate_dense(np.array([-1, 5, 9], np.int32), None, 3, 10) == oracle.INVALID_ARGUMENT
    assert oracle.validate_dense(L, np.array([4, 0, 2], np.int32), 5, 10) == oracle.OK
    assert oracle.validate_dense(L, np.array([4, 0, 4], np.int32), 5, 10) == oracle.INVALID_ARGUMENT
    assert oracle.validate_dense(L, np.array([4, 0, 5], np.int32), 5, 10) == oracle.INVALID_ARGUMENT
    assert oracle.validate_dense(L, np.array([4, -1, 2], np.int32), 5, 10) == oracle.INVALID_ARGUMENT


def test_validate_paged_rules():
    """[P5]: every entry -1 or in [0, num_blocks), no repeats within a row;
    our reading: the blocks holding slots 0..lengths[b] must be real."""
    bt = np.array([[3, 1, -1, -1], [0, 2, 5, -1]], np.int32)
    L = np.array([7, 11], np.int32)          # block size 4: needs 2 and 3 blocks
    ok = lambda t, l=L: oracle.validate_paged(l, t, 6, 4)
    assert ok(bt) == oracle.OK
    bad = bt.copy(); bad[1, 3] = 6
    assert ok(bad) == oracle.INVALID_ARGUMENT                 # out of range
    bad = bt.copy(); bad[1, 3] = -2
    assert ok(bad) == oracle.INVALID_ARGUMENT                 # negative, not -1
    bad = bt.copy(); bad[1, 2] = 0
    assert ok(bad) == oracle.INVALID_ARGUMENT                 # repeat in a row
    rep = bt.copy(); rep[1, 3] = 3
    assert ok(rep) == oracle.OK                               # a block in two rows is allowed
    assert ok(bt, np.array([8, 11], np.int32)) == oracle.INVALID_ARGUMENT   # slot 8 needs entry 2 (-1)
    assert ok(bt, np.array([7, 16], np.int32)) == oracle.INVALID_ARGUMENT   # beyond max_blocks*bs
    # a failed validation means no append and no output
    q = np.zeros((2, 2, 4), np.float32)
    kb = np.zeros((6, 1, 4, 4), np.float32)
    bad = bt.copy(); bad[0, 1] = 3
    r = oracle.decode_paged(q, np.ones((2, 1, 4), np.float32), np.ones((2, 1, 4), np.float32),
                            kb, kb.copy(), bad, L)
    assert r.status == oracle.INVALID_ARGUMENT and not kb.any()


# ------------------------------------------------- read-only attend (no append)
#
# [P2] is itself the read-only form: its lengths count the valid slots (the
# new token already stored among them), the query is float32 and the caches
# float32 or bfloat16. [P5]'s attention_over_cache reads the cache and
# writes nothing.

def _to_bf16_bits_exact(a):
    """float32 array -> bf16 bit pattern; asserts every value is representable."""
    a = np.ascontiguousarray(a, np.float32)
    bits = (a.view(np.uint32) >> 16).astype(np.uint16)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(back, a), "value not exactly representable in bfloat16"
    return bits


@pytest.mark.parametrize("cache_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ex", _golden("grouped_query_decode_step_examples.json")["examples"],
                         ids=lambda e: e["name"])
def test_p2_examples_attend(ex, cache_dtype):
    """[P2] Examples 1-3 in the page's own contract: lengths as printed,
    float32 query, the cache transposed to (B,Hkv,S,D). Every value printed in
    the examples is exact in bfloat16, so a bfloat16 cache must give the same
    outputs; nothing is written."""
    q = np.asarray(ex["query"], np.float32)
    kc = np.ascontiguousarray(np.asarray(ex["key_cache"], np.float32).transpose(0, 2, 1, 3))
    vc = np.ascontiguousarray(np.asarray(ex["value_cache"], np.float32).transpose(0, 2, 1, 3))
    if cache_dtype == "bf16":
        kc, vc = _to_bf16_bits_exact(kc), _to_bf16_bits_exact(vc)
    before = kc.tobytes() + vc.tobytes()
    r = oracle.attend_dense(q, kc, vc, np.asarray(ex["lengths"], np.int32))
    assert r.status == oracle.OK
    np.testing.assert_allclose(r.out, ex["output"], rtol=0, atol=5e-7)
    assert kc.tobytes() + vc.tobytes() == before


def _attend_brute(q, kc, vc, lens):
    """[P2] formula literally, pure Python: w_j = e^{s_j} / sum_m e^{s_m} over
    the slots j < lengths[b]."""
    B, Hq, D = q.shape
    G = Hq // kc.shape[1]
    out = np.zeros((B, Hq, D))
    for b in range(B):
        n = int(lens[b])
        for h in range(Hq):
            qs = [float(x) for x in q[b, h]]
            e = [math.exp(sum(a * float(c) for a, c in zip(qs, kc[b, h // G, j])) / math.sqrt(D))
                 for j in range(n)]
            z = sum(e)
            for d in range(D):
                out[b, h, d] = sum(e[j] * float(vc[b, h // G, j, d]) for j in range(n)) / z
    return out


@pytest.mark.parametrize("seed", range(8))
def test_attend_brute_force_tiny(seed):
    """Random tiny cases within the [P2] Constraints (B 1-3, S 3-8, Hq 2-8,
    D 2-4, Hkv | Hq, 1 <= lengths <= S, stale slots much larger)."""
    rng = np.random.default_rng(100 + seed)
    B, S, D = rng.integers(1, 4), rng.integers(3, 9), rng.integers(2, 5)
    Hq = int(rng.choice([2, 3, 4, 6, 8]))
    Hkv = int(rng.choice([d for d in range(1, Hq + 1) if Hq % d == 0]))
    lens = rng.integers(1, S + 1, size=B).astype(np.int32)
    q = rng.normal(size=(B, Hq, D)).astype(np.float32)
    kc = (rng.normal(size=(B, Hkv, S, D)) * 50).astype(np.float32)
    vc = (rng.normal(size=(B, Hkv, S, D)) * 50).astype(np.float32)
    for b in range(B):
        kc[b, :, :lens[b]] /= 50
        vc[b, :, :lens[b]] /= 50
    r = oracle.attend_dense(q, kc, vc, lens)
    np.testing.assert_allclose(r.out, _attend_brute(q, kc, vc, lens), rtol=1e-12, atol=1e-12)


def test_attend_float32_query_over_bf16_cache_library_sdpa():
    """[P2] Requirements: a float32 query over bfloat16 caches widened to
    float32. torch's scaled_dot_product_attention in float64 on the widened
    valid prefix must agree; the query carries bits below bfloat16's
    precision, so an oracle that rounded it would be off by ~1e-3."""
    w = W.small("llama3_8b", dtype="bf16", B=3, Hq=8, Hkv=2, D=32, Smax=40,
                len_lo=1, len_hi=39, seed=31)
    t = W.generate(w)
    q32 = torch.randn(w.B, w.Hq, w.D, generator=torch.Generator().manual_seed(5)) * (1 + 2 ** -12)
    lens = t["lengths"] + 1                   # valid-slot counts in [2, 40]
    a = oracle_inputs(t)
    r = oracle.attend_dense(to_np(q32), a["k_cache"], a["v_cache"], to_np(lens))
    assert r.status == oracle.OK
    G = w.Hq // w.Hkv
    for b in range(w.B):
        n = int(lens[b])
        k = t["k_cache"][b, :, :n].double().repeat_interleave(G, 0)
        v = t["v_cache"][b, :, :n].double().repeat_interleave(G, 0)
        o = torch.nn.functional.scaled_dot_product_attention(q32[b][:, None].double(), k, v)[:, 0]
        np.testing.assert_allclose(r.out[b], o.numpy(), rtol=1e-12, atol=1e-12)
        qr = q32[b].to(torch.bfloat16).double()
        o_rounded = torch.nn.functional.scaled_dot_product_attention(qr[:, None], k, v)[:, 0]
        assert np.abs(r.out[b] - o_rounded.numpy()).max() > 1e-6


def test_attend_single_slot_returns_value():
    """[P2] Example 2 row 1: one valid slot -> every head returns its value."""
    w, a = _rand_case(32)
    lens = np.ones(w.B, np.int32)
    r = oracle.attend_dense(a["q"], a["k_cache"], a["v_cache"], lens)
    want = np.repeat(a["v_cache"][:, :, 0].astype(np.float64), w.G, 1)
    assert np.array_equal(r.out, want)


def test_attend_stale_slots_cannot_matter():
    """[P2]: slot lengths[b] and beyond get zero weight, whatever they hold."""
    w, a = _rand_case(33)
    lens = a["lengths"] + 1
    r0 = oracle.attend_dense(a["q"], a["k_cache"], a["v_cache"], lens)
    for fill in (1e30, np.inf, np.nan):
        kc, vc = a["k_cache"].copy(), a["v_cache"].copy()
        for b in range(w.B):
            kc[b, :, lens[b]:] = fill
            vc[b, :, lens[b]:] = -fill
        assert oracle.attend_dense(a["q"], kc, vc, lens).out.tobytes() == r0.out.tobytes()


def test_attend_paged_equals_dense_and_slot_ids():
    """The same logical content through a paged table, through slot_ids and
    densely gives bit-identical outputs; unused blocks (NaN) are never read."""
    bs, max_blocks = 4, 6
    w = W.small("paged", dtype="bf16", B=3, Hq=8, Hkv=2, D=8, num_blocks=24, block_size=bs,
                max_blocks=max_blocks, len_lo=0, len_hi=22, seed=34)
    a = oracle_inputs(W.generate(w))
    bt = a["block_table"]
    lens = a["lengths"] + 1
    Smax = max_blocks * bs
    dense_k = np.zeros((w.B, w.Hkv, Smax, w.D), np.uint16)
    dense_v = np.zeros_like(dense_k)
    for b in range(w.B):
        for s in range(Smax):
            if bt[b, s // bs] >= 0:
                dense_k[b, :, s] = a["k_blocks"][bt[b, s // bs], :, s % bs]
                dense_v[b, :, s] = a["v_blocks"][bt[b, s // bs], :, s % bs]
    used = set(bt[bt >= 0].tolist())
    kb, vb = a["k_blocks"].copy(), a["v_blocks"].copy()
    for blk in range(w.num_blocks):
        if blk not in used:
            kb[blk] = vb[blk] = 0x7FC0
    r0 = oracle.attend_dense(a["q"], dense_k, dense_v, lens)
    r1 = oracle.attend_paged(a["q"], kb, vb, bt, lens)
    assert r1.status == oracle.OK and r0.out.tobytes() == r1.out.tobytes()
    sid = np.array([4, 0, 2], np.int32)
    rows_k = np.full((5, w.Hkv, Smax, w.D), 0x7FC0, np.uint16)
    rows_v = rows_k.copy()
    rows_k[sid], rows_v[sid] = dense_k, dense_v
    r2 = oracle.attend_dense(a["q"], rows_k, rows_v, lens, sid)
    assert r2.out.tobytes() == r0.out.tobytes()


def test_attend_validate_rules():
    """Our reading of [P2] Constraints for the read-only attend: 1 <= lengths
    <= Smax (zero valid slots has no softmax); paged, the entries holding
    slots 0..lengths[b]-1 must be real; [P5] slot_ids rules unchanged."""
    ok = oracle.OK
    bad = oracle.INVALID_ARGUMENT
    assert oracle.validate_attend_dense(np.array([1, 10], np.int32), None, 2, 10) == ok
    assert oracle.validate_attend_dense(np.array([0, 10], np.int32), None, 2, 10) == bad
    assert oracle.validate_attend_dense(np.array([1, 11], np.int32), None, 2, 10) == bad
    assert oracle.validate_attend_dense(np.array([1, 2], np.int32), np.array([3, 3], np.int32), 4, 10) == bad
    bt = np.array([[3, -1, -1], [0, 2, -1]], np.int32)
    assert oracle.validate_attend_paged(np.array([4, 8], np.int32), bt, 6, 4) == ok    # exactly full blocks
    assert oracle.validate_attend_paged(np.array([5, 8], np.int32), bt, 6, 4) == bad   # slot 4 needs entry 1
    assert oracle.validate_attend_paged(np.array([4, 0], np.int32), bt, 6, 4) == bad
    assert oracle.validate_attend_paged(np.array([4, 13], np.int32), bt, 6, 4) == bad  # beyond the table
    # the decode step's reading of the same numbers differs by one slot
    assert oracle.validate_paged(np.array([4, 7], np.int32), bt, 6, 4) == bad          # slot 4 for the append
    r = oracle.attend_dense(np.zeros((1, 1, 2), np.float32), np.zeros((1, 1, 3, 2), np.float32),
                            np.zeros((1, 1, 3, 2), np.float32), np.array([0], np.int32))
    assert r.status == bad and np.isnan(r.out).all()


# ------------------------------------------- softmax modifiers (sink, window)
#
# [P5] groupQueryAttention: head_sink is a per-head virtual logit folded into
# the softmax denominator; kept_prefix keeps the first P keys attended beside
# the sliding window (a key is attended when it is inside the first P keys or
# inside the window; the window alone without P); a negative P is refused.
# Readings: the window holds the W positions ending at the query's own; the
# sink is in the units of the scaled scores.

def _mods_case(seed, **kw):
    base = dict(B=3, Hq=8, Hkv=2, D=16, Smax=40, len_lo=5, len_hi=39, seed=seed)
    base.update(kw)
    w = W.small("llama3_8b", dtype="f32", **base)
    return w, oracle_inputs(W.generate(w))


def _mods_brute(q, kc, vc, kn, vn, lens, sink, window, prefix):
    """[P5] rules and the softmax, literally, in pure Python on tiny shapes:
    w_j = e^{s_j} / (e^{sink_h} + sum over attended slots e^{s_i})."""
    B, Hq, D = q.shape
    G = Hq // kc.shape[1]
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(lens[b])
        P = int(prefix[b]) if np.ndim(prefix) else int(prefix)
        keep = [j for j in range(L + 1) if window == 0 or j > L - window or j < P]
        for h in range(Hq):
            g = h // G
            qs = [float(x) for x in q[b, h]]
            key = lambda j: kn[b, g] if j == L else kc[b, g, j]
            val = lambda j: vn[b, g] if j == L else vc[b, g, j]
            e = {j: math.exp(sum(a * float(c) for a, c in zip(qs, key(j))) / math.sqrt(D)) for j in keep}
            z = sum(e.values()) + (math.exp(float(sink[h])) if sink is not None else 0.0)
            for d in range(D):
                out[b, h, d] = sum(e[j] * float(val(j)[d]) for j in keep) / z
    return out


@pytest.mark.parametrize("seed", range(6))
def test_mods_brute_force_tiny(seed):
    rng = np.random.default_rng(300 + seed)
    B, S, D, Hq, Hkv = 3, 12, 4, 4, 2
    lens = rng.integers(0, S, size=B).astype(np.int32)
    q = rng.normal(size=(B, Hq, D)).astype(np.float32)
    kc = rng.normal(size=(B, Hkv, S, D)).astype(np.float32)
    vc = rng.normal(size=(B, Hkv, S, D)).astype(np.float32)
    kn = rng.normal(size=(B, Hkv, D)).astype(np.float32)
    vn = rng.normal(size=(B, Hkv, D)).astype(np.float32)
    sink = rng.normal(size=Hq).astype(np.float32) * 2 if seed % 2 == 0 else None
    window = int(rng.integers(1, 6))
    prefix = rng.integers(0, 4, size=B).astype(np.int32) if seed % 3 else int(rng.integers(0, 3))
    r = oracle.decode_dense(q, kn, vn, kc.copy(), vc.copy(), lens, sink=sink, window=window,
                            kept_prefix=prefix)
    assert r.status == oracle.OK
    want = _mods_brute(q, kc, vc, kn, vn, lens, sink, window, prefix)
    np.testing.assert_allclose(r.out, want, rtol=1e-12, atol=1e-12)


def test_sink_as_virtual_key_library_sdpa():
    """A sink logit equals one more key per query head whose score is the sink
    and whose value is zero: torch SDPA in float64 on the valid slots plus that
    virtual key must agree with the oracle's sink."""
    w, a = _mods_case(41)
    sink = np.linspace(-2, 3, w.Hq).astype(np.float32)
    r = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(), a["v_cache"].copy(),
                            a["lengths"], sink=sink)
    G = w.G
    for b in range(w.B):
        L = int(a["lengths"][b])
        k = torch.cat([torch.from_numpy(a["k_cache"][b, :, :L]), torch.from_numpy(a["k_new"][b])[:, None]], 1)
        v = torch.cat([torch.from_numpy(a["v_cache"][b, :, :L]), torch.from_numpy(a["v_new"][b])[:, None]], 1)
        k = k.double().repeat_interleave(G, 0)
        v = v.double().repeat_interleave(G, 0)
        qb = torch.from_numpy(a["q"][b]).double()
        ks = qb * (torch.from_numpy(sink).double() * math.sqrt(w.D) / (qb * qb).sum(-1))[:, None]
        k = torch.cat([k, ks[:, None]], 1)
        v = torch.cat([v, torch.zeros(w.Hq, 1, w.D, dtype=torch.float64)], 1)
        o = torch.nn.functional.scaled_dot_product_attention(qb[:, None], k, v)[:, 0]
        np.testing.assert_allclose(r.out[b], o.numpy(), rtol=1e-11, atol=1e-12)


def test_window_equals_compacted_cache():
    """Window and kept prefix select slots: the same output comes from a
    cache that holds only the selected slots, in order (bit for bit, the sums
    run over the same terms in the same order)."""
    w, a = _mods_case(42, Smax=64, len_lo=20, len_hi=60)
    W_, P = 9, 4
    r = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(), a["v_cache"].copy(),
                            a["lengths"], window=W_, kept_prefix=P)
    for b in range(w.B):
        L = int(a["lengths"][b])
        keep = [j for j in range(L) if j > L - W_ or j < P]
        kc = np.ascontiguousarray(a["k_cache"][b:b + 1][:, :, keep + [0]])
        vc = np.ascontiguousarray(a["v_cache"][b:b + 1][:, :, keep + [0]])
        rb = oracle.decode_dense(a["q"][b:b + 1], a["k_new"][b:b + 1], a["v_new"][b:b + 1], kc, vc,
                                 np.array([len(keep)], np.int32))
        assert rb.out.tobytes() == r.out[b:b + 1].tobytes()


def test_window_one_returns_new_value_and_wide_window_is_plain():
    w, a = _mods_case(43)
    r1 = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(), a["v_cache"].copy(),
                             a["lengths"], window=1)
    assert np.array_equal(r1.out, np.repeat(a["v_new"].astype(np.float64), w.G, 1))
    r0 = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(), a["v_cache"].copy(),
                             a["lengths"])
    big = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(), a["v_cache"].copy(),
                              a["lengths"], window=w.Smax + 1)
    prefix_only = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(),
                                      a["v_cache"].copy(), a["lengths"], kept_prefix=7)
    minus_inf = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(),
                                    a["v_cache"].copy(), a["lengths"],
                                    sink=np.full(w.Hq, -np.inf, np.float32))
    for r in (big, prefix_only, minus_inf):
        assert r.out.tobytes() == r0.out.tobytes()


def test_kept_prefix_per_row_matches_scalar():
    w, a = _mods_case(44)
    per = np.array([0, 3, 11], np.int32)
    r = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(), a["v_cache"].copy(),
                            a["lengths"], window=5, kept_prefix=per)
    for b in range(w.B):
        rb = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(), a["v_cache"].copy(),
                                 a["lengths"], window=5, kept_prefix=int(per[b]), rows=[b])
        assert rb.out[b].tobytes() == r.out[b].tobytes()


def test_mods_attend_and_paged_agree_with_dense_decode():
    """The modifiers act on the query position L in every form: the attend
    of lengths L + 1 over a cache holding the new token equals the decode
    step's output; paged equals dense."""
    w, a = _mods_case(45)
    sink = np.linspace(-1, 1, w.Hq).astype(np.float32)
    kc, vc = a["k_cache"].copy(), a["v_cache"].copy()
    r_dec = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], kc, vc, a["lengths"], sink=sink,
                                window=6, kept_prefix=2)
    r_att = oracle.attend_dense(a["q"], kc, vc, a["lengths"] + 1, sink=sink, window=6, kept_prefix=2)
    assert r_att.out.tobytes() == r_dec.out.tobytes()
    bs = 4
    nb = w.Smax // bs
    kb = np.ascontiguousarray(kc.reshape(w.B, w.Hkv, nb, bs, w.D).transpose(0, 2, 1, 3, 4)
                              .reshape(w.B * nb, w.Hkv, bs, w.D))
    vb = np.ascontiguousarray(vc.reshape(w.B, w.Hkv, nb, bs, w.D).transpose(0, 2, 1, 3, 4)
                              .reshape(w.B * nb, w.Hkv, bs, w.D))
    bt = np.arange(w.B * nb, dtype=np.int32).reshape(w.B, nb)
    r_pg = oracle.attend_paged(a["q"], kb, vb, bt, a["lengths"] + 1, sink=sink, window=6, kept_prefix=2)
    assert r_pg.out.tobytes() == r_dec.out.tobytes()


def test_mods_refused():
    w, a = _mods_case(46)
    for kw in (dict(window=-1), dict(window=4, kept_prefix=-1),
               dict(window=4, kept_prefix=np.array([0, -2, 1], np.int32))):
        r = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"].copy(), a["v_cache"].copy(),
                                a["lengths"], **kw)
        assert r.status == oracle.INVALID_ARGUMENT


# ------------------------------------------------ multi-token append (q_len > 1)
#
# [P5] groupQueryAttention: q/k/v are packed over the tokens of all sequences
# ([sum S, heads * head_dim]); each row's write offset is cu_seqlens_k[b] -
# q_len[b] (our lengths[b]); the new keys and values are appended in place;
# "under the causal bound" token i sees the keys up to its own position.

def _multi_case(seed, q_lens, Smax=24, dtype="f32", Hq=4, Hkv=2, D=8):
    rng = np.random.default_rng(seed)
    B = len(q_lens)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = int(cu[-1])
    lens = np.array([rng.integers(0, Smax - n + 1) for n in q_lens], np.int32)
    f = lambda *sh: rng.normal(size=sh).astype(np.float32)
    q, kn, vn = f(T, Hq, D), f(T, Hkv, D), f(T, Hkv, D)
    kc, vc = f(B, Hkv, Smax, D), f(B, Hkv, Smax, D)
    if dtype == "bf16":
        q, kn, vn, kc, vc = (to_np(torch.from_numpy(a).to(torch.bfloat16)) for a in (q, kn, vn, kc, vc))
    return dict(q=q, k_new=kn, v_new=vn, k_cache=kc, v_cache=vc, lengths=lens, cu_q=cu, T=T)


def test_multi_q_len_one_is_the_decode_step():
    c = _multi_case(50, [1, 1, 1, 1], dtype="bf16")
    kc1, vc1 = c["k_cache"].copy(), c["v_cache"].copy()
    r1 = oracle.decode_multi_dense(c["q"], c["k_new"], c["v_new"], kc1, vc1, c["lengths"], c["cu_q"])
    kc2, vc2 = c["k_cache"].copy(), c["v_cache"].copy()
    r2 = oracle.decode_dense(c["q"], c["k_new"], c["v_new"], kc2, vc2, c["lengths"])
    assert r1.status == oracle.OK
    assert r1.out.tobytes() == r2.out.tobytes()
    assert kc1.tobytes() == kc2.tobytes() and vc1.tobytes() == vc2.tobytes()


@pytest.mark.parametrize("mods", [{}, dict(window=5, kept_prefix=2, sink=np.linspace(-1, 1, 4).astype(np.float32))])
def test_multi_equals_successive_decode_steps(mods):
    """Appending n tokens at once with the causal bound is the same as n
    decode steps, each appending one token and attending up to it (bit for
    bit: the same terms in the same order)."""
    q_lens = [3, 1, 5, 2]
    c = _multi_case(51, q_lens)
    kcm, vcm = c["k_cache"].copy(), c["v_cache"].copy()
    rm = oracle.decode_multi_dense(c["q"], c["k_new"], c["v_new"], kcm, vcm, c["lengths"], c["cu_q"], **mods)
    assert rm.status == oracle.OK
    kcs, vcs = c["k_cache"].copy(), c["v_cache"].copy()
    for b, n in enumerate(q_lens):
        for i in range(n):
            t = int(c["cu_q"][b]) + i
            kb, vb = np.ascontiguousarray(kcs[b:b + 1]), np.ascontiguousarray(vcs[b:b + 1])
            m = dict(mods)
            r = oracle.decode_dense(c["q"][t:t + 1], c["k_new"][t:t + 1], c["v_new"][t:t + 1], kb, vb,
                                    np.array([c["lengths"][b] + i], np.int32), **m)
            kcs[b:b + 1], vcs[b:b + 1] = kb, vb
            assert r.out.tobytes() == rm.out[t:t + 1].tobytes(), (b, i)
    assert kcs.tobytes() == kcm.tobytes() and vcs.tobytes() == vcm.tobytes()


def test_multi_causal_library_sdpa():
    """torch SDPA in float64 with an explicit causal mask: row b's n queries
    over its lengths[b] + n keys, query i masked beyond key lengths[b] + i."""
    q_lens = [4, 2, 6]
    c = _multi_case(52, q_lens, Smax=30, Hq=6, Hkv=2, D=16)
    kc, vc = c["k_cache"].copy(), c["v_cache"].copy()
    r = oracle.decode_multi_dense(c["q"], c["k_new"], c["v_new"], kc, vc, c["lengths"], c["cu_q"])
    G = 3
    for b, n in enumerate(q_lens):
        Lb = int(c["lengths"][b])
        t0 = int(c["cu_q"][b])
        k = torch.from_numpy(kc[b, :, :Lb + n]).double().repeat_interleave(G, 0)   # (Hq, S, D)
        v = torch.from_numpy(vc[b, :, :Lb + n]).double().repeat_interleave(G, 0)
        qb = torch.from_numpy(c["q"][t0:t0 + n]).double().permute(1, 0, 2)          # (Hq, n, D)
        mask = torch.arange(Lb + n)[None, :] <= (Lb + torch.arange(n))[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(qb, k, v, attn_mask=mask)
        np.testing.assert_allclose(r.out[t0:t0 + n], o.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


def test_multi_brute_force_tiny():
    q_lens = [2, 0, 3]
    c = _multi_case(53, q_lens, Smax=9, Hq=4, Hkv=1, D=3)
    kc, vc = c["k_cache"].copy(), c["v_cache"].copy()
    r = oracle.decode_multi_dense(c["q"], c["k_new"], c["v_new"], kc, vc, c["lengths"], c["cu_q"])
    want = np.full_like(r.out, np.nan)
    for b, n in enumerate(q_lens):
        Lb, t0 = int(c["lengths"][b]), int(c["cu_q"][b])
        keys = [c["k_cache"][b, 0, j] for j in range(Lb)] + [c["k_new"][t0 + i, 0] for i in range(n)]
        vals = [c["v_cache"][b, 0, j] for j in range(Lb)] + [c["v_new"][t0 + i, 0] for i in range(n)]
        for i in range(n):
            for h in range(4):
                qs = [float(x) for x in c["q"][t0 + i, h]]
                e = [math.exp(sum(a * float(k) for a, k in zip(qs, keys[j])) / math.sqrt(3))
                     for j in range(Lb + i + 1)]
                z = sum(e)
                for d in range(3):
                    want[t0 + i, h, d] = sum(e[j] * float(vals[j][d]) for j in range(Lb + i + 1)) / z
    np.testing.assert_allclose(r.out, want, rtol=1e-12, atol=1e-12)


def test_multi_append_and_no_append():
    """The n new tokens' bits land at slots lengths[b] .. lengths[b]+n-1 and
    nothing else changes; without the append the outputs are the same and
    the cache untouched."""
    q_lens = [3, 1, 0, 4]
    c = _multi_case(54, q_lens, dtype="bf16")
    kc, vc = c["k_cache"].copy(), c["v_cache"].copy()
    r = oracle.decode_multi_dense(c["q"], c["k_new"], c["v_new"], kc, vc, c["lengths"], c["cu_q"])
    want_k, want_v = c["k_cache"].copy(), c["v_cache"].copy()
    for b, n in enumerate(q_lens):
        for i in range(n):
            want_k[b, :, c["lengths"][b] + i] = c["k_new"][c["cu_q"][b] + i]
            want_v[b, :, c["lengths"][b] + i] = c["v_new"][c["cu_q"][b] + i]
    assert kc.tobytes() == want_k.tobytes() and vc.tobytes() == want_v.tobytes()
    kc2, vc2 = c["k_cache"].copy(), c["v_cache"].copy()
    r2 = oracle.decode_multi_dense(c["q"], c["k_new"], c["v_new"], kc2, vc2, c["lengths"], c["cu_q"],
                                   append=False)
    assert r2.out.tobytes() == r.out.tobytes()
    assert kc2.tobytes() == c["k_cache"].tobytes()


def test_multi_paged_equals_dense():
    q_lens = [3, 2, 4]
    c = _multi_case(55, q_lens, Smax=24, dtype="bf16")
    bs, nb = 4, 6
    B = len(q_lens)
    kb = np.ascontiguousarray(c["k_cache"].reshape(B, 2, nb, bs, 8).transpose(0, 2, 1, 3, 4).reshape(B * nb, 2, bs, 8))
    vb = np.ascontiguousarray(c["v_cache"].reshape(B, 2, nb, bs, 8).transpose(0, 2, 1, 3, 4).reshape(B * nb, 2, bs, 8))
    perm = np.random.default_rng(5).permutation(B * nb)
    kb2, vb2 = np.empty_like(kb), np.empty_like(vb)
    kb2[perm], vb2[perm] = kb, vb
    bt = perm.reshape(B, nb).astype(np.int32)
    kc, vc = c["k_cache"].copy(), c["v_cache"].copy()
    rd = oracle.decode_multi_dense(c["q"], c["k_new"], c["v_new"], kc, vc, c["lengths"], c["cu_q"])
    rp = oracle.decode_multi_paged(c["q"], c["k_new"], c["v_new"], kb2, vb2, bt, c["lengths"], c["cu_q"])
    assert rp.status == oracle.OK and rp.out.tobytes() == rd.out.tobytes()
    back = kb2[perm].reshape(B, nb, 2, bs, 8).transpose(0, 2, 1, 3, 4).reshape(B, 2, nb * bs, 8)
    assert back.tobytes() == kc.tobytes()


def test_multi_validate_rules():
    ok, bad = oracle.OK, oracle.INVALID_ARGUMENT
    L = np.array([3, 0, 5], np.int32)
    assert oracle.validate_multi_dense(L, np.array([0, 2, 2, 5], np.int32), None, 5, 3, 10) == ok
    assert oracle.validate_multi_dense(L, np.array([1, 2, 2, 5], np.int32), None, 5, 3, 10) == bad   # cu_q[0] != 0
    assert oracle.validate_multi_dense(L, np.array([0, 3, 2, 5], np.int32), None, 5, 3, 10) == bad   # decreasing
    assert oracle.validate_multi_dense(L, np.array([0, 2, 2, 4], np.int32), None, 5, 3, 10) == bad   # cu_q[B] != T
    assert oracle.validate_multi_dense(L, np.array([0, 2, 2, 5], np.int32), None, 5, 3, 7) == bad    # 5 + 3 > 7
    assert oracle.validate_multi_dense(L, np.array([0, 2, 2, 5], np.int32), None, 5, 3, 8) == ok     # exactly full
    assert oracle.validate_multi_dense(np.array([3, -1, 5], np.int32), np.array([0, 2, 2, 5], np.int32),
                                       None, 5, 3, 10) == bad
    assert oracle.validate_multi_dense(L, np.array([0, 2, 2, 5], np.int32), np.array([1, 1, 0], np.int32),
                                       5, 3, 10) == bad
    bt = np.array([[0, 1, -1], [2, -1, -1], [3, 4, -1]], np.int32)
    Lp = np.array([3, 1, 4], np.int32)
    assert oracle.validate_multi_paged(Lp, np.array([0, 2, 3, 5], np.int32), bt, 5, 6, 4) == ok       # 4 + 1 slots / 8
    assert oracle.validate_multi_paged(Lp, np.array([0, 2, 3, 8], np.int32), bt, 8, 6, 4) == bad      # 4 + 5 > 8


# ------------------------------------------------------ E4M3 (FP8) KV cache
#
# [P5] names kScale / vScale and says no more. Reading: OCP FP8 E4M3 bytes
# with one float32 scale per cache head, K = k_scale * K8; the append stores
# E4M3(float32(k_new) / k_scale), round to nearest even, saturating at 448.

def _e4m3_lib(x):
    """torch's float8_e4m3fn (a library routine) for in-range float32 values."""
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_matches_library_and_closed_forms():
    codes = np.arange(256, dtype=np.uint8)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    ours = np.array([oracle.e4m3_decode(int(c)) for c in codes])
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    ok = ~np.isnan(ours)
    assert np.array_equal(ours[ok], lib[ok].astype(np.float64))
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6 and oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert math.copysign(1.0, oracle.e4m3_decode(0x80)) == -1.0 and np.isnan(oracle.e4m3_decode(0x7F))


def test_e4m3_encode_round_trip_and_saturation():
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)
    assert oracle.e4m3_encode(1000.0) == 0x7E and oracle.e4m3_encode(-1e9) == 0xFE
    assert oracle.e4m3_encode(float("inf")) == 0x7E and oracle.e4m3_encode(float("-inf")) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def test_e4m3_encode_matches_library_rounding():
    """Random in-range floats and every midpoint between neighbouring codes
    (ties go to the even code) against torch's cast."""
    rng = np.random.default_rng(60)
    xs = np.concatenate([rng.uniform(-440, 440, 2000), rng.normal(0, 1, 2000), rng.normal(0, 0.01, 2000)])
    mids = []
    for c in range(0x7E):
        mids.append((oracle.e4m3_decode(c) + oracle.e4m3_decode(c + 1)) / 2)
    xs = np.concatenate([xs, mids, -np.asarray(mids)]).astype(np.float32)
    ours = np.array([oracle.e4m3_encode(float(x)) for x in xs], np.uint8)
    assert np.array_equal(ours, _e4m3_lib(xs))


def _e4m3_case(seed, Hkv=2, B=3, S=20, D=8):
    rng = np.random.default_rng(seed)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    kc = rng.choice(finite, size=(B, Hkv, S, D)).astype(np.uint8)
    vc = rng.choice(finite, size=(B, Hkv, S, D)).astype(np.uint8)
    lens = rng.integers(0, S, size=B).astype(np.int32)
    dec = np.vectorize(oracle.e4m3_decode)
    kn_codes = rng.choice(finite, size=(B, Hkv, D)).astype(np.uint8)
    vn_codes = rng.choice(finite, size=(B, Hkv, D)).astype(np.uint8)
    return kc, vc, lens, dec, kn_codes, vn_codes


def test_e4m3_unit_scales_equal_the_bf16_step():
    """E4M3 values are exact in bf16: with scales 1 the quantised step equals
    the bf16 step on the decoded values bit for bit, and the append stores
    the new values' own codes."""
    kc, vc, lens, dec, knc, vnc = _e4m3_case(61)
    B, Hkv, S, D = kc.shape
    to_bf16 = lambda a: to_np(torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16))
    q = to_bf16(np.random.default_rng(1).normal(size=(B, 4, D)))
    kn, vn = to_bf16(dec(knc)), to_bf16(dec(vnc))
    one = np.ones(Hkv, np.float32)
    k8, v8 = kc.copy(), vc.copy()
    r8 = oracle.decode_dense(q, kn, vn, k8, v8, lens, k_scale=one, v_scale=one)
    kb, vb = to_bf16(dec(kc)), to_bf16(dec(vc))
    rb = oracle.decode_dense(q, kn, vn, kb, vb, lens)
    assert r8.status == oracle.OK and r8.out.tobytes() == rb.out.tobytes()
    for b in range(B):
        assert k8[b, :, lens[b]].tobytes() == knc[b].tobytes() and v8[b, :, lens[b]].tobytes() == vnc[b].tobytes()


def test_e4m3_scales_multiply_per_cache_head():
    """Power-of-two scales are exact multipliers: the E4M3 step with
    k_scale = 2^a, v_scale = 2^c per head equals the bf16 step on
    scale * decoded values bit for bit."""
    kc, vc, lens, dec, knc, vnc = _e4m3_case(62)
    B, Hkv, S, D = kc.shape
    ks = np.array([0.25, 4.0], np.float32)
    vs = np.array([2.0, 0.5], np.float32)
    to_bf16 = lambda a: to_np(torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16))
    q = to_bf16(np.random.default_rng(2).normal(size=(B, 4, D)))
    kn = to_bf16(dec(knc) * ks[None, :, None])
    vn = to_bf16(dec(vnc) * vs[None, :, None])
    r8 = oracle.decode_dense(q, kn, vn, kc.copy(), vc.copy(), lens, k_scale=ks, v_scale=vs)
    rb = oracle.decode_dense(q, kn, vn, to_bf16(dec(kc) * ks[None, :, None, None]),
                             to_bf16(dec(vc) * vs[None, :, None, None]), lens)
    assert r8.out.tobytes() == rb.out.tobytes()


def test_e4m3_append_quantises_after_division():
    """The stored byte is the library's E4M3 cast of float32(k_new) / k_scale."""
    kc, vc, lens, dec, _, _ = _e4m3_case(63)
    B, Hkv, S, D = kc.shape
    rng = np.random.default_rng(3)
    # in range for the library cast (torch's cast does not saturate)
    kn = np.clip(rng.normal(size=(B, Hkv, D)), -4, 4).astype(np.float32) * 3
    vn = np.clip(rng.normal(size=(B, Hkv, D)), -4, 4).astype(np.float32)
    ks = np.array([0.03, 0.11], np.float32)
    vs = np.array([0.02, 0.05], np.float32)
    q = rng.normal(size=(B, 4, D)).astype(np.float32)
    k8, v8 = kc.copy(), vc.copy()
    r = oracle.decode_dense(q, kn, vn, k8, v8, lens, k_scale=ks, v_scale=vs)
    assert r.status == oracle.OK
    for b in range(B):
        assert np.abs(kn[b] / ks[:, None]).max() < 448
        assert np.array_equal(k8[b, :, lens[b]], _e4m3_lib(kn[b] / ks[:, None]))
        assert np.array_equal(v8[b, :, lens[b]], _e4m3_lib(vn[b] / vs[:, None]))


def test_e4m3_library_sdpa_on_dequantised_cache():
    """torch SDPA in float64 over scale * decoded slots (the stored new token
    included), per cache head, repeated for the G query heads."""
    kc, vc, lens, dec, _, _ = _e4m3_case(64, Hkv=2, B=3, S=24, D=16)
    B, Hkv, S, D = kc.shape
    rng = np.random.default_rng(4)
    q = rng.normal(size=(B, 6, D)).astype(np.float32)
    kn = rng.normal(size=(B, Hkv, D)).astype(np.float32)
    vn = rng.normal(size=(B, Hkv, D)).astype(np.float32)
    ks = np.array([0.05, 0.02], np.float32)
    vs = np.array([0.01, 0.03], np.float32)
    k8, v8 = kc.copy(), vc.copy()
    r = oracle.decode_dense(q, kn, vn, k8, v8, lens, k_scale=ks, v_scale=vs)
    for b in range(B):
        L = int(lens[b])
        k = torch.from_numpy(dec(k8[b, :, :L + 1]) * ks[:, None, None].astype(np.float64)).repeat_interleave(3, 0)
        v = torch.from_numpy(dec(v8[b, :, :L + 1]) * vs[:, None, None].astype(np.float64)).repeat_interleave(3, 0)
        o = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q[b]).double()[:, None], k, v)[:, 0]
        np.testing.assert_allclose(r.out[b], o.numpy(), rtol=1e-12, atol=1e-12)


def _e4m3_multi_case(seed, q_lens, Smax=24, Hq=4, Hkv=2, D=8):
    rng = np.random.default_rng(seed)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    B = len(q_lens)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = int(cu[-1])
    lens = np.array([rng.integers(0, Smax - n + 1) for n in q_lens], np.int32)
    to_bf16 = lambda a: to_np(torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16))
    q, kn, vn = (to_bf16(rng.normal(size=sh)) for sh in ((T, Hq, D), (T, Hkv, D), (T, Hkv, D)))
    kc = rng.choice(finite, size=(B, Hkv, Smax, D)).astype(np.uint8)
    vc = rng.choice(finite, size=(B, Hkv, Smax, D)).astype(np.uint8)
    return dict(q=q, k_new=kn, v_new=vn, k_cache=kc, v_cache=vc, lengths=lens, cu_q=cu,
                k_scale=np.array([0.013, 0.011], np.float32), v_scale=np.array([0.0113, 0.021], np.float32))


def test_e4m3_multi_equals_successive_decode_steps():
    """Over an E4M3 cache too, n tokens appended at once under the causal
    bound equal n single-token steps (quantised appends and outputs, bit for
    bit): each token is quantised on its own, and later tokens of the run
    attend to the stored (quantised) earlier ones."""
    q_lens = [3, 1, 4, 2]
    c = _e4m3_multi_case(64, q_lens)
    sc = dict(k_scale=c["k_scale"], v_scale=c["v_scale"])
    kcm, vcm = c["k_cache"].copy(), c["v_cache"].copy()
    rm = oracle.decode_multi_dense(c["q"], c["k_new"], c["v_new"], kcm, vcm, c["lengths"], c["cu_q"], **sc)
    assert rm.status == oracle.OK
    kcs, vcs = c["k_cache"].copy(), c["v_cache"].copy()
    for b, n in enumerate(q_lens):
        for i in range(n):
            t = int(c["cu_q"][b]) + i
            kb, vb = np.ascontiguousarray(kcs[b:b + 1]), np.ascontiguousarray(vcs[b:b + 1])
            r = oracle.decode_dense(c["q"][t:t + 1], c["k_new"][t:t + 1], c["v_new"][t:t + 1], kb, vb,
                                    np.array([c["lengths"][b] + i], np.int32), **sc)
            kcs[b:b + 1], vcs[b:b + 1] = kb, vb
            assert r.out.tobytes() == rm.out[t:t + 1].tobytes(), (b, i)
    assert kcs.tobytes() == kcm.tobytes() and vcs.tobytes() == vcm.tobytes()


def test_e4m3_multi_appends_the_library_cast():
    """Each appended token's bytes are the library's E4M3 cast of
    float32(k_new) / k_scale (in-range values), at slot lengths[b] + i."""
    q_lens = [2, 3]
    c = _e4m3_multi_case(65, q_lens)
    kc, vc = c["k_cache"].copy(), c["v_cache"].copy()
    r = oracle.decode_multi_dense(c["q"], c["k_new"], c["v_new"], kc, vc, c["lengths"], c["cu_q"],
                                  k_scale=c["k_scale"], v_scale=c["v_scale"])
    assert r.status == oracle.OK
    bf = lambda a: (a.astype(np.uint32) << 16).view(np.float32)
    for b, n in enumerate(q_lens):
        for i in range(n):
            t = int(c["cu_q"][b]) + i
            s = int(c["lengths"][b]) + i
            want_k = _e4m3_lib(bf(c["k_new"][t]) / c["k_scale"][:, None])
            want_v = _e4m3_lib(bf(c["v_new"][t]) / c["v_scale"][:, None])
            assert kc[b, :, s].tobytes() == want_k.tobytes() and vc[b, :, s].tobytes() == want_v.tobytes()


def test_e4m3_without_append_reads_the_stored_new_values():
    """Without the append, the new token is read from k_new / v_new as the
    cache would store it (quantised): the outputs equal the appending step's
    bit for bit and the cache is untouched (single and multi-token)."""
    c = _e4m3_multi_case(66, [1, 1, 1])
    sc = dict(k_scale=c["k_scale"], v_scale=c["v_scale"])
    q, kn, vn = c["q"], c["k_new"], c["v_new"]
    kc, vc = c["k_cache"].copy(), c["v_cache"].copy()
    r1 = oracle.decode_dense(q, kn, vn, kc, vc, c["lengths"], **sc)
    kc2, vc2 = c["k_cache"].copy(), c["v_cache"].copy()
    r2 = oracle.decode_dense(q, kn, vn, kc2, vc2, c["lengths"], append=False, **sc)
    assert r1.status == r2.status == oracle.OK
    assert r1.out.tobytes() == r2.out.tobytes()
    assert kc2.tobytes() == c["k_cache"].tobytes() and vc2.tobytes() == c["v_cache"].tobytes()
    m = _e4m3_multi_case(67, [3, 2, 4])
    sc = dict(k_scale=m["k_scale"], v_scale=m["v_scale"])
    kc, vc = m["k_cache"].copy(), m["v_cache"].copy()
    r3 = oracle.decode_multi_dense(m["q"], m["k_new"], m["v_new"], kc, vc, m["lengths"], m["cu_q"], **sc)
    kc2, vc2 = m["k_cache"].copy(), m["v_cache"].copy()
    r4 = oracle.decode_multi_dense(m["q"], m["k_new"], m["v_new"], kc2, vc2, m["lengths"], m["cu_q"],
                                   append=False, **sc)
    assert r3.out.tobytes() == r4.out.tobytes()
    assert kc2.tobytes() == m["k_cache"].tobytes()
