"""Inputs and checks that see every single slot (shared by the GPU tests in
test_gpu_slots.py and their CPU self-checks in test_slot_checks.py).

Dominant slot. In every (row, cache head) unit the query rows of the group
share one random direction u (q = u + 0.3 noise) and one slot j* holds the
key 6 sqrt(128 / D) u, so its score beats every other attended slot by far more than 30
(natural units; the check measures the margin on the data it built). The
softmax then gives j* a weight of 1 - O(L e^-30), and every query row that
attends j* must return V_{j*} -- "Grouped-Query Decode Step", formula: the
output is the weight-sum of the attended values. Each slot carries its own
random value, so a lost or misplaced j* shows at once. j* sits at a tile's
first or last slot, at a cut between CTAs, at the new token, at the last
valid slot.

Zero query. With q = 0 every attended slot gets the same weight ("KV cache
decode step", Example 2: a zero query averages the values), so the output is
the mean of the attended values; with every weight exactly 1 in the kernels'
arithmetic only float32 summation error is left, and one slot too many or
too few moves the mean by about |V_j| / n, far above the tight bar here.

No expected value comes from the CUDA path: the oracle and the planted
values decide."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W
from helpers import to_np

C_DOM = 6.0       # the dominant key is C_DOM * sqrt(128 / D) * u (a score lead near 68)
MARGIN = 30.0     # least lead of the dominant score the construction must give
DOM_TOL = 1e-3    # dominated rows: |out - V_{j*}| <= DOM_TOL * max|V|
UNI_TOL = 2e-5    # zero query: |out - oracle| <= UNI_TOL * max|V|
BF16_REL_TOL = 2e-2
TILE = 64         # slots per tile of the tensor-core kernel
PAD = 3           # schedule-only tiles per unit (the library's default)
E4M3_KEY_RANGE = 32.0   # the E4M3 key scale represents keys up to 32 (6u fits)


class Step:
    """One call's inputs (CPU tensors until `finish`) and its kind:
    "decode", "attend" or "multi"."""

    def __init__(self, w, kind, q_lens=None, fp8=False, q_f32=False):
        self.w, self.kind, self.fp8 = w, kind, fp8
        self.attend = kind == "attend"
        self.multi = kind == "multi"
        self.t = W.generate(w, "cpu", attend=self.attend, q_f32=q_f32,
                            q_lens=q_lens if self.multi else None)
        L = self.t["lengths"].long()
        if self.multi:
            cu = self.t["cu_q"].long()
            self.tok0 = cu[:-1].tolist()
            self.qlen = (cu[1:] - cu[:-1]).tolist()
        else:
            self.tok0 = list(range(w.B))
            self.qlen = [1] * w.B
        # first slot holding a new token; last attended slot of each row's last token
        self.Lb = [int(x) if not self.attend else 1 << 30 for x in L.tolist()]
        self.last = [int(x) - 1 if self.attend else int(x) + n - 1 for x, n in zip(L.tolist(), self.qlen)]
        self.host = None

    def rows(self, b):
        """(token index, last attended slot) of row b's query tokens."""
        if self.attend:
            return [(b, self.last[b])]
        return [(self.tok0[b] + i, self.Lb[b] + i) for i in range(self.qlen[b])]

    def live(self, b):
        return self.qlen[b] > 0 and self.last[b] >= 0

    def key_slot(self, b, kvh, j, name="k"):
        """The tensor and index holding K (name 'k') or V ('v') of slot j of
        unit (b, kvh): a new token's row of k_new / v_new, else the cache."""
        w, t = self.w, self.t
        if not self.attend and j >= self.Lb[b]:
            return t[name + "_new"], (self.tok0[b] + j - self.Lb[b], kvh)
        if w.paged:
            blk = int(t["block_table"][b, j // w.block_size])
            return t[name + "_blocks"], (blk, kvh, j % w.block_size)
        r = int(t["slot_ids"][b]) if "slot_ids" in t else b
        return t[name + "_cache"], (r, kvh, j)

    def finish(self):
        """E4M3: quantise the cache (the new tokens stay bfloat16). Then the
        oracle's host copies."""
        if self.fp8:
            W.quantise_cache(self.w, self.t, key_range=E4M3_KEY_RANGE)
        self.host = {k: to_np(v) for k, v in self.t.items()}
        return self

    def device(self):
        return {k: v.cuda() for k, v in self.t.items()}

    def unit_kv(self, b, kvh, n):
        """K and V of slots 0..n-1 of unit (b, kvh) as the step reads them
        (float64; E4M3 bytes dequantised, new tokens quantised like the
        append)."""
        w, t = self.w, self.t
        j = torch.arange(n)
        cached = j if self.attend else j[j < self.Lb[b]]
        new_tok = (self.tok0[b] + j[len(cached):] - (0 if self.attend else self.Lb[b])).long()
        out = []
        for name in ("k", "v"):
            if w.paged:
                blk = t["block_table"][b, cached // w.block_size].long()
                c = t[name + "_blocks"][blk, kvh, cached % w.block_size]
            else:
                r = int(t["slot_ids"][b]) if "slot_ids" in t else b
                c = t[name + "_cache"][r, kvh, cached]
            nw = t[name + "_new"][new_tok, kvh] if len(new_tok) else None
            if self.fp8:
                s = float(t[name + "_scale"][kvh])
                c = c.view(torch.float8_e4m3fn).double() * s
                if nw is not None:
                    nw = (nw.float() / s).clamp(-448, 448).to(torch.float8_e4m3fn).double() * s
            x = c.double() if nw is None else torch.cat([c.double(), nw.double()])
            out.append(x.numpy())
        return out

    def vmax(self):
        """max |V| over the attended values of every live unit."""
        v = 0.0
        for b in range(self.w.B):
            if self.live(b):
                for kvh in range(self.w.Hkv):
                    v = max(v, float(np.abs(self.unit_kv(b, kvh, self.last[b] + 1)[1]).max()))
        return v


def run_oracle(st):
    """The oracle on the step's host copies (appending into them)."""
    w, a = st.w, st.host
    om = {}
    if st.fp8:
        om.update(k_scale=a["k_scale"], v_scale=a["v_scale"])
    if st.multi:
        if w.paged:
            r = oracle.decode_multi_paged(a["q"], a["k_new"], a["v_new"], a["k_blocks"], a["v_blocks"],
                                          a["block_table"], a["lengths"], a["cu_q"], **om)
        else:
            r = oracle.decode_multi_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"], a["v_cache"],
                                          a["lengths"], a["cu_q"], a.get("slot_ids"), **om)
    elif st.attend:
        if w.paged:
            r = oracle.attend_paged(a["q"], a["k_blocks"], a["v_blocks"], a["block_table"], a["lengths"], **om)
        else:
            r = oracle.attend_dense(a["q"], a["k_cache"], a["v_cache"], a["lengths"], a.get("slot_ids"), **om)
    elif w.paged:
        r = oracle.decode_paged(a["q"], a["k_new"], a["v_new"], a["k_blocks"], a["v_blocks"], a["block_table"],
                                a["lengths"], **om)
    else:
        r = oracle.decode_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"], a["v_cache"], a["lengths"],
                                a.get("slot_ids"), **om)
    assert r.status == oracle.OK
    return r.out


def cut_slots(st, grid):
    """Slots at the cuts between CTAs of a `grid`-CTA tensor-core launch of a
    single-token step: the first slot of each CTA range that starts inside a
    unit, and the slot before it. {(b, kvh): [slots]}."""
    w = st.w
    n_unit = [(st.last[b] // TILE + 1) + PAD if st.last[b] >= 0 else 1 + PAD for b in range(w.B)]
    starts, run = [], 0
    for b in range(w.B):
        for kvh in range(w.Hkv):
            starts.append((run, b, kvh))
            run += n_unit[b]
    N = run
    C = min(grid, N)
    cuts = {}
    for i in range(1, C):
        g = i * N // C
        for s, b, kvh in starts:
            if s <= g < s + n_unit[b]:
                t = g - s
                if 0 < t <= st.last[b] // TILE:
                    cuts.setdefault((b, kvh), []).extend([t * TILE, t * TILE - 1])
    return cuts


def part_slots(st, b, k):
    """Slots at the edges of the parts the small-cache kernel shares a unit of
    row b out in, when a cluster of 2, 4 or 8 CTAs (by k) takes the unit:
    either its staged rows (the attended slots, the new token last) cut into
    equal contiguous parts, or (a dense cache staged before the lengths are
    known) the row's capacity cut so. The first slot of each part after the
    first, and the slot before it, for both cuts."""
    cl = (2, 4, 8)[k % 3]
    n = st.last[b] + 1
    cap = st.w.max_blocks * st.w.block_size if st.w.paged else st.w.Smax
    out = []
    for chunk in (-(-n // cl), -(-cap // cl)):
        for m in range(1, cl):
            if m * chunk < n:
                out += [m * chunk, m * chunk - 1]
    return out


def plant_dominant(st, seed, grid=0, unit_parts=False):
    """Gives every unit a shared query direction and one dominant slot j*;
    returns {(b, kvh): j*}. j* sits at a CTA cut of a `grid`-CTA tensor-core
    launch, or (`unit_parts`) at a part edge of the small-cache kernel, or
    else at tile edges, the new token and the last slot."""
    w, t = st.w, st.t
    g = torch.Generator().manual_seed(seed)
    cuts = cut_slots(st, grid) if grid and not st.multi else {}
    dom = {}
    k = 0
    for b in range(w.B):
        if not st.live(b):
            continue
        last = st.last[b]
        first_new = st.Lb[b] if not st.attend else last
        cand = [0, 63, 64, 127, 128, last - 1, last, first_new, first_new - 1, 16, 15, 31, 32, 47, 48]
        for kvh in range(w.Hkv):
            u = torch.randn(w.D, generator=g)
            for tok, _ in st.rows(b):
                for h in range(kvh * w.G, (kvh + 1) * w.G):
                    t["q"][tok, h] = (u + 0.3 * torch.randn(w.D, generator=g)).to(t["q"].dtype)
            c = part_slots(st, b, k) if unit_parts else cuts.get((b, kvh))
            j = c[(k // 3 if unit_parts else k) % len(c)] if c else cand[k % len(cand)]
            j = min(max(j, 0), last)
            ten, idx = st.key_slot(b, kvh, j, "k")
            ten[idx] = (C_DOM * (128.0 / w.D) ** 0.5 * u).to(ten.dtype)
            dom[(b, kvh)] = j
            k += 1
    return dom


def dominated_rows(st, dom):
    """{(token, head): V_{j*}} for every query row that attends its unit's
    j*, after checking the construction's margin on the data; and max|V|."""
    w = st.w
    q = st.host["q"]
    vmax, exp = 0.0, {}
    for (b, kvh), j in dom.items():
        K, V = st.unit_kv(b, kvh, st.last[b] + 1)
        vmax = max(vmax, float(np.abs(V).max()))
        for tok, lim in st.rows(b):
            if j > lim:
                continue
            for h in range(kvh * w.G, (kvh + 1) * w.G):
                qv = (q[tok, h].astype(np.uint32) << 16).view(np.float32).astype(np.float64) \
                    if q.dtype == np.uint16 else q[tok, h].astype(np.float64)
                s = K[:lim + 1] @ qv / np.sqrt(w.D)
                lead = s[j] - np.delete(s, j).max() if lim > 0 else np.inf
                assert lead >= MARGIN, f"construction: unit {(b, kvh)} lead {lead:.1f} < {MARGIN}"
                exp[(tok, h)] = V[j]
    return exp, vmax


def check_dominant(st, dom, got, want):
    """`got`: the outputs under test; `want`: the oracle's. Every dominated
    row within DOM_TOL max|V| of V_{j*}; every row within the stated bar of
    the oracle. Returns the number of dominated rows."""
    exp, vmax = dominated_rows(st, dom)
    for (tok, h), v in exp.items():
        d_orc = float(np.abs(want[tok, h] - v).max())
        assert d_orc <= DOM_TOL * vmax, f"oracle: row {tok} head {h} off V_j* by {d_orc}"
        d = float(np.abs(got[tok, h] - v).max())
        assert d <= DOM_TOL * vmax, f"row {tok} head {h}: |out - V_j*| = {d:.3e} > {DOM_TOL * vmax:.3e}"
    assert len(exp) > 0
    assert float(np.abs(got - want).max()) <= BF16_REL_TOL * vmax
    return len(exp)


def check_uniform(st, got, want):
    """Zero query: `got` within UNI_TOL max|V| of the oracle's mean of the
    attended values. Returns the error relative to max|V|."""
    vmax = st.vmax()
    err = float(np.abs(got - want).max())
    assert err <= UNI_TOL * vmax, f"zero query: max |out - mean| {err:.3e} > {UNI_TOL * vmax:.3e}"
    return err / vmax


SINGLE = [
    # name, family, sizes
    ("dense_g4", "llama3_8b", dict(B=8, Smax=520, len_lo=0, len_hi=519, seed=601)),
    ("dense_g8", "long_context", dict(B=4, Smax=700, len_lo=60, len_hi=699, key_scale=1.0, seed=602)),
    ("slots_g8", "ragged_slots", dict(B=6, R=11, Smax=600, len_lo=1, len_hi=599, seed=603)),
    ("paged16_g6", "paged", dict(B=6, num_blocks=6 * 40, max_blocks=40, len_lo=0, len_hi=630, seed=604)),
    ("paged8_g4", "paged", dict(Hq=8, Hkv=2, B=5, block_size=8, num_blocks=5 * 70, max_blocks=70,
                                len_lo=0, len_hi=550, seed=605)),
]

MULTI = [
    # name, family, sizes, q_lens: query rows per unit G * q_len (up to 8: rows on
    # the N side of the products; 9 to 16: the M side, one warp per 16 slots; 17
    # to 32: the M side, two warps per 16 rows; 40: two chunks)
    ("rows8_g4", "llama3_8b", dict(B=6, Smax=520, len_lo=0, len_hi=500, seed=611), [2, 1, 2, 0, 2, 2]),
    ("rows16_g4", "llama3_8b", dict(B=5, Smax=520, len_lo=0, len_hi=500, seed=612), [4, 3, 4, 1, 4]),
    ("rows16_g8_paged16", "paged", dict(Hq=16, Hkv=2, B=4, num_blocks=4 * 40, max_blocks=40, len_lo=0,
                                        len_hi=600, seed=613), [2, 2, 1, 2]),
    ("rows18_g6_paged16", "paged", dict(B=4, num_blocks=4 * 40, max_blocks=40, len_lo=0, len_hi=600,
                                        seed=614), [3, 3, 2, 3]),
    ("rows8_g4_paged8", "paged", dict(Hq=8, Hkv=2, B=4, block_size=8, num_blocks=4 * 70, max_blocks=70,
                                      len_lo=0, len_hi=540, seed=615), [2, 2, 1, 2]),
    ("rows32_g4", "llama3_8b", dict(B=5, Smax=520, len_lo=0, len_hi=500, seed=616), [8, 5, 8, 1, 7]),
    ("rows40_g8", "long_context", dict(B=4, Smax=600, len_lo=60, len_hi=560, key_scale=1.0, seed=617),
     [5, 4, 5, 2]),
]

# capacities the small-cache kernel takes (K and V of a row within 200 KB of
# one CTA's shared memory); few units are shared out over clusters of 2 to 8
# CTAs, 128 units (the first case) take one CTA each; the dense float32 and
# the two-row bfloat16 cases stage the capacity before the lengths are known
UNIT = [
    ("dense_g4_cap384_b16", "llama3_8b", dict(B=16, Smax=384, len_lo=0, len_hi=383, seed=625)),
    ("dense_g4_cap384", "llama3_8b", dict(B=8, Smax=384, len_lo=0, len_hi=383, seed=621)),
    ("dense_g4_cap256_b2", "llama3_8b", dict(B=2, Smax=256, len_lo=0, len_hi=255, seed=626)),
    ("slots_g8_cap320", "ragged_slots", dict(B=6, R=11, Smax=320, len_lo=1, len_hi=319, seed=622)),
    ("paged16_g6_cap384", "paged", dict(B=6, num_blocks=6 * 24, max_blocks=24, len_lo=0, len_hi=380, seed=623)),
    ("f32_d64_g4_cap256", "pr1_fp32", dict(B=4, Smax=256, len_lo=0, len_hi=255, seed=624)),
]
