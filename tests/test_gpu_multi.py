"""GPU parity of the multi-token step (speculative / chunked decode): the
packed tokens cu_q[b] .. cu_q[b+1]-1 of row b are appended in place at slots
lengths[b] + i and token i attends slots 0 .. lengths[b] + i
("groupQueryAttention": packed q/k/v, write offset cu_seqlens_k[b] - q_len[b],
the causal bound). Against the CPU oracle on the same seeded inputs, both
kernels, dense / slot_ids / paged, group sizes 1..8 (tokens per chunk: 32 / G
on the tensor cores, 8 / G on the CUDA cores; units of up to 8, 16 and 32
query rows on the tensor cores),
rows with q_len 0, chunks crossing tiles, the softmax modifiers, E4M3 caches
(each appended token quantised); the whole cache is compared with the
oracle's appended host copy bit for bit. Bars: float32 1e-5; bfloat16 and
E4M3 2e-2 max|V|."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_cases import BF16_REL_TOL, F32_TOL, guard, path_of
from helpers import to_np

pytestmark = pytest.mark.gpu


def _tc_ok(w):
    return w.dtype == "bf16" and w.D == 128 and (
        not w.paged or (w.block_size >= 8 and (w.block_size & (w.block_size - 1)) == 0))


def _run_gpu(w, t, max_q, kernel="auto", grid=0, status=None, **mods):
    import gqa_kv_cache_gb300 as gqa
    kw = dict(max_q_len=max_q, kernel=kernel, grid_ctas=grid, status=status, **mods)
    if "k_scale" in t:                        # an E4M3 cache
        kw.update(k_scale=t["k_scale"], v_scale=t["v_scale"])
    if w.paged:
        return gqa.decode_multi_paged(t["q"], t["k_new"], t["v_new"], t["k_blocks"], t["v_blocks"],
                                      t["block_table"], t["lengths"], t["cu_q"], **kw)
    return gqa.decode_multi(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["lengths"],
                            t["cu_q"], t.get("slot_ids"), **kw)


def _run_oracle(w, a, **mods):
    om = {}
    if mods.get("sink") is not None:
        om["sink"] = mods["sink"].cpu().numpy()
    om["window"] = mods.get("window", 0)
    om["kept_prefix"] = mods.get("kept_prefix", 0)
    if "k_scale" in a:
        om.update(k_scale=a["k_scale"], v_scale=a["v_scale"])
    if w.paged:
        r = oracle.decode_multi_paged(a["q"], a["k_new"], a["v_new"], a["k_blocks"], a["v_blocks"],
                                      a["block_table"], a["lengths"], a["cu_q"], **om)
    else:
        r = oracle.decode_multi_dense(a["q"], a["k_new"], a["v_new"], a["k_cache"], a["v_cache"],
                                      a["lengths"], a["cu_q"], a.get("slot_ids"), **om)
    assert r.status == oracle.OK
    return r.out


def _vmax(w, a):
    """max |V| over the values the step attends: each row's cached slots
    0 .. lengths[b]-1 (E4M3 bytes times the per-head scale) and the new values."""
    f = lambda x: (x.astype(np.uint32) << 16).view(np.float32) if x.dtype == np.uint16 else x
    v = a["v_blocks"] if "v_blocks" in a else a["v_cache"]
    if v.dtype == np.uint8:
        v = torch.from_numpy(v).view(torch.float8_e4m3fn).double().numpy() * a["v_scale"].reshape(1, -1, 1, 1)
    else:
        v = f(v)
    vals = [float(np.abs(f(a["v_new"])).max())] if a["v_new"].size else [0.0]
    cu, L = a["cu_q"], a["lengths"]
    for b in range(len(L)):
        n = int(L[b])
        if cu[b + 1] == cu[b] or n <= 0:
            continue
        if "v_blocks" in a:
            bs = v.shape[2]
            blk = a["block_table"][b, np.arange(n) // bs]
            vals.append(float(np.abs(v[blk, :, np.arange(n) % bs]).max()))
        else:
            r = int(a["slot_ids"][b]) if "slot_ids" in a else b
            vals.append(float(np.abs(v[r, :, :n]).max()))
    return max(vals)


def check_multi(w, q_lens, kernel="auto", grid=0, fp8=False, **mods):
    t = {k: v.cuda() for k, v in W.generate(w, q_lens=q_lens, kv_e4m3=fp8).items()}
    a = {k: to_np(v) for k, v in t.items()}
    max_q = max(max(q_lens), 1)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _run_gpu(w, t, max_q, kernel, grid, st, **mods)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    vmax = _vmax(w, a)                        # before the oracle appends into the host copies
    want = _run_oracle(w, a, **mods)
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    tol = F32_TOL if w.dtype == "f32" else BF16_REL_TOL * vmax
    err = float(np.abs(got - want).max()) if got.size else 0.0
    assert err <= tol, f"max abs error {err} > {tol}"
    G = w.Hq // w.Hkv
    tpc = max(1, min(32 // G if kernel != "simt" else 8 // G, max_q))   # tokens of a full chunk
    guard(path_of(w, kernel, fp8=fp8, unit_rows=G * tpc), err, vmax)
    for n in (("k_blocks", "v_blocks") if w.paged else ("k_cache", "v_cache")):
        assert to_np(t[n]).tobytes() == a[n].tobytes(), f"{n} differs from the oracle's appended copy"
    return err


CASES = [
    # name, workload family, sizes, q_lens (chunks of 8 / G tokens)
    ("g4", "llama3_8b", dict(B=6, Smax=300, len_lo=0, len_hi=290, seed=401), [1, 2, 3, 0, 5, 8]),
    ("g8", "long_context", dict(B=4, Smax=400, len_lo=50, len_hi=390, seed=402), [3, 1, 6, 2]),
    ("g2", "llama3_8b", dict(Hq=4, Hkv=2, B=4, Smax=260, len_lo=0, len_hi=250, seed=403), [4, 7, 1, 9]),
    ("g1", "llama3_8b", dict(Hq=2, Hkv=2, B=3, Smax=200, len_lo=0, len_hi=190, seed=404), [8, 13, 2]),
    ("g6_paged16", "paged", dict(B=4, num_blocks=4 * 30, max_blocks=30, len_lo=0, len_hi=470, seed=405), [2, 4, 1, 3]),
    ("g3", "llama3_8b", dict(Hq=6, Hkv=2, B=3, Smax=300, len_lo=0, len_hi=290, seed=406), [5, 2, 4]),
    ("g8_slots", "ragged_slots", dict(B=5, R=9, Smax=300, len_lo=1, len_hi=290, seed=407), [2, 3, 1, 4, 2]),
    ("g4_paged8", "paged", dict(Hq=8, Hkv=2, B=3, block_size=8, num_blocks=3 * 40, max_blocks=40,
                                len_lo=0, len_hi=310, seed=408), [3, 6, 2]),
    ("f32_d64", "pr1_fp32", dict(B=3, Smax=256, len_lo=0, len_hi=250, seed=409), [3, 1, 4]),
    # full 16-row units on the tensor cores (and two 8-row chunks on the CUDA cores)
    ("g4_rows16", "llama3_8b", dict(B=3, Smax=400, len_lo=0, len_hi=390, seed=413), [4, 4, 3]),
    ("g2_rows16", "llama3_8b", dict(Hq=4, Hkv=2, B=2, Smax=300, len_lo=0, len_hi=290, seed=414), [8, 16]),
    ("g1_rows16", "llama3_8b", dict(Hq=2, Hkv=2, B=2, Smax=300, len_lo=0, len_hi=280, seed=415), [16, 5]),
    # units of 17 to 32 query rows on the tensor cores (two warps per 16 rows),
    # and rows of more tokens than one unit holds (several chunks)
    ("g4_rows32", "llama3_8b", dict(B=3, Smax=400, len_lo=0, len_hi=390, seed=423), [8, 5, 7]),
    ("g6_rows18_paged16", "paged", dict(B=4, num_blocks=4 * 30, max_blocks=30, len_lo=0, len_hi=460, seed=424),
     [3, 3, 2, 3]),
    ("g8_rows32", "long_context", dict(B=3, Smax=400, len_lo=50, len_hi=390, seed=425), [4, 3, 4]),
    ("g8_rows40", "long_context", dict(B=3, Smax=400, len_lo=50, len_hi=390, seed=426), [5, 2, 6]),
    ("g2_rows32_slots", "ragged_slots", dict(Hq=8, Hkv=4, B=3, R=7, Smax=300, len_lo=1, len_hi=280, seed=427),
     [16, 11, 9]),
    ("g4_rows32_paged8", "paged", dict(Hq=8, Hkv=2, B=3, block_size=8, num_blocks=3 * 40, max_blocks=40,
                                       len_lo=0, len_hi=300, seed=428), [8, 6, 8]),
    # units of at most 8 query rows (one chunk): on the tensor cores the rows
    # sit on the N = 8 side of the products
    ("g4_rows8", "llama3_8b", dict(B=5, Smax=400, len_lo=0, len_hi=390, seed=417), [2, 1, 0, 2, 2]),
    ("g2_rows8", "llama3_8b", dict(Hq=4, Hkv=2, B=3, Smax=300, len_lo=0, len_hi=290, seed=418), [4, 3, 1]),
    ("g1_rows8", "llama3_8b", dict(Hq=2, Hkv=2, B=3, Smax=300, len_lo=0, len_hi=290, seed=419), [8, 5, 3]),
    ("g8_rows8", "long_context", dict(B=4, Smax=400, len_lo=50, len_hi=390, seed=420), [1, 1, 0, 1]),
    ("g6_rows6_paged16", "paged", dict(B=4, num_blocks=4 * 30, max_blocks=30, len_lo=0, len_hi=470, seed=421),
     [1, 1, 1, 0]),
    ("g4_rows8_paged8", "paged", dict(Hq=8, Hkv=2, B=3, block_size=8, num_blocks=3 * 40, max_blocks=40,
                                      len_lo=0, len_hi=310, seed=422), [2, 2, 1]),
]


@pytest.mark.parametrize("kernel", ["simt", "tc"])
@pytest.mark.parametrize("name,base,kw,q_lens", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("grid", [0, 7])
def test_multi_small_cases(name, base, kw, q_lens, kernel, grid):
    w = W.small(base, **kw)
    if kernel == "tc" and not _tc_ok(w):
        pytest.skip("kernel does not take these sizes")
    check_multi(w, q_lens, kernel, grid)


FP8_CASES = [c for c in CASES if c[0] not in ("f32_d64",)]

# units of 17 to 32 query rows (and, after them, a second chunk)
T5_CASES = [c for c in CASES if c[0] in ("g4", "g8", "g2", "g2_rows16", "g4_rows32", "g6_rows18_paged16",
                                          "g8_rows32", "g8_rows40", "g2_rows32_slots", "g4_rows32_paged8")]


@pytest.mark.parametrize("name,base,kw,q_lens", T5_CASES, ids=[c[0] for c in T5_CASES])
@pytest.mark.parametrize("grid", [0, 7])
def test_multi_tcgen05_units(name, base, kw, q_lens, grid):
    """The opt-in tcgen05 form (kernel="tc5"): units of 17 to 32 query rows
    with S and O in tensor memory; smaller units and other chunks of the same
    call take the mma.sync forms. Same bars and cache check as above."""
    check_multi(W.small(base, **kw), q_lens, "tc5", grid)


@pytest.mark.parametrize("name,base,kw,q_lens", FP8_CASES, ids=[c[0] for c in FP8_CASES])
@pytest.mark.parametrize("grid", [0, 7])
def test_multi_fp8_small_cases(name, base, kw, q_lens, grid):
    """E4M3 caches (tensor-core kernel): the quantised tokens appended bit for
    bit, outputs within 2e-2 max|V| of the oracle over the same bytes."""
    check_multi(W.small(base, **kw), q_lens, "tc", grid, fp8=True)


@pytest.mark.parametrize("q_lens", [[7, 8, 1, 5], [3, 4, 1, 2], [2, 2, 1, 2]], ids=["rows32", "rows16", "rows8"])
def test_multi_fp8_window_sink(q_lens):
    w = W.small("llama3_8b", B=4, Smax=500, len_lo=100, len_hi=490, seed=416)
    g = torch.Generator().manual_seed(4)
    check_multi(w, q_lens, "tc", 0, fp8=True, window=70, kept_prefix=9,
                sink=(torch.randn(w.Hq, generator=g)).cuda())


@pytest.mark.parametrize("q_lens", [[7, 8, 1, 5], [3, 4, 1, 2], [2, 2, 1, 2]], ids=["rows32", "rows16", "rows8"])
@pytest.mark.parametrize("kernel", ["simt", "tc", "tc5"])
def test_multi_with_window_and_sink(kernel, q_lens):
    w = W.small("llama3_8b", B=4, Smax=500, len_lo=100, len_hi=490, seed=410)
    g = torch.Generator().manual_seed(3)
    check_multi(w, q_lens, kernel, 0, window=70, kept_prefix=9,
                sink=(torch.randn(w.Hq, generator=g)).cuda())


# One or two long rows over many CTAs: each unit is cut into more pieces than
# one pass of the merge's shared-memory weights takes (8 partials for 32-row
# units, 16 for 16-row units, 32 for 8-row units), so the merge goes through
# them in chunks (bfloat16 cache: in the CTA's own last segment end, and in
# the finisher warp's when a CTA ends a cut unit in the middle of its walk)
# or element by element (E4M3 cache, CUDA-core kernel).
MANY_PIECES = [
    ("rows32_g8", "long_context", dict(B=1, Hq=8, Hkv=1, Smax=2400, len_lo=2300, len_hi=2390, seed=431), [4]),
    ("rows16_g4", "llama3_8b", dict(B=2, Hq=4, Hkv=1, Smax=2400, len_lo=2200, len_hi=2390, seed=432), [4, 3]),
    ("rows8_g4", "llama3_8b", dict(B=1, Hq=4, Hkv=1, Smax=4200, len_lo=4000, len_hi=4190, seed=433), [2]),
]


@pytest.mark.parametrize("sink", [False, True], ids=["plain", "sink"])
@pytest.mark.parametrize("grid", [0, 40])
@pytest.mark.parametrize("kernel", ["tc", "tc_e4m3", "tc5", "simt"])
@pytest.mark.parametrize("name,base,kw,q_lens", MANY_PIECES, ids=[c[0] for c in MANY_PIECES])
def test_multi_unit_cut_into_many_pieces(name, base, kw, q_lens, kernel, grid, sink):
    import gqa_kv_cache_gb300 as gqa
    if kernel == "tc5" and not name.startswith("rows32"):
        pytest.skip("the tcgen05 form takes units of more than 16 rows only")
    w = W.small(base, **kw)
    mods = {}
    if sink:
        g = torch.Generator().manual_seed(5)
        mods["sink"] = torch.randn(w.Hq, generator=g).cuda()
    check_multi(w, q_lens, "tc" if kernel == "tc_e4m3" else kernel, grid, fp8=kernel == "tc_e4m3", **mods)
    ws = gqa._ws_cache.get(torch.device("cuda", torch.cuda.current_device()))
    if ws is not None:
        assert int(torch.count_nonzero(ws).item()) == 0


def test_tcgen05_choice_leaves_other_steps_on_tc():
    """kernel="tc5" changes only 17- to 32-row multi-token units over a bf16
    cache: a single-token step and an 8-row multi-token step give the very
    bits of kernel="tc"."""
    import gqa_kv_cache_gb300 as gqa
    w = W.small("llama3_8b", B=4, Smax=400, len_lo=0, len_hi=390, seed=429)
    res = {}
    for kernel in ("tc", "tc5"):
        t = {k: v.cuda() for k, v in W.generate(w).items()}
        a = gqa.decode_step(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["lengths"], kernel=kernel)
        t = {k: v.cuda() for k, v in W.generate(w, q_lens=[2, 1, 2, 2]).items()}
        b = _run_gpu(w, t, 2, kernel)
        res[kernel] = (a.clone(), b.clone())
    assert torch.equal(res["tc"][0], res["tc5"][0]) and torch.equal(res["tc"][1], res["tc5"][1])


@pytest.mark.parametrize("kernel", ["simt", "tc"])
def test_multi_q_len_one_matches_decode_step(kernel):
    """q_len = 1 everywhere is the decode step: the same appended bytes and
    outputs within the bf16 bar."""
    import gqa_kv_cache_gb300 as gqa
    w = W.small("llama3_8b", B=5, Smax=600, len_lo=0, len_hi=590, seed=411)
    t = {k: v.cuda() for k, v in W.generate(w, q_lens=[1] * w.B).items()}
    t2 = {k: v.clone() for k, v in t.items()}
    a = _run_gpu(w, t, 1, kernel).clone()
    b = gqa.decode_step(t2["q"], t2["k_new"], t2["v_new"], t2["k_cache"], t2["v_cache"], t2["lengths"],
                        kernel=kernel)
    vmax = max(t["v_cache"].float().abs().max().item(), t["v_new"].float().abs().max().item())
    assert (a - b).abs().max().item() <= BF16_REL_TOL * vmax
    assert torch.equal(t["k_cache"], t2["k_cache"]) and torch.equal(t["v_cache"], t2["v_cache"])


@pytest.mark.parametrize("kernel", ["simt", "tc"])
def test_multi_bad_rows(kernel):
    """A q_len above max_q_len and a write offset that does not leave room
    for the tokens: status bits, NaN (or nothing) for those rows only."""
    w = W.small("llama3_8b", B=3, Smax=128, len_lo=10, len_hi=100, seed=412)
    t = {k: v.cuda() for k, v in W.generate(w, q_lens=[2, 5, 2]).items()}
    t["lengths"][2] = 127                     # 127 + 2 > 128
    out = torch.full((int(t["cu_q"][-1]), w.Hq, w.D), 7.0, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    import gqa_kv_cache_gb300 as gqa
    gqa.decode_multi(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["lengths"], t["cu_q"],
                     max_q_len=4, out=out, status=st, kernel=kernel)
    torch.cuda.synchronize()
    s = int(st.item())
    assert s & 32 and s & 1
    assert torch.isfinite(out[0:2]).all()               # row 0
    assert (out[2:7] == 7.0).all()                      # row 1: q_len 5 > 4, not written
    assert torch.isnan(out[7:9]).all()                  # row 2: bad length
    assert not gqa.validate_multi(t["lengths"], t["cu_q"], 9, R=w.B, Smax=w.Smax)


def test_validate_multi_matches_oracle_rules():
    import gqa_kv_cache_gb300 as gqa
    rng = np.random.default_rng(2)
    for trial in range(60):
        B, T = 3, 7
        cu = np.sort(rng.integers(0, T + 1, size=B + 1)).astype(np.int32)
        if trial % 2:
            cu[0], cu[-1] = 0, T
        if trial % 5 == 0:
            cu[1], cu[2] = cu[2], cu[1]
        L = rng.integers(-1, 15, size=B).astype(np.int32)
        want = oracle.validate_multi_dense(L, cu, None, T, 3, 16) == oracle.OK
        got = gqa.validate_multi(torch.from_numpy(L).cuda(), torch.from_numpy(cu).cuda(), T, R=3, Smax=16)
        assert got == want, (trial, cu, L)
        bt = rng.integers(-2, 17, size=(B, 5)).astype(np.int32)
        if trial % 3 == 0:
            bt = rng.permutation(16)[:B * 5].reshape(B, 5).astype(np.int32)
        want = oracle.validate_multi_paged(L, cu, bt, T, 16, 4) == oracle.OK
        got = gqa.validate_multi(torch.from_numpy(L).cuda(), torch.from_numpy(cu).cuda(), T,
                                 block_table=torch.from_numpy(bt).cuda(), num_blocks=16, block_size=4)
        assert got == want, (trial, cu, L, bt)


@pytest.mark.parametrize("name,q_len,fp8", [("llama3_8b", 2, False), ("llama3_8b", 4, False), ("paged", 3, False),
                                            ("llama3_8b", 8, False), ("llama3_8b", 4, True), ("paged", 3, True)])
def test_multi_full_size(name, q_len, fp8):
    """Full-size caches with q_len new tokens per row: the tokens of 3
    sampled rows against the oracle (the sampled rows' caches copied to the
    host), the appended slots bit for bit."""
    import gqa_kv_cache_gb300 as gqa
    w = W.WORKLOADS[name]
    t = W.generate(w, "cuda", q_lens=[q_len] * w.B, kv_e4m3=fp8)
    rows = [0, w.B // 2, w.B - 1]
    sel = torch.tensor(rows, device="cuda")
    tok = torch.cat([torch.arange(int(t["cu_q"][b]), int(t["cu_q"][b + 1]), device="cuda") for b in rows])
    a = {"q": to_np(t["q"][tok]), "k_new": to_np(t["k_new"][tok]), "v_new": to_np(t["v_new"][tok]),
         "lengths": to_np(t["lengths"][sel]),
         "cu_q": np.arange(0, q_len * (len(rows) + 1), q_len, dtype=np.int32)}
    if fp8:
        a["k_scale"], a["v_scale"] = to_np(t["k_scale"]), to_np(t["v_scale"])
    if w.paged:
        bt = t["block_table"][sel].cpu().numpy()
        used = sorted(set(int(x) for x in bt[bt >= 0].tolist()))
        remap = {b: i for i, b in enumerate(used)}
        idx = torch.tensor(used, device="cuda")
        a["k_blocks"], a["v_blocks"] = to_np(t["k_blocks"][idx]), to_np(t["v_blocks"][idx])
        a["block_table"] = np.vectorize(lambda x: remap.get(int(x), -1))(bt).astype(np.int32)
    else:
        a["k_cache"], a["v_cache"] = to_np(t["k_cache"][sel]), to_np(t["v_cache"][sel])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _run_gpu(w, t, q_len, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    vmax = _vmax(w, a)
    want = _run_oracle(w, a)
    got = out[tok].double().cpu().numpy()
    err = float(np.abs(got - want).max())
    assert err <= BF16_REL_TOL * vmax
    G = w.Hq // w.Hkv
    guard(path_of(w, "tc", fp8=fp8, unit_rows=G * max(1, min(32 // G, q_len))), err, vmax)
    if w.paged:
        assert to_np(t["k_blocks"][idx]).tobytes() == a["k_blocks"].tobytes()
    else:
        assert to_np(t["k_cache"][sel]).tobytes() == a["k_cache"].tobytes()
