"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs. Cases span several tiles and ragged tails, every
addressing form, both kernels, several CTA counts, empty and single-slot rows,
NaN-filled stale slots, bad content, and the five decode workloads at full
size (sampled rows against the oracle, the whole cache bit-exact)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_cases import check_step, make_inputs, run_gpu, host_problem, run_oracle, supports, tolerance, attended_vmax
from helpers import to_np

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------ page examples

def test_page_examples_kv_cache_decode_step():
    """'KV cache decode step' Examples 1-3 through the library (D = 1 and 2,
    fp32): output within 1e-5 of the printed values, caches extended."""
    import gqa_kv_cache_gb300 as gqa
    g = json.load(open(os.path.join(GOLDEN, "kv_cache_decode_step_examples.json")))
    for ex in g["examples"]:
        f = lambda x: torch.tensor(x, dtype=torch.float32, device="cuda")
        q, kn, vn = f(ex["query"]), f(ex["new_key"]), f(ex["new_value"])
        kc0, vc0 = f(ex["key_cache"]), f(ex["value_cache"])
        B, Hkv, S, D = kc0.shape
        kc = torch.zeros(B, Hkv, S + 1, D, device="cuda")
        vc = torch.zeros_like(kc)
        kc[:, :, :S], vc[:, :, :S] = kc0, vc0
        out = gqa.decode_step(q, kn, vn, kc, vc, torch.full((B,), S, dtype=torch.int32, device="cuda"),
                              kernel="simt")
        np.testing.assert_allclose(out.cpu().numpy(), ex["output"], atol=1e-5)
        np.testing.assert_allclose(kc.cpu().numpy(), ex["new_key_cache"], atol=5e-7)
        np.testing.assert_allclose(vc.cpu().numpy(), ex["new_value_cache"], atol=5e-7)


def test_page_examples_grouped_query_decode_step():
    """'Grouped-Query Decode Step' Examples 1-3 (D = 2 and 4, fp32, the stale
    slots included), mapped onto the append-slot convention."""
    import gqa_kv_cache_gb300 as gqa
    g = json.load(open(os.path.join(GOLDEN, "grouped_query_decode_step_examples.json")))
    for ex in g["examples"]:
        q = torch.tensor(ex["query"], dtype=torch.float32, device="cuda")
        kc = torch.tensor(ex["key_cache"], dtype=torch.float32).permute(0, 2, 1, 3).contiguous().cuda()
        vc = torch.tensor(ex["value_cache"], dtype=torch.float32).permute(0, 2, 1, 3).contiguous().cuda()
        lens = torch.tensor(ex["lengths"], dtype=torch.int32, device="cuda")
        b = torch.arange(q.shape[0], device="cuda")
        kn = kc[b, :, lens.long() - 1].contiguous()
        vn = vc[b, :, lens.long() - 1].contiguous()
        out = gqa.decode_step(q, kn, vn, kc, vc, lens - 1, kernel="simt")
        np.testing.assert_allclose(out.cpu().numpy(), ex["output"], atol=1e-5)


# ------------------------------------------------------------- small cases

SMALL = [
    # name, overrides: several tiles (64 slots), ragged tails, empty rows
    ("f32_d64", "pr1_fp32", dict(B=3, Smax=300, len_lo=0, len_hi=299, seed=101)),
    ("f32_d128_g8", "pr1_fp32", dict(D=128, Hq=16, Hkv=2, B=3, Smax=200, len_lo=0, len_hi=199, seed=102)),
    ("bf16_d128_g4", "llama3_8b", dict(B=5, Smax=700, len_lo=0, len_hi=699, seed=103)),
    ("bf16_d128_g8", "long_context", dict(B=3, Smax=1000, len_lo=60, len_hi=999, seed=104)),
    ("bf16_d128_g6_paged16", "paged", dict(B=5, num_blocks=5 * 40, max_blocks=40, len_lo=0, len_hi=639, seed=105)),
    ("bf16_d128_g8_slots", "ragged_slots", dict(B=6, R=11, Smax=600, len_lo=1, len_hi=599, seed=106)),
    ("bf16_d64_g2", "llama3_8b", dict(D=64, Hq=4, Hkv=2, B=3, Smax=260, len_lo=0, len_hi=259, seed=107)),
    ("bf16_d256_g1", "llama3_8b", dict(D=256, Hq=2, Hkv=2, B=2, Smax=130, len_lo=0, len_hi=129, seed=108)),
    ("bf16_d128_g3", "llama3_8b", dict(Hq=6, Hkv=2, B=2, Smax=300, len_lo=0, len_hi=299, seed=109)),
    ("bf16_d128_g4_paged64", "paged", dict(Hq=16, Hkv=4, B=3, block_size=64, num_blocks=3 * 10,
                                           max_blocks=10, len_lo=0, len_hi=639, seed=110)),
    ("bf16_d128_g4_paged8", "paged", dict(Hq=8, Hkv=2, B=3, block_size=8, num_blocks=3 * 50,
                                          max_blocks=50, len_lo=0, len_hi=399, seed=111)),
    ("f32_d16_paged3", "paged", dict(dtype="f32", D=16, Hq=4, Hkv=2, B=3, block_size=3,
                                     num_blocks=3 * 30, max_blocks=30, len_lo=0, len_hi=89, seed=112)),
    ("f32_d4_g2", "pr1_fp32", dict(D=4, Hq=4, Hkv=2, B=3, Smax=90, len_lo=0, len_hi=89, seed=113)),
]


@pytest.mark.parametrize("kernel", ["simt", "tc", "unit"])
@pytest.mark.parametrize("name,base,kw", SMALL, ids=[s[0] for s in SMALL])
@pytest.mark.parametrize("grid_ctas", [0, 1, 7])
def test_small_cases(name, base, kw, kernel, grid_ctas):
    w = W.small(base, **kw)
    if not supports(kernel, w):
        pytest.skip("kernel does not take these sizes")
    err, tol, _ = check_step(w, kernel=kernel, grid_ctas=grid_ctas)
    assert err <= tol, f"max abs error {err} > {tol}"


@pytest.mark.parametrize("kernel", ["simt", "tc", "unit"])
def test_lengths_zero_and_full(kernel):
    """Rows with an empty cache (output = v_new) and rows at capacity - 1."""
    w = W.small("llama3_8b", B=4, Smax=256, len_lo=0, len_hi=0, seed=120)
    t = make_inputs(w)
    t["lengths"] = torch.tensor([0, 255, 0, 255], dtype=torch.int32, device="cuda")
    prob = host_problem(w, t)
    out = run_gpu(w, t, kernel)
    want = run_oracle(w, prob)
    got = out.double().cpu().numpy()
    assert np.abs(got - want).max() <= tolerance(w, attended_vmax(prob))
    # one valid slot: the output is the new value itself
    vn = t["v_new"].float()
    for b in (0, 2):
        assert torch.equal(out[b], vn[b].repeat_interleave(w.G, 0))


@pytest.mark.parametrize("kernel", ["simt", "tc", "unit"])
def test_stale_slots_nan(kernel):
    """NaN / Inf in every stale slot and in the (stale) append slot cannot
    change a single output bit."""
    w = W.small("llama3_8b", B=4, Smax=400, len_lo=0, len_hi=399, seed=121)
    t = make_inputs(w)
    ref = run_gpu(w, {k: v.clone() for k, v in t.items()}, kernel).clone()
    L = t["lengths"].long()
    j = torch.arange(w.Smax, device="cuda")
    stale = (j[None, :] >= L[:, None])[:, None, :, None]
    for fill in (float("nan"), float("inf")):
        t2 = {k: v.clone() for k, v in t.items()}
        t2["k_cache"] = torch.where(stale, torch.full_like(t["k_cache"], fill), t["k_cache"])
        t2["v_cache"] = torch.where(stale, torch.full_like(t["v_cache"], -fill), t["v_cache"])
        out = run_gpu(w, t2, kernel)
        assert torch.equal(out, ref)


@pytest.mark.parametrize("slots", [False, True], ids=["rows", "slot_ids"])
@pytest.mark.parametrize("window", [0, 40], ids=["full", "window40"])
@pytest.mark.parametrize("grid_ctas", [0, 7])
def test_stale_slots_nan_in_partly_copied_tiles(grid_ctas, window, slots):
    """A dense cache's partly read tiles (a unit's last, a window's first) are
    copied in 16-slot parts; the parts not copied keep whatever the ring
    stage held before. With few CTAs each walking many short units, those
    are often NaN / Inf rows of an earlier unit's stale slots: not a single
    output bit may change against the clean cache."""
    import gqa_kv_cache_gb300 as gqa
    base = "ragged_slots" if slots else "llama3_8b"
    kw = dict(R=40) if slots else {}
    w = W.small(base, B=24, Hq=8, Hkv=2, Smax=256, len_lo=1, len_hi=250, seed=131 + window + slots, **kw)
    t = make_inputs(w)
    mods = dict(window=window, kept_prefix=5) if window else {}

    def run(tt):
        return gqa.decode_step(tt["q"], tt["k_new"], tt["v_new"], tt["k_cache"], tt["v_cache"], tt["lengths"],
                               tt.get("slot_ids"), kernel="tc", grid_ctas=grid_ctas, **mods)

    ref = run({k: v.clone() for k, v in t.items()}).clone()
    L = t["lengths"].long()
    rows = t["slot_ids"].long() if slots else torch.arange(w.B, device="cuda")
    j = torch.arange(w.Smax, device="cuda")
    for fill in (float("nan"), float("inf")):
        t2 = {k: v.clone() for k, v in t.items()}
        stale = torch.ones(t["k_cache"].shape[0], w.Smax, dtype=torch.bool, device="cuda")
        stale[rows] = j[None, :] >= L[:, None]
        if window:   # slots outside every query's window and the kept prefix are not read either
            lo = (L - window + 1).clamp(min=0)
            stale[rows] |= (j[None, :] < lo[:, None]) & (j[None, :] >= 5)
        stale = stale[:, None, :, None]
        t2["k_cache"] = torch.where(stale, torch.full_like(t["k_cache"], fill), t["k_cache"])
        t2["v_cache"] = torch.where(stale, torch.full_like(t["v_cache"], -fill), t["v_cache"])
        out = run(t2)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), (fill, grid_ctas, window, slots)


@pytest.mark.parametrize("kernel", ["simt", "tc", "unit"])
def test_paged_unused_blocks_nan(kernel):
    """Blocks the table does not name, and the unused tail of the last block,
    hold NaN: the output must equal the clean run bit for bit."""
    w = W.small("paged", B=4, num_blocks=4 * 30 + 17, max_blocks=30, len_lo=0, len_hi=479, seed=122)
    if not supports(kernel, w):
        w = W.small("paged", B=4, num_blocks=4 * 20 + 17, max_blocks=20, len_lo=0, len_hi=319, seed=122)
    t = make_inputs(w)
    ref = run_gpu(w, {k: v.clone() for k, v in t.items()}, kernel).clone()
    used = set(t["block_table"][t["block_table"] >= 0].tolist())
    unused = torch.tensor([i for i in range(w.num_blocks) if i not in used], device="cuda")
    t2 = {k: v.clone() for k, v in t.items()}
    t2["k_blocks"][unused] = float("nan")
    t2["v_blocks"][unused] = float("nan")
    out = run_gpu(w, t2, kernel)
    assert torch.equal(out, ref)


@pytest.mark.parametrize("kernel", ["simt", "tc"])
def test_split_counts_agree_and_are_deterministic(kernel):
    """Different CTA counts split the sequences differently: outputs agree
    within float32 rounding; the same count twice gives the same bits."""
    w = W.small("long_context", B=2, Smax=5000, len_lo=3000, len_hi=4999, seed=123)
    t = make_inputs(w)
    outs = {}
    for c in (1, 2, 5, 33, 0):
        outs[c] = run_gpu(w, {k: v.clone() for k, v in t.items()}, kernel, c).clone()
    again = run_gpu(w, {k: v.clone() for k, v in t.items()}, kernel, 33)
    assert torch.equal(again, outs[33])
    for c, o in outs.items():
        assert (o - outs[1]).abs().max().item() < 1e-4, c


def test_kernels_agree():
    """The CUDA-core and tensor-core kernels agree within the bf16 bar."""
    w = W.small("llama3_8b", B=4, Smax=900, len_lo=0, len_hi=899, seed=124)
    t = make_inputs(w)
    a = run_gpu(w, {k: v.clone() for k, v in t.items()}, "simt").clone()
    b = run_gpu(w, {k: v.clone() for k, v in t.items()}, "tc").clone()
    assert (a - b).abs().max().item() <= 2e-2 * t["v_cache"].float().abs().max().item()


# ------------------------------------------------------------- bad content

def test_bad_content_reports_and_never_faults():
    import gqa_kv_cache_gb300 as gqa
    w = W.small("ragged_slots", B=4, R=6, Smax=128, len_lo=1, len_hi=127, seed=130)
    t = make_inputs(w)
    t["lengths"][1] = 128              # beyond capacity
    t["slot_ids"][2] = 9               # out of range
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc0 = t["k_cache"].clone()
    out = run_gpu(w, t, "simt", 0, st)
    torch.cuda.synchronize()
    assert int(st.item()) & 1 and int(st.item()) & 2
    assert torch.isnan(out[1]).all() and torch.isnan(out[2]).all()
    assert torch.isfinite(out[0]).all() and torch.isfinite(out[3]).all()
    assert not gqa.validate(t["lengths"], slot_ids=t["slot_ids"], R=w.R, Smax=w.Smax)


@pytest.mark.parametrize("kernel", ["simt", "tc", "unit"])
def test_bad_block_reports(kernel):
    w = W.small("paged", B=3, num_blocks=3 * 20, max_blocks=20, len_lo=100, len_hi=300, seed=131)
    t = make_inputs(w)
    t["block_table"][1, 2] = w.num_blocks + 5      # out of range, inside the needed range
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_gpu(w, t, kernel, 0, st)
    torch.cuda.synchronize()
    assert int(st.item()) & 4
    assert torch.isnan(out[1]).all()
    assert torch.isfinite(out[0]).all() and torch.isfinite(out[2]).all()


def test_validate_matches_oracle_rules():
    """The GPU validation and the oracle's rules agree on random (mostly
    broken) tables and slot maps."""
    import gqa_kv_cache_gb300 as gqa
    rng = np.random.default_rng(0)
    for trial in range(60):
        B, nb, bs, mb = 3, 16, 4, 5
        bt = rng.integers(-2, nb + 1, size=(B, mb)).astype(np.int32)
        if trial % 3 == 0:
            bt = rng.permutation(nb)[:B * mb].reshape(B, mb).astype(np.int32)
        L = rng.integers(-1, mb * bs + 1, size=B).astype(np.int32)
        want = oracle.validate_paged(L, bt, nb, bs) == oracle.OK
        got = gqa.validate(torch.from_numpy(L).cuda(), block_table=torch.from_numpy(bt).cuda(),
                           num_blocks=nb, block_size=bs)
        assert got == want, (trial, bt, L)
        sid = rng.integers(-1, 8, size=B).astype(np.int32)
        L2 = rng.integers(-1, 17, size=B).astype(np.int32)
        want = oracle.validate_dense(L2, sid, 7, 16) == oracle.OK
        got = gqa.validate(torch.from_numpy(L2).cuda(), slot_ids=torch.from_numpy(sid).cuda(), R=7, Smax=16)
        assert got == want, (trial, sid, L2)


def test_empty_batch_and_errors():
    import gqa_kv_cache_gb300 as gqa
    q = torch.zeros(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    c = torch.zeros(1, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    out = gqa.decode_step(q, kv, kv, c, c, torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert out.shape == (0, 8, 128)
    q = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(1, 2, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gqa.GqaError):
        gqa.decode_step(q, kv, kv, c, c, torch.zeros(1, dtype=torch.int32, device="cuda"), kernel="tc",
                        workspace=torch.zeros(16, dtype=torch.uint8, device="cuda"))   # too small a workspace


# ----------------------------------------------------- full-size workloads

FULL = ["pr1_fp32", "llama3_8b", "long_context", "ragged_slots", "paged"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workloads(name):
    """Each decode workload at its full size in the default launch (the one
    the benchmark times): every output of 4 sampled batch rows (first, last,
    the longest and a random one) against the oracle, the whole cache
    bit-exact on the device."""
    w = W.WORKLOADS[name]
    small_enough = name == "pr1_fp32"
    err, tol, _ = check_step(w, rows=None if small_enough else "sample4", gpu_gen=not small_enough)
    assert err <= tol, f"{name}: max abs error {err} > {tol}"


@pytest.mark.parametrize("kernel", ["simt", "tc"])
def test_workspace_left_zero_across_sizes(kernel):
    """One caller-owned workspace, zero-filled once, serves calls of growing
    and shrinking sizes: each output matches the oracle and after every call
    the workspace is all zero again (counters reset, merged partials cleared)."""
    import gqa_kv_cache_gb300 as gqa
    cases = [W.small("llama3_8b", B=2, Smax=300, len_lo=100, len_hi=299, seed=140),
             W.small("long_context", B=5, Smax=2000, len_lo=500, len_hi=1999, seed=141),
             W.small("llama3_8b", B=3, Smax=900, len_lo=0, len_hi=899, seed=142)]
    need = max(gqa.workspace_bytes(w.B, w.Hq, w.Hkv, w.D, torch.bfloat16, kernel, 37) for w in cases)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for w in cases:
        t = make_inputs(w)
        prob = host_problem(w, t)
        out = gqa.decode_step(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["lengths"],
                              kernel=kernel, grid_ctas=37, workspace=ws)
        torch.cuda.synchronize()
        want = run_oracle(w, prob)
        assert np.abs(out.double().cpu().numpy() - want).max() <= tolerance(w, attended_vmax(prob))
        assert int(torch.count_nonzero(ws).item()) == 0


@pytest.mark.parametrize("kernel", ["simt", "tc"])
@pytest.mark.parametrize("sched_pad", [0, 1, 3, 7])
def test_schedule_padding(kernel, sched_pad):
    """Schedule-only padding tiles change which CTA streams which tiles, never
    the result: outputs within the bar of the oracle, cache bit-exact, for
    several CTA counts including ranges that start or end inside a unit's
    padding."""
    import gqa_kv_cache_gb300 as gqa
    for name, kw, grids in (("llama3_8b", dict(B=5, Smax=700, len_lo=0, len_hi=699, seed=150), (0, 3, 11)),
                            ("ragged_slots", dict(B=9, R=13, Smax=500, len_lo=1, len_hi=499, seed=151), (0, 5, 23))):
        w = W.small(name, **kw)
        for grid in grids:
            t = make_inputs(w)
            prob = host_problem(w, t)
            out = gqa.decode_step(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["lengths"],
                                  t.get("slot_ids"), kernel=kernel, grid_ctas=grid, sched_pad=sched_pad)
            torch.cuda.synchronize()
            want = run_oracle(w, prob)
            assert np.abs(out.double().cpu().numpy() - want).max() <= tolerance(w, attended_vmax(prob)), (name, grid)
            idx = torch.tensor(prob["cache_rows"], dtype=torch.long, device="cuda")
            assert to_np(t["k_cache"][idx]).tobytes() == prob["k_cache"].tobytes()


@pytest.mark.parametrize("kernel", ["simt", "tc"])
@pytest.mark.parametrize("grid_ctas", [40, 150])
def test_unit_cut_into_many_pieces(kernel, grid_ctas):
    """One or two long sequences over many CTAs: every unit is cut into far
    more pieces than the in-shared-memory merge takes (more than 32), so the
    merge falls back to its general form; outputs against the oracle, the
    cache bit-exact, the workspace left zero-filled."""
    import gqa_kv_cache_gb300 as gqa
    w = W.small("long_context", B=2, Hq=8, Hkv=1, Smax=9000, len_lo=7000, len_hi=8999, key_scale=1.0, seed=160)
    err, tol, _ = check_step(w, kernel=kernel, grid_ctas=grid_ctas)
    assert err <= tol, f"max abs error {err} > {tol}"
    ws = gqa._ws_cache.get(torch.device("cuda", torch.cuda.current_device()))
    if ws is not None:
        assert int(torch.count_nonzero(ws).item()) == 0
