"""GPU parity of the read-only attend (no append): the CUDA path through the
C ABI against the CPU oracle on the same seeded inputs.

The attend follows "Grouped-Query Decode Step" (statement, Constraints):
lengths[b] counts the valid slots, slots 0..lengths[b]-1 are attended, the
query is float32 (or bfloat16) over a float32 or bfloat16 cache, and
"groupQueryAttention" (attention_over_cache): nothing but the output is
written. Bars: float32 cache max abs error <= 1e-5; bfloat16 cache
<= 2e-2 * max|V|, and with a float32 query <= 2e-4 * max|V| (the query is not
rounded to bfloat16: rounding it alone would cost ~1e-3); the caches are
compared bit for bit before and after."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_cases import BF16_REL_TOL, F32_TOL, attended_vmax, guard, host_problem, path_of, supports
from helpers import to_np

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32Q_REL_TOL = 2e-4


def inputs(w, q_f32, gpu_gen=False):
    if gpu_gen:
        return W.generate(w, "cuda", attend=True, q_f32=q_f32)
    return {k: v.cuda() for k, v in W.generate(w, "cpu", attend=True, q_f32=q_f32).items()}


def run_gpu(w, t, kernel="auto", grid_ctas=0, status=None):
    import gqa_kv_cache_gb300 as gqa
    if w.paged:
        return gqa.attend_paged(t["q"], t["k_blocks"], t["v_blocks"], t["block_table"], t["lengths"],
                                kernel=kernel, grid_ctas=grid_ctas, status=status)
    return gqa.attend(t["q"], t["k_cache"], t["v_cache"], t["lengths"], t.get("slot_ids"),
                      kernel=kernel, grid_ctas=grid_ctas, status=status)


def run_oracle(w, prob):
    if w.paged:
        r = oracle.attend_paged(prob["q"], prob["k_blocks"], prob["v_blocks"], prob["block_table"],
                                prob["lengths"])
    else:
        r = oracle.attend_dense(prob["q"], prob["k_cache"], prob["v_cache"], prob["lengths"])
    assert r.status == oracle.OK
    return r.out


def tolerance(w, q_f32, vmax):
    if w.dtype == "f32":
        return F32_TOL
    return (F32Q_REL_TOL if q_f32 else BF16_REL_TOL) * vmax


def _bits(x):
    return x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32)


def check_attend(w, q_f32, kernel="auto", grid_ctas=0, rows=None, gpu_gen=False):
    t = inputs(w, q_f32, gpu_gen)
    if rows == "sample4":
        L = t["lengths"]
        rows = [0, w.B - 1, int(torch.argmax(L).item()),
                int(np.random.default_rng(w.seed).integers(0, w.B))]
    prob = host_problem(w, t, rows)
    names = ("k_blocks", "v_blocks") if w.paged else ("k_cache", "v_cache")
    before = {n: t[n].clone() for n in names}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_gpu(w, t, kernel, grid_ctas, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    for n in names:
        assert torch.equal(_bits(before[n]), _bits(t[n])), f"{n} was written by a read-only attend"
    want = run_oracle(w, prob)
    got = out[torch.tensor(prob["rows"], device="cuda")].double().cpu().numpy()
    assert np.isfinite(got).all()
    err, vmax = float(np.abs(got - want).max()), attended_vmax(prob)
    guard(path_of(w, kernel, q_f32=q_f32), err, vmax)
    return err, tolerance(w, q_f32, vmax), out


# ------------------------------------------------------------ page examples

@pytest.mark.parametrize("cache_dtype", [torch.float32, torch.bfloat16])
def test_page_examples_attend(cache_dtype):
    """'Grouped-Query Decode Step' Examples 1-3 in the page's own contract
    (lengths as printed, float32 query); the printed values are exact in
    bfloat16, so a bfloat16 cache gives the same outputs."""
    import gqa_kv_cache_gb300 as gqa
    g = json.load(open(os.path.join(GOLDEN, "grouped_query_decode_step_examples.json")))
    for ex in g["examples"]:
        q = torch.tensor(ex["query"], dtype=torch.float32, device="cuda")
        kc = torch.tensor(ex["key_cache"], dtype=torch.float32).permute(0, 2, 1, 3).contiguous()
        vc = torch.tensor(ex["value_cache"], dtype=torch.float32).permute(0, 2, 1, 3).contiguous()
        kc, vc = kc.to(cache_dtype).cuda(), vc.to(cache_dtype).cuda()
        assert torch.equal(kc.float().cpu(), torch.tensor(ex["key_cache"]).permute(0, 2, 1, 3))
        lens = torch.tensor(ex["lengths"], dtype=torch.int32, device="cuda")
        out = gqa.attend(q, kc, vc, lens)
        np.testing.assert_allclose(out.cpu().numpy(), ex["output"], atol=1e-5)


# ------------------------------------------------------------- small cases

SMALL = [
    ("f32_d64", "pr1_fp32", dict(B=3, Smax=300, len_lo=0, len_hi=299, seed=201)),
    ("bf16_d128_g4", "llama3_8b", dict(B=5, Smax=700, len_lo=0, len_hi=699, seed=203)),
    ("bf16_d128_g8", "long_context", dict(B=3, Smax=1000, len_lo=60, len_hi=999, seed=204)),
    ("bf16_d128_g6_paged16", "paged", dict(B=5, num_blocks=5 * 40, max_blocks=40, len_lo=0, len_hi=639,
                                           seed=205)),
    ("bf16_d128_g8_slots", "ragged_slots", dict(B=6, R=11, Smax=600, len_lo=1, len_hi=599, seed=206)),
    ("bf16_d64_g2", "llama3_8b", dict(D=64, Hq=4, Hkv=2, B=3, Smax=260, len_lo=0, len_hi=259, seed=207)),
    ("bf16_d128_g3", "llama3_8b", dict(Hq=6, Hkv=2, B=2, Smax=300, len_lo=0, len_hi=299, seed=209)),
    ("bf16_d128_g4_paged8", "paged", dict(Hq=8, Hkv=2, B=3, block_size=8, num_blocks=3 * 50, max_blocks=50,
                                          len_lo=0, len_hi=399, seed=211)),
    ("f32_d16_paged3", "paged", dict(dtype="f32", D=16, Hq=4, Hkv=2, B=3, block_size=3, num_blocks=3 * 30,
                                     max_blocks=30, len_lo=0, len_hi=89, seed=212)),
]


@pytest.mark.parametrize("kernel", ["simt", "tc", "unit"])
@pytest.mark.parametrize("q_f32", [True, False], ids=["q_f32", "q_cache_dtype"])
@pytest.mark.parametrize("name,base,kw", SMALL, ids=[s[0] for s in SMALL])
@pytest.mark.parametrize("grid_ctas", [0, 7])
def test_attend_small_cases(name, base, kw, q_f32, kernel, grid_ctas):
    w = W.small(base, **kw)
    if not supports(kernel, w):
        pytest.skip("kernel does not take these sizes")
    err, tol, _ = check_attend(w, q_f32, kernel, grid_ctas)
    assert err <= tol, f"max abs error {err} > {tol}"


@pytest.mark.parametrize("kernel", ["simt", "tc", "unit"])
def test_bf16_query_over_f32_cache_and_mixed(kernel):
    """A bfloat16 query over a float32 cache (CUDA-core kernel only) matches
    the oracle at the float32 bar."""
    if kernel == "tc":
        pytest.skip("the tensor-core kernel takes bfloat16 caches")
    import gqa_kv_cache_gb300 as gqa
    w = W.small("pr1_fp32", B=3, Smax=300, len_lo=0, len_hi=299, seed=215)
    t = inputs(w, q_f32=True)
    t["q"] = t["q"].to(torch.bfloat16)
    prob = host_problem(w, t)
    out = gqa.attend(t["q"], t["k_cache"], t["v_cache"], t["lengths"], kernel=kernel)
    want = run_oracle(w, prob)
    assert np.abs(out.double().cpu().numpy() - want).max() <= F32_TOL


@pytest.mark.parametrize("kernel", ["simt", "tc", "unit"])
def test_attend_one_slot_and_full(kernel):
    """lengths 1 (every head returns slot 0's value exactly) and lengths Smax."""
    import gqa_kv_cache_gb300 as gqa
    w = W.small("llama3_8b", B=4, Smax=256, len_lo=0, len_hi=0, seed=220)
    t = inputs(w, q_f32=True)
    t["lengths"] = torch.tensor([1, 256, 1, 256], dtype=torch.int32, device="cuda")
    prob = host_problem(w, t)
    out = gqa.attend(t["q"], t["k_cache"], t["v_cache"], t["lengths"], kernel=kernel)
    want = run_oracle(w, prob)
    assert np.abs(out.double().cpu().numpy() - want).max() <= F32Q_REL_TOL * attended_vmax(prob)
    for b in (0, 2):
        assert torch.equal(out[b], t["v_cache"][b, :, 0].float().repeat_interleave(w.G, 0))


@pytest.mark.parametrize("kernel", ["simt", "tc", "unit"])
def test_attend_stale_nan(kernel):
    """NaN / Inf at and beyond lengths[b] cannot change a single output bit."""
    w = W.small("llama3_8b", B=4, Smax=400, len_lo=0, len_hi=398, seed=221)
    t = inputs(w, q_f32=True)
    ref = run_gpu(w, t, kernel).clone()
    j = torch.arange(w.Smax, device="cuda")
    stale = (j[None, :] >= t["lengths"].long()[:, None])[:, None, :, None]
    for fill in (float("nan"), float("inf")):
        t2 = dict(t)
        t2["k_cache"] = torch.where(stale, torch.full_like(t["k_cache"], fill), t["k_cache"])
        t2["v_cache"] = torch.where(stale, torch.full_like(t["v_cache"], -fill), t["v_cache"])
        assert torch.equal(run_gpu(w, t2, kernel), ref)


@pytest.mark.parametrize("kernel", ["simt", "tc", "unit"])
def test_attend_after_decode_step_is_bit_identical(kernel):
    """A decode step appends slot L and attends 0..L; the read-only attend of
    the resulting cache with lengths L + 1 attends the same slots and must
    return the same bits (bfloat16 query for both)."""
    import gqa_kv_cache_gb300 as gqa
    w = W.small("llama3_8b", B=5, Smax=700, len_lo=0, len_hi=698, seed=222)
    if not supports(kernel, w):
        w = W.small("llama3_8b", B=5, Smax=400, len_lo=0, len_hi=398, seed=222)
    t = {k: v.cuda() for k, v in W.generate(w).items()}
    dec = gqa.decode_step(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["lengths"],
                          kernel=kernel).clone()
    att = gqa.attend(t["q"], t["k_cache"], t["v_cache"], t["lengths"] + 1, kernel=kernel)
    assert torch.equal(dec, att)


@pytest.mark.parametrize("kernel", ["simt", "tc", "unit"])
def test_attend_bad_lengths(kernel):
    """lengths 0 and Smax + 1 are bad rows: NaN outputs and the length bit;
    the other rows are unaffected; gqa_validate_attend rejects the content."""
    import gqa_kv_cache_gb300 as gqa
    w = W.small("llama3_8b", B=4, Smax=128, len_lo=1, len_hi=126, seed=223)
    t = inputs(w, q_f32=True)
    t["lengths"][1] = 0
    t["lengths"][2] = 129
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_gpu(w, t, kernel, 0, st)
    torch.cuda.synchronize()
    assert int(st.item()) & 1
    assert torch.isnan(out[1]).all() and torch.isnan(out[2]).all()
    assert torch.isfinite(out[0]).all() and torch.isfinite(out[3]).all()
    assert not gqa.validate_attend(t["lengths"], R=w.B, Smax=w.Smax)
    t["lengths"][1], t["lengths"][2] = 1, 128
    assert gqa.validate_attend(t["lengths"], R=w.B, Smax=w.Smax)


def test_validate_attend_matches_oracle_rules():
    import gqa_kv_cache_gb300 as gqa
    rng = np.random.default_rng(1)
    for trial in range(60):
        B, nb, bs, mb = 3, 16, 4, 5
        bt = rng.integers(-2, nb + 1, size=(B, mb)).astype(np.int32)
        if trial % 3 == 0:
            bt = rng.permutation(nb)[:B * mb].reshape(B, mb).astype(np.int32)
        L = rng.integers(-1, mb * bs + 2, size=B).astype(np.int32)
        want = oracle.validate_attend_paged(L, bt, nb, bs) == oracle.OK
        got = gqa.validate_attend(torch.from_numpy(L).cuda(), block_table=torch.from_numpy(bt).cuda(),
                                  num_blocks=nb, block_size=bs)
        assert got == want, (trial, bt, L)
        sid = rng.integers(-1, 8, size=B).astype(np.int32)
        L2 = rng.integers(-1, 18, size=B).astype(np.int32)
        want = oracle.validate_attend_dense(L2, sid, 7, 16) == oracle.OK
        got = gqa.validate_attend(torch.from_numpy(L2).cuda(), slot_ids=torch.from_numpy(sid).cuda(),
                                  R=7, Smax=16)
        assert got == want, (trial, sid, L2)


# ----------------------------------------------------- full-size workloads

@pytest.mark.parametrize("name", ["pr1_fp32", "llama3_8b", "long_context", "ragged_slots", "paged"])
def test_attend_full_size_workloads(name):
    """The read-only attend with a float32 query on each workload's full-size
    cache in the default launch: 4 sampled rows against the oracle, the
    whole cache unchanged."""
    w = W.WORKLOADS[name]
    small_enough = name == "pr1_fp32"
    err, tol, _ = check_attend(w, True, rows=None if small_enough else "sample4", gpu_gen=not small_enough)
    assert err <= tol, f"{name}: max abs error {err} > {tol}"
