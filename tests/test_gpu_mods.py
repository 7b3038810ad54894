"""GPU parity of the softmax modifiers: attention sink, sliding window and
kept prefix ("groupQueryAttention": head_sink, slidingWindow, kept_prefix),
on the decode step and the read-only attend, dense / slot_ids / paged, both
kernels, against the CPU oracle on the same seeded inputs.

Readings: the window holds the W positions up to and including the query's
own (L); slot j <= L is attended when j > L - W or j < P; the sink is a logit
in the units of the scaled scores added to the softmax denominator. Bars as
for the plain step (float32 1e-5; bfloat16 2e-2 max|V|); the caches are
compared bit for bit (the decode step's append, nothing else written)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_cases import attended_vmax, host_problem, make_inputs, supports, tolerance
from helpers import to_np

pytestmark = pytest.mark.gpu


def _gpu(w, t, attend, kernel, grid, mods, status=None):
    import gqa_kv_cache_gb300 as gqa
    kw = dict(kernel=kernel, grid_ctas=grid, status=status, **mods)
    if attend:
        if w.paged:
            return gqa.attend_paged(t["q"], t["k_blocks"], t["v_blocks"], t["block_table"], t["lengths"], **kw)
        return gqa.attend(t["q"], t["k_cache"], t["v_cache"], t["lengths"], t.get("slot_ids"), **kw)
    if w.paged:
        return gqa.decode_step_paged(t["q"], t["k_new"], t["v_new"], t["k_blocks"], t["v_blocks"],
                                     t["block_table"], t["lengths"], **kw)
    return gqa.decode_step(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["lengths"],
                           t.get("slot_ids"), **kw)


def _oracle(w, prob, attend, mods, rows):
    om = {}
    if mods.get("sink") is not None:
        om["sink"] = mods["sink"].cpu().numpy()
    om["window"] = mods.get("window", 0)
    kp = mods.get("kept_prefix", 0)
    om["kept_prefix"] = kp.cpu().numpy()[rows] if isinstance(kp, torch.Tensor) else kp
    if attend:
        f = oracle.attend_paged if w.paged else oracle.attend_dense
        r = f(prob["q"], *( (prob["k_blocks"], prob["v_blocks"], prob["block_table"]) if w.paged
                            else (prob["k_cache"], prob["v_cache"]) ), prob["lengths"], **om)
    elif w.paged:
        r = oracle.decode_paged(prob["q"], prob["k_new"], prob["v_new"], prob["k_blocks"], prob["v_blocks"],
                                prob["block_table"], prob["lengths"], **om)
    else:
        r = oracle.decode_dense(prob["q"], prob["k_new"], prob["v_new"], prob["k_cache"], prob["v_cache"],
                                prob["lengths"], **om)
    assert r.status == oracle.OK
    return r.out


def _inputs(w, attend):
    if attend:
        return {k: v.cuda() for k, v in W.generate(w, "cpu", attend=True, q_f32=True).items()}
    return make_inputs(w)


def _mods(kind, w, seed):
    g = torch.Generator().manual_seed(seed)
    sink = (torch.randn(w.Hq, generator=g) * 2).cuda()
    if kind == "sink":
        return dict(sink=sink)
    if kind == "window1":
        return dict(window=1)
    if kind == "window64":
        return dict(window=64)
    if kind == "window100_prefix10":
        return dict(window=100, kept_prefix=10)
    if kind == "window70_prefix200":          # the prefix reaches into the window: one run of tiles
        return dict(window=70, kept_prefix=200)
    if kind == "window37_prefix_rows_sink":
        P = torch.randint(0, 90, (w.B,), generator=g, dtype=torch.int32).cuda()
        return dict(window=37, kept_prefix=P, sink=sink)
    raise ValueError(kind)


CASES = [
    ("bf16_dense", "llama3_8b", dict(B=5, Smax=700, len_lo=0, len_hi=699, seed=301)),
    ("bf16_slots", "ragged_slots", dict(B=6, R=11, Smax=600, len_lo=1, len_hi=599, seed=302)),
    ("bf16_paged16", "paged", dict(B=5, num_blocks=5 * 40, max_blocks=40, len_lo=0, len_hi=639, seed=303)),
    ("f32_d64", "pr1_fp32", dict(B=3, Smax=300, len_lo=0, len_hi=299, seed=304)),
    # capacities the small-cache kernel stages whole
    ("bf16_dense_cap380", "llama3_8b", dict(B=5, Smax=380, len_lo=0, len_hi=379, seed=305)),
    ("bf16_paged16_cap384", "paged", dict(B=5, num_blocks=5 * 24, max_blocks=24, len_lo=0, len_hi=383,
                                          seed=306)),
]
MODS = ["sink", "window1", "window64", "window100_prefix10", "window70_prefix200",
        "window37_prefix_rows_sink"]


@pytest.mark.parametrize("kernel", ["simt", "tc", "unit"])
@pytest.mark.parametrize("attend", [False, True], ids=["decode", "attend"])
@pytest.mark.parametrize("mod", MODS)
@pytest.mark.parametrize("name,base,kw", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("grid", [0, 7])
def test_mods_against_oracle(name, base, kw, mod, attend, kernel, grid):
    w = W.small(base, **kw)
    if not supports(kernel, w):
        pytest.skip("kernel does not take these sizes")
    t = _inputs(w, attend)
    mods = _mods(mod, w, kw["seed"])
    prob = host_problem(w, t)
    names = ("k_blocks", "v_blocks") if w.paged else ("k_cache", "v_cache")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _gpu(w, t, attend, kernel, grid, mods, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    want = _oracle(w, prob, attend, mods, list(range(w.B)))
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - want).max()
    tol = tolerance(w, attended_vmax(prob))
    assert err <= tol, f"max abs error {err} > {tol}"
    # the oracle appended into its host copies (decode step): the device
    # storage must hold the same bytes
    if w.paged:
        idx = torch.tensor(prob["blocks"], dtype=torch.long, device="cuda")
    else:
        idx = torch.tensor(prob["cache_rows"], dtype=torch.long, device="cuda")
    for n in names:
        assert to_np(t[n][idx]).tobytes() == prob[n].tobytes()


@pytest.mark.parametrize("kernel", ["simt", "tc", "unit"])
def test_masked_region_never_matters(kernel):
    """NaN in every slot outside the window and the kept prefix (below the
    query position) changes no output bit: those tiles are not read, and the
    masked rows of partly covered tiles are masked by selection and zeroed."""
    w = W.small("llama3_8b", B=4, Smax=900, len_lo=300, len_hi=899, seed=310)
    if not supports(kernel, w):
        w = W.small("llama3_8b", B=4, Smax=400, len_lo=250, len_hi=399, seed=310)
    t = make_inputs(w)
    mods = dict(window=150, kept_prefix=20)
    ref = _gpu(w, {k: v.clone() for k, v in t.items()}, False, kernel, 0, mods).clone()
    L = t["lengths"].long()
    j = torch.arange(w.Smax, device="cuda")[None, :]
    masked = ((j <= L[:, None] - 150) & (j >= 20))[:, None, :, None]
    t2 = {k: v.clone() for k, v in t.items()}
    t2["k_cache"] = torch.where(masked, torch.full_like(t["k_cache"], float("nan")), t["k_cache"])
    t2["v_cache"] = torch.where(masked, torch.full_like(t["v_cache"], float("nan")), t["v_cache"])
    out = _gpu(w, t2, False, kernel, 0, mods)
    assert torch.equal(out, ref)


@pytest.mark.parametrize("kernel", ["simt", "tc", "unit"])
def test_paged_blocks_outside_window_may_be_unmapped(kernel):
    """Table entries whose blocks hold no attended slot (between the kept
    prefix and the window) may be -1: the result is the same bits and no
    status bit is set."""
    w = W.small("paged", B=4, num_blocks=4 * 60, max_blocks=60, len_lo=500, len_hi=959, seed=311)
    if not supports(kernel, w):
        w = W.small("paged", B=4, num_blocks=4 * 25, max_blocks=25, len_lo=300, len_hi=399, seed=311)
    t = make_inputs(w)
    mods = dict(window=100, kept_prefix=16)
    ref = _gpu(w, {k: v.clone() for k, v in t.items()}, False, kernel, 0, mods).clone()
    t2 = {k: v.clone() for k, v in t.items()}
    for b in range(w.B):
        L = int(t["lengths"][b])
        lo = L - 100 + 1
        for i in range(w.max_blocks):
            s0, s1 = i * 16, i * 16 + 15
            if s0 >= 16 and s1 < lo:
                t2["block_table"][b, i] = -1
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _gpu(w, t2, False, kernel, 0, mods, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out, ref)


@pytest.mark.parametrize("kernel", ["simt", "tc", "unit"])
def test_negative_prefix_row_is_bad(kernel):
    w = W.small("llama3_8b", B=3, Smax=300, len_lo=100, len_hi=299, seed=312)
    t = make_inputs(w)
    P = torch.tensor([5, -1, 7], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _gpu(w, t, False, kernel, 0, dict(window=50, kept_prefix=P), st)
    torch.cuda.synchronize()
    assert int(st.item()) & 16
    assert torch.isnan(out[1]).all() and torch.isfinite(out[0]).all() and torch.isfinite(out[2]).all()


def test_negative_window_or_prefix_rejected_on_the_host():
    import gqa_kv_cache_gb300 as gqa
    w = W.small("llama3_8b", B=2, Smax=128, len_lo=1, len_hi=100, seed=313)
    t = make_inputs(w)
    for kw in (dict(window=-1), dict(window=4, kept_prefix=-3)):
        with pytest.raises(gqa.GqaError):
            _gpu(w, t, False, "auto", 0, kw)


@pytest.mark.parametrize("name", ["long_context", "paged"])
def test_full_size_window_sink(name):
    """Full-size workloads with a 4096-position window, a 64-key prefix and a
    sink: 4 sampled rows against the oracle, cache bytes as the oracle left
    them."""
    w = W.WORKLOADS[name]
    t = W.generate(w, "cuda")
    L = t["lengths"]
    rows = sorted({0, w.B - 1, int(torch.argmax(L).item())})
    prob = host_problem(w, t, rows)
    g = torch.Generator().manual_seed(7)
    mods = dict(window=4096, kept_prefix=64, sink=torch.randn(w.Hq, generator=g).cuda())
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _gpu(w, t, False, "auto", 0, mods, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    want = _oracle(w, prob, False, mods, rows)
    got = out[torch.tensor(rows, device="cuda")].double().cpu().numpy()
    assert np.abs(got - want).max() <= tolerance(w, attended_vmax(prob))
