"""The bounded-wait abort paths, made to run out safely.

Tensor-core kernels: a wait of a consumer warp for a tile to land is
bounded; when it gives up the CTA aborts: it reports GQA_STATUS_TIMEOUT, the
units it touches get NaN, and before it exits every copy it issued still
lands (its producer's waits keep their full limit), so the context and the
workspace stay usable. Here every consumer warp's first wait also waits on an
on-chip barrier that nothing completes, with the consumers' limit cut to
about a microsecond, so that wait runs out in every working CTA whatever the
timing of the copies. The small-cache kernel: each CTA's wait for its staged
rows does the same, then waits (with the full limit) for its copies to land
before it exits; its unit gets NaN (its append, issued before the wait, may
have landed: nothing else of the cache changes). Nothing faults or hangs:
the wait simply ends.

Checked: the status is exactly the timeout bit; every output is NaN; no byte
of the cache changed (no append ran); and the next call with the default
limit, reusing the same workspace, is correct in full (outputs against the
oracle, the whole cache bit for bit)."""
import numpy as np
import pytest
import torch

import workloads as W
from helpers import from_np
from slot_cases import BF16_REL_TOL, Step, run_oracle

pytestmark = pytest.mark.gpu

CASES = [
    # name, family, sizes, kind, q_lens, fp8 (kernel "tc"; "tc5" for the
    # tcgen05 case, "unit" for the small-cache cases: clusters of 8 CTAs with
    # the capacity staged before the lengths, clusters of 2 over paged
    # blocks, one CTA a unit)
    ("decode_dense", "llama3_8b", dict(B=16, Smax=2048, len_lo=900, len_hi=2000, seed=701), "decode", None, False),
    ("decode_paged", "paged", dict(B=8, num_blocks=8 * 128, max_blocks=128, len_lo=900, len_hi=2000, seed=702),
     "decode", None, False),
    ("decode_e4m3", "llama3_8b", dict(B=16, Smax=2048, len_lo=900, len_hi=2000, seed=703), "decode", None, True),
    ("multi_rows16", "llama3_8b", dict(B=8, Smax=2048, len_lo=900, len_hi=2000, seed=704), "multi", [4] * 8,
     False),
    ("multi_rows32", "llama3_8b", dict(B=8, Smax=2048, len_lo=900, len_hi=2000, seed=705), "multi", [8] * 8,
     False),
    ("multi_rows32_tcgen05", "llama3_8b", dict(B=8, Smax=2048, len_lo=900, len_hi=2000, seed=706), "multi",
     [8] * 8, False),
    ("unit_f32_clusters", "pr1_fp32", dict(B=4, Smax=256, len_lo=1, len_hi=255, seed=707), "decode", None, False),
    ("unit_paged", "paged", dict(B=6, num_blocks=6 * 24, max_blocks=24, len_lo=1, len_hi=380, seed=708), "decode",
     None, False),
    ("unit_one_cta", "llama3_8b", dict(B=16, Smax=384, len_lo=1, len_hi=383, seed=709), "decode", None, False),
]


def _kernel(name):
    return "unit" if name.startswith("unit_") else ("tc5" if name.endswith("tcgen05") else "tc")


def _call(st, t, **kw):
    import gqa_kv_cache_gb300 as gqa
    w = st.w
    if st.fp8:
        kw.update(k_scale=t["k_scale"], v_scale=t["v_scale"])
    if st.multi:
        if w.paged:
            return gqa.decode_multi_paged(t["q"], t["k_new"], t["v_new"], t["k_blocks"], t["v_blocks"],
                                          t["block_table"], t["lengths"], t["cu_q"], max_q_len=max(st.qlen), **kw)
        return gqa.decode_multi(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["lengths"],
                                t["cu_q"], max_q_len=max(st.qlen), **kw)
    if w.paged:
        return gqa.decode_step_paged(t["q"], t["k_new"], t["v_new"], t["k_blocks"], t["v_blocks"],
                                     t["block_table"], t["lengths"], **kw)
    return gqa.decode_step(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["lengths"], **kw)


@pytest.mark.parametrize("name,base,kw,kind,q_lens,fp8", CASES, ids=[c[0] for c in CASES])
def test_wait_runs_out_then_next_call_is_correct(name, base, kw, kind, q_lens, fp8):
    w = W.small(base, **kw)
    st = Step(w, kind, q_lens=q_lens, fp8=fp8).finish()
    want = run_oracle(st)                       # appends into the host copies
    t = st.device()
    names = ("k_blocks", "v_blocks") if w.paged else ("k_cache", "v_cache")
    before = {n: t[n].clone() for n in names}
    appended = {n: from_np(st.host[n]).cuda() for n in names}   # the oracle's post-step caches
    vmax = st.vmax()

    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((t["q"].shape[0], w.Hq, w.D), 7.0, device="cuda")
    kernel = _kernel(name)
    _call(st, t, out=out, status=status, kernel=kernel, wait_limit_cycles=2000, test_stall=True)
    torch.cuda.synchronize()
    s = int(status.item())
    assert s == 8, f"status {s}: expected exactly the timeout bit"
    assert torch.isnan(out).all(), "an aborted step left an output that is not NaN"
    for n in names:
        now, was, new = (x.view(torch.uint8) for x in (t[n], before[n], appended[n]))
        if kernel == "unit":   # the append slots old or new, every other byte unchanged
            assert bool(((now == was) | (now == new)).all()), f"{n}: an aborted step changed more than its append"
        else:
            assert torch.equal(now, was), f"{n} changed by an aborted step"

    # the next call, default limit, same workspace: correct in full
    status.zero_()
    out2 = _call(st, t, status=status, kernel=kernel)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got2 = out2.double().cpu().numpy()
    assert np.isfinite(got2).all()
    assert np.abs(got2 - want).max() <= BF16_REL_TOL * vmax
    for n in names:
        assert torch.equal(t[n].view(torch.uint8), appended[n].view(torch.uint8)), f"{n} after the next call"
