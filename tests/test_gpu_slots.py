"""GPU parity that sees every single slot (constructions in slot_cases.py):
a dominant slot per unit, placed at tile edges, CTA cuts, the new token and
the last slot, must come out as its own value; a zero query must give the
mean of exactly the attended values. Either check fails for a kernel that
drops, duplicates or misplaces one slot, which the stated bar on random data
(2e-2 max|V| for bfloat16) cannot see.

Covered: the bfloat16 single-token tensor-core kernel (dense, slot ids,
paged blocks of 16 and 8; the default grid, 7 and 33 CTAs so units are cut),
the CUDA-core kernel, the small-cache kernel (decode and attend; the
dominant slot at the edges of the parts a cluster of CTAs shares out), the
read-only attend (bfloat16 and float32 query, bfloat16 and E4M3 caches), the
E4M3 decode kernels, the multi-token units of up to 8, 16 and 32 query
rows (and a step of two chunks), and the opt-in tcgen05 form of the units
of more than 16 rows."""
import pytest
import torch

import workloads as W
from slot_cases import MULTI, SINGLE, UNIT, Step, check_dominant, check_uniform, plant_dominant, run_oracle

pytestmark = pytest.mark.gpu


def run_gpu(st, kernel="auto", grid=0):
    import gqa_kv_cache_gb300 as gqa
    w, t = st.w, st.device()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = dict(kernel=kernel, grid_ctas=grid, status=status)
    if st.fp8:
        kw.update(k_scale=t["k_scale"], v_scale=t["v_scale"])
    if st.multi:
        mq = max(max(st.qlen), 1)
        if w.paged:
            out = gqa.decode_multi_paged(t["q"], t["k_new"], t["v_new"], t["k_blocks"], t["v_blocks"],
                                         t["block_table"], t["lengths"], t["cu_q"], max_q_len=mq, **kw)
        else:
            out = gqa.decode_multi(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["lengths"],
                                   t["cu_q"], t.get("slot_ids"), max_q_len=mq, **kw)
    elif st.attend:
        if w.paged:
            out = gqa.attend_paged(t["q"], t["k_blocks"], t["v_blocks"], t["block_table"], t["lengths"], **kw)
        else:
            out = gqa.attend(t["q"], t["k_cache"], t["v_cache"], t["lengths"], t.get("slot_ids"), **kw)
    elif w.paged:
        out = gqa.decode_step_paged(t["q"], t["k_new"], t["v_new"], t["k_blocks"], t["v_blocks"],
                                    t["block_table"], t["lengths"], **kw)
    else:
        out = gqa.decode_step(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["lengths"],
                              t.get("slot_ids"), **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    return out.double().cpu().numpy()


def dominant(st, seed, kernel, grid, cut_grid=None, unit_parts=False):
    dom = plant_dominant(st, seed, grid if cut_grid is None else cut_grid, unit_parts)
    st.finish()
    got = run_gpu(st, kernel, grid)
    check_dominant(st, dom, got, run_oracle(st))


def uniform(st, kernel, grid):
    st.t["q"].zero_()
    st.finish()
    got = run_gpu(st, kernel, grid)
    check_uniform(st, got, run_oracle(st))


@pytest.mark.parametrize("grid", [0, 7, 33])
@pytest.mark.parametrize("kernel", ["tc", "simt"])
@pytest.mark.parametrize("name,base,kw", SINGLE, ids=[c[0] for c in SINGLE])
def test_dominant_decode(name, base, kw, kernel, grid):
    st = Step(W.small(base, **kw), "decode")
    # cut positions are those of the tensor-core kernel's 64-slot tiles
    dominant(st, 11, kernel, grid, cut_grid=grid if kernel == "tc" else 0)


@pytest.mark.parametrize("grid", [0, 33])
@pytest.mark.parametrize("name,base,kw", SINGLE, ids=[c[0] for c in SINGLE])
def test_dominant_decode_e4m3(name, base, kw, grid):
    dominant(Step(W.small(base, **kw), "decode", fp8=True), 12, "tc", grid)


@pytest.mark.parametrize("q_f32", [False, True], ids=["q_bf16", "q_f32"])
@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("name,base,kw", [SINGLE[0], SINGLE[3]], ids=["dense_g4", "paged16_g6"])
def test_dominant_attend(name, base, kw, fp8, q_f32):
    st = Step(W.small(base, **dict(kw, len_lo=1)), "attend", fp8=fp8, q_f32=q_f32)
    dominant(st, 13, "tc", 33)


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("grid", [0, 7])
@pytest.mark.parametrize("name,base,kw,q_lens", MULTI, ids=[c[0] for c in MULTI])
def test_dominant_multi(name, base, kw, q_lens, grid, fp8):
    dominant(Step(W.small(base, **kw), "multi", q_lens=q_lens, fp8=fp8), 14, "tc", grid)


# the multi-token cases with units of more than 16 query rows
MULTI_T5 = [c for c in MULTI if c[0] in ("rows18_g6_paged16", "rows32_g4", "rows40_g8")]


@pytest.mark.parametrize("grid", [0, 7])
@pytest.mark.parametrize("name,base,kw,q_lens", MULTI_T5, ids=[c[0] for c in MULTI_T5])
def test_dominant_multi_tcgen05(name, base, kw, q_lens, grid):
    dominant(Step(W.small(base, **kw), "multi", q_lens=q_lens), 14, "tc5", grid)


@pytest.mark.parametrize("grid", [0, 7])
@pytest.mark.parametrize("name,base,kw,q_lens", MULTI_T5, ids=[c[0] for c in MULTI_T5])
def test_zero_query_multi_tcgen05(name, base, kw, q_lens, grid):
    uniform(Step(W.small(base, **kw), "multi", q_lens=q_lens), "tc5", grid)


@pytest.mark.parametrize("grid", [0, 7, 33])
@pytest.mark.parametrize("kernel", ["tc", "simt"])
@pytest.mark.parametrize("name,base,kw", SINGLE, ids=[c[0] for c in SINGLE])
def test_zero_query_decode(name, base, kw, kernel, grid):
    uniform(Step(W.small(base, **kw), "decode"), kernel, grid)


@pytest.mark.parametrize("grid", [0, 33])
@pytest.mark.parametrize("name,base,kw", SINGLE, ids=[c[0] for c in SINGLE])
def test_zero_query_decode_e4m3(name, base, kw, grid):
    uniform(Step(W.small(base, **kw), "decode", fp8=True), "tc", grid)


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("name,base,kw", [SINGLE[0], SINGLE[3]], ids=["dense_g4", "paged16_g6"])
def test_zero_query_attend(name, base, kw, fp8):
    uniform(Step(W.small(base, **dict(kw, len_lo=1)), "attend", fp8=fp8), "tc", 33)


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("grid", [0, 7])
@pytest.mark.parametrize("name,base,kw,q_lens", MULTI, ids=[c[0] for c in MULTI])
def test_zero_query_multi(name, base, kw, q_lens, grid, fp8):
    uniform(Step(W.small(base, **kw), "multi", q_lens=q_lens, fp8=fp8), "tc", grid)


@pytest.mark.parametrize("kind", ["decode", "attend"])
@pytest.mark.parametrize("name,base,kw", UNIT, ids=[c[0] for c in UNIT])
def test_dominant_small_cache_kernel(name, base, kw, kind):
    w = W.small(base, **(dict(kw, len_lo=1) if kind == "attend" else kw))
    dominant(Step(w, kind), 15, "unit", 0, unit_parts=True)


@pytest.mark.parametrize("kind", ["decode", "attend"])
@pytest.mark.parametrize("name,base,kw", UNIT, ids=[c[0] for c in UNIT])
def test_zero_query_small_cache_kernel(name, base, kw, kind):
    w = W.small(base, **(dict(kw, len_lo=1) if kind == "attend" else kw))
    uniform(Step(w, kind), "unit", 0)
