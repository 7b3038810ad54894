"""GPU parity of the E4M3 (FP8) KV cache: OCP FP8 E4M3 bytes with one float32
scale per cache head (K = k_scale * K8, V = v_scale * V8; "groupQueryAttention"
names kScale / vScale without semantics, this reading is stated in the
oracle). The decode step quantises the appended token (float32 division by
the scale, round to nearest even, saturating): its bytes must equal the
oracle's bit for bit, the whole cache compared; outputs within 2e-2 max|V|
of the float64 oracle over the same bytes. Dense, slot_ids, paged, the
read-only attend, the softmax modifiers, full-size caches."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_cases import BF16_REL_TOL, guard, host_problem, path_of
from helpers import to_np

pytestmark = pytest.mark.gpu


def _gpu(w, t, attend=False, kernel="auto", grid=0, status=None, **mods):
    import gqa_kv_cache_gb300 as gqa
    kw = dict(kernel=kernel, grid_ctas=grid, status=status, k_scale=t["k_scale"], v_scale=t["v_scale"], **mods)
    if attend:
        if w.paged:
            return gqa.attend_paged(t["q"], t["k_blocks"], t["v_blocks"], t["block_table"], t["lengths"], **kw)
        return gqa.attend(t["q"], t["k_cache"], t["v_cache"], t["lengths"], t.get("slot_ids"), **kw)
    if w.paged:
        return gqa.decode_step_paged(t["q"], t["k_new"], t["v_new"], t["k_blocks"], t["v_blocks"],
                                     t["block_table"], t["lengths"], **kw)
    return gqa.decode_step(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["lengths"],
                           t.get("slot_ids"), **kw)


def _oracle(w, prob, attend, ks, vs, **mods):
    om = dict(k_scale=ks, v_scale=vs, window=mods.get("window", 0), kept_prefix=mods.get("kept_prefix", 0))
    if mods.get("sink") is not None:
        om["sink"] = mods["sink"].cpu().numpy()
    if attend:
        if w.paged:
            r = oracle.attend_paged(prob["q"], prob["k_blocks"], prob["v_blocks"], prob["block_table"],
                                    prob["lengths"], **om)
        else:
            r = oracle.attend_dense(prob["q"], prob["k_cache"], prob["v_cache"], prob["lengths"], **om)
    elif w.paged:
        r = oracle.decode_paged(prob["q"], prob["k_new"], prob["v_new"], prob["k_blocks"], prob["v_blocks"],
                                prob["block_table"], prob["lengths"], **om)
    else:
        r = oracle.decode_dense(prob["q"], prob["k_new"], prob["v_new"], prob["k_cache"], prob["v_cache"],
                                prob["lengths"], **om)
    assert r.status == oracle.OK
    return r.out


def _vmax(t, w, prob):
    """max |V| over the values the call attends (the valid slots of the
    compared rows, dequantised, and the new values)."""
    v = prob["v_blocks"] if w.paged else prob["v_cache"]
    vs = t["v_scale"].cpu().numpy()
    vf = torch.from_numpy(v).view(torch.float8_e4m3fn).double().numpy() * vs.reshape(1, -1, 1, 1)
    L = prob["lengths"]
    vals = [float(t["v_new"].float().abs().max().item())] if "v_new" in t else [0.0]
    # cached valid slots of row i: lengths[i] (decode: 0..L-1 and the new
    # value; attend: its L valid slots)
    if w.paged:
        bs = vf.shape[2]
        for i in range(len(L)):
            for s in range(int(L[i])):
                vals.append(float(np.abs(vf[prob["block_table"][i, s // bs], :, s % bs]).max()))
    else:
        for i in range(len(L)):
            if int(L[i]) > 0:
                vals.append(float(np.abs(vf[i, :, :int(L[i])]).max()))
    return max(vals)


def check_fp8(w, attend=False, q_f32=False, kernel="auto", grid=0, rows=None, gpu_gen=False, **mods):
    if gpu_gen:
        t = W.generate(w, "cuda", attend=attend, q_f32=q_f32, kv_e4m3=True)
    else:
        t = {k: v.cuda() for k, v in W.generate(w, "cpu", attend=attend, q_f32=q_f32, kv_e4m3=True).items()}
    if rows == "sample":
        rows = sorted({0, w.B - 1, int(torch.argmax(t["lengths"]).item())})
    prob = host_problem(w, t, rows)
    ks, vs = t["k_scale"].cpu().numpy(), t["v_scale"].cpu().numpy()
    names = ("k_blocks", "v_blocks") if w.paged else ("k_cache", "v_cache")
    before = {n: t[n].clone() for n in names} if attend else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _gpu(w, t, attend, kernel, grid, st, **mods)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    want = _oracle(w, prob, attend, ks, vs, **mods)          # appends into the host copies
    sel = torch.tensor(prob["rows"], device="cuda")
    got = out[sel].double().cpu().numpy()
    assert np.isfinite(got).all()
    err = float(np.abs(got - want).max())
    vmax = _vmax(t, w, prob)
    tol = BF16_REL_TOL * vmax
    assert err <= tol, f"max abs error {err} > {tol}"
    guard(path_of(w, kernel, fp8=True), err, vmax)
    if attend:
        for n in names:
            assert torch.equal(before[n], t[n]), f"{n} written by a read-only attend"
    elif w.paged:
        idx = torch.tensor(prob["blocks"], dtype=torch.long, device="cuda")
        for n in names:
            assert to_np(t[n][idx]).tobytes() == prob[n].tobytes(), f"{n}: appended bytes differ"
    else:
        idx = torch.tensor(prob["cache_rows"], dtype=torch.long, device="cuda")
        for n in names:
            assert to_np(t[n][idx]).tobytes() == prob[n].tobytes(), f"{n}: appended bytes differ"
    return err, tol


CASES = [
    ("dense_g4", "llama3_8b", dict(B=5, Smax=700, len_lo=0, len_hi=699, seed=501)),
    ("dense_g8", "long_context", dict(B=3, Smax=1000, len_lo=60, len_hi=999, seed=502)),
    ("slots_g8", "ragged_slots", dict(B=6, R=11, Smax=600, len_lo=1, len_hi=599, seed=503)),
    ("paged16_g6", "paged", dict(B=5, num_blocks=5 * 40, max_blocks=40, len_lo=0, len_hi=639, seed=504)),
    ("paged8_g4", "paged", dict(Hq=8, Hkv=2, B=3, block_size=8, num_blocks=3 * 50, max_blocks=50,
                                len_lo=0, len_hi=399, seed=505)),
    ("dense_g3", "llama3_8b", dict(Hq=6, Hkv=2, B=2, Smax=300, len_lo=0, len_hi=299, seed=506)),
]


@pytest.mark.parametrize("name,base,kw", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("grid", [0, 7])
def test_fp8_decode(name, base, kw, grid):
    check_fp8(W.small(base, **kw), grid=grid)


@pytest.mark.parametrize("q_f32", [True, False], ids=["q_f32", "q_bf16"])
@pytest.mark.parametrize("name,base,kw", CASES[:4], ids=[c[0] for c in CASES[:4]])
def test_fp8_attend(name, base, kw, q_f32):
    check_fp8(W.small(base, **kw), attend=True, q_f32=q_f32)


def test_fp8_window_sink():
    w = W.small("llama3_8b", B=4, Smax=900, len_lo=200, len_hi=899, seed=507)
    g = torch.Generator().manual_seed(5)
    check_fp8(w, window=150, kept_prefix=20, sink=torch.randn(w.Hq, generator=g).cuda())


def test_fp8_stale_bytes_never_matter():
    """Stale slots hold NaN codes (0x7F): no output bit changes."""
    w = W.small("llama3_8b", B=4, Smax=400, len_lo=0, len_hi=398, seed=508)
    t = {k: v.cuda() for k, v in W.generate(w, kv_e4m3=True).items()}
    ref = _gpu(w, {k: v.clone() for k, v in t.items()}).clone()
    j = torch.arange(w.Smax, device="cuda")
    stale = (j[None, :] >= t["lengths"].long()[:, None] + 1)[:, None, :, None]
    t2 = {k: v.clone() for k, v in t.items()}
    t2["k_cache"] = torch.where(stale, torch.full_like(t["k_cache"], 0x7F), t["k_cache"])
    t2["v_cache"] = torch.where(stale, torch.full_like(t["v_cache"], 0x7F), t["v_cache"])
    assert torch.equal(_gpu(w, t2), ref)


def test_fp8_argument_errors():
    import gqa_kv_cache_gb300 as gqa
    w = W.small("llama3_8b", B=2, Smax=128, len_lo=1, len_hi=100, seed=509)
    t = {k: v.cuda() for k, v in W.generate(w, kv_e4m3=True).items()}
    with pytest.raises(gqa.GqaError):           # no scales
        gqa.decode_step(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["lengths"])
    with pytest.raises(gqa.GqaError):           # the CUDA-core kernel takes no E4M3 cache
        _gpu(w, t, kernel="simt")


@pytest.mark.parametrize("name", ["llama3_8b", "paged"])
def test_fp8_full_size(name):
    check_fp8(W.WORKLOADS[name], rows="sample", gpu_gen=True)
