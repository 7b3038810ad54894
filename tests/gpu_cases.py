"""Shared driver for the GPU parity tests: run one decode step through the
library (C ABI, via the Python binding) and the same step through the CPU
oracle on identical seeded inputs, then compare.

Bars (the decode step's stated accuracy):
  * append and addressing: bit-exact, the whole cache compared;
  * float32 data: max |out - oracle| <= 1e-5;
  * bfloat16 data: max |out - oracle| <= 2e-2 * max|V| over the attended
    values, the oracle running on the same bf16 bits.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W
from helpers import to_np

F32_TOL = 1e-5
BF16_REL_TOL = 2e-2

# Regression guards, per arithmetic path: the largest error relative to
# max|V| observed on GB300 over the random parity cases, times 5. They sit far
# inside the stated bar (2e-2 max|V| for bfloat16 and E4M3 caches), which
# stays the acceptance criterion; a guard catches a kernel change that loses
# accuracy long before that bar would. Paths: "tc_bf16" (P as bf16 + bf16
# remainder), "tc_bf16_q32" (float32 query split in two), "tc_bf16_m16"
# (16-row multi-token units, P in bf16), "tc_e4m3" / "tc_e4m3_m16" (P in f16),
# "simt_bf16" (CUDA-core FMA), "unit_bf16" (the small-cache kernel, FMA).
# Float32 caches keep their absolute 1e-5 bar.
GUARD = {"tc_bf16": 1.2e-5, "tc_bf16_q32": 2e-5, "tc_bf16_m16": 8e-3, "tc_e4m3": 1.2e-3,
         "tc_e4m3_m16": 1.2e-3, "simt_bf16": 2e-6, "unit_bf16": 3e-7, "tc5_bf16": 8e-3}
OBSERVED = []   # (test id, path, error / max|V|), written out by conftest


UNIT_SMEM_MAX = 200 * 1024


def supports(kernel: str, w: W.Workload) -> bool:
    """Whether the kernel asked for takes these sizes (single-token steps):
    the CUDA-core kernel takes every size; the tensor-core kernel bfloat16,
    D = 128, G <= 8, paged blocks a power of two >= 8; the small-cache kernel
    float32 or bfloat16, D in {32, 64, 128, 256}, G <= 8 and K and V of a
    row's capacity within 200 KB of shared memory."""
    if kernel in ("simt", "auto"):
        return True
    if kernel == "tc":
        return w.dtype == "bf16" and w.D == 128 and w.G <= 8 and (
            not w.paged or (w.block_size >= 8 and (w.block_size & (w.block_size - 1)) == 0))
    if kernel == "unit":
        cap = w.max_blocks * w.block_size if w.paged else w.Smax
        return w.D in (32, 64, 128, 256) and w.G <= 8 and 2 * cap * w.D * w.elem_bytes <= UNIT_SMEM_MAX
    raise ValueError(kernel)


def path_of(w: W.Workload, kernel="auto", fp8=False, q_f32=False, unit_rows=None):
    """Arithmetic path a call takes: the kernel ("auto" resolved as the
    library does) and the form of its products."""
    tc_ok = w.dtype == "bf16" and w.D == 128 and w.G <= 8 and (
        not w.paged or (w.block_size >= 8 and (w.block_size & (w.block_size - 1)) == 0))
    if w.dtype == "f32":
        return None
    if kernel == "unit":
        return "unit_bf16"
    if kernel == "tc5" and not fp8 and unit_rows is not None and unit_rows > 16:
        return "tc5_bf16"
    tc = kernel in ("tc", "tc5") or (kernel == "auto" and tc_ok) or fp8
    if not tc:
        return "simt_bf16"
    m16 = unit_rows is not None and unit_rows > 8
    if fp8:
        return "tc_e4m3_m16" if m16 else "tc_e4m3"
    if m16:
        return "tc_bf16_m16"
    return "tc_bf16_q32" if q_f32 else "tc_bf16"


def guard(path, err, vmax):
    """Records the error of a parity case and holds it to its path's guard."""
    import os
    if path is None or vmax <= 0:
        return
    rel = err / vmax
    OBSERVED.append((os.environ.get("PYTEST_CURRENT_TEST", ""), path, rel))
    if path in GUARD:
        assert rel <= GUARD[path], f"regression guard {path}: error {rel:.3e} max|V| > {GUARD[path]:.1e} max|V|"


def tolerance(w: W.Workload, vmax: float) -> float:
    return F32_TOL if w.dtype == "f32" else BF16_REL_TOL * vmax


def make_inputs(w: W.Workload, on_gpu_generation: bool = False):
    """Inputs on cuda:0. Small cases are drawn on the CPU and copied (so the
    oracle sees the very same values); large ones are drawn on the GPU."""
    if on_gpu_generation:
        return W.generate(w, "cuda")
    t = W.generate(w, "cpu")
    return {k: v.cuda() for k, v in t.items()}


def _sample_rows(w, rows):
    return list(range(w.B)) if rows is None else sorted(set(int(r) for r in rows))


def host_problem(w: W.Workload, t: dict, rows=None):
    """Host copies of what the oracle needs for batch rows `rows` (all when
    None), taken BEFORE the GPU step runs. Dense/slot_ids: the rows' cache
    rows become a compact cache addressed by slot_ids 0..n-1. Paged: the rows'
    blocks become a compact block pool with a renumbered table. Returns
    (problem dict, mapping back to the original storage)."""
    rows = _sample_rows(w, rows)
    sel = torch.tensor(rows, dtype=torch.long, device=t["q"].device)
    prob = {k: to_np(t[k][sel]) for k in ("q", "k_new", "v_new", "lengths") if k in t}
    prob["rows"] = rows
    if w.paged:
        bt = t["block_table"][sel].cpu().numpy()
        used = sorted(set(int(x) for x in bt[bt >= 0].tolist()))
        remap = {blk: i for i, blk in enumerate(used)}
        idx = torch.tensor(used, dtype=torch.long, device=t["q"].device)
        prob["k_blocks"] = to_np(t["k_blocks"][idx])
        prob["v_blocks"] = to_np(t["v_blocks"][idx])
        prob["block_table"] = np.vectorize(lambda x: remap.get(int(x), -1))(bt).astype(np.int32) \
            if bt.size else bt.astype(np.int32)
        prob["blocks"] = used
        return prob
    cache_rows = (t["slot_ids"][sel].long() if "slot_ids" in t else sel)
    prob["k_cache"] = to_np(t["k_cache"][cache_rows])
    prob["v_cache"] = to_np(t["v_cache"][cache_rows])
    prob["cache_rows"] = cache_rows.cpu().tolist()
    return prob


def run_oracle(w: W.Workload, prob: dict):
    """Oracle on the host problem (appends into the host copies)."""
    if w.paged:
        r = oracle.decode_paged(prob["q"], prob["k_new"], prob["v_new"], prob["k_blocks"],
                                prob["v_blocks"], prob["block_table"], prob["lengths"])
    else:
        r = oracle.decode_dense(prob["q"], prob["k_new"], prob["v_new"], prob["k_cache"],
                                prob["v_cache"], prob["lengths"])
    assert r.status == oracle.OK
    return r.out


def run_gpu(w: W.Workload, t: dict, kernel="auto", grid_ctas=0, status=None):
    import gqa_kv_cache_gb300 as gqa
    if w.paged:
        return gqa.decode_step_paged(t["q"], t["k_new"], t["v_new"], t["k_blocks"], t["v_blocks"],
                                     t["block_table"], t["lengths"], kernel=kernel,
                                     grid_ctas=grid_ctas, status=status)
    return gqa.decode_step(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["lengths"],
                           t.get("slot_ids"), kernel=kernel, grid_ctas=grid_ctas, status=status)


def attended_vmax(prob: dict) -> float:
    """max |V| over the values the call attends: the valid slots below
    lengths[b] and, in the decode step, the new value."""
    vals = [np.abs(_as_float(prob["v_new"])).max()] if "v_new" in prob else [0.0]
    L = prob["lengths"]
    if "k_blocks" in prob:
        vb = _as_float(prob["v_blocks"])
        bs = vb.shape[2]
        for i in range(len(L)):
            for s in range(int(L[i])):
                vals.append(np.abs(vb[prob["block_table"][i, s // bs], :, s % bs]).max())
    else:
        vc = _as_float(prob["v_cache"])
        for i in range(len(L)):
            if L[i] > 0:
                vals.append(np.abs(vc[i, :, :L[i]]).max())
    return float(max(vals))


def _as_float(a):
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a


def check_step(w: W.Workload, kernel="auto", grid_ctas=0, rows=None, gpu_gen=False,
               full_cache_check=True):
    """Runs one step on the GPU and compares with the oracle. Returns
    (max abs error, tolerance, gpu out) for the compared rows."""
    t = make_inputs(w, gpu_gen)
    if rows == "sample4":   # first, last, longest and one random batch row
        L = t["lengths"]
        rows = [0, w.B - 1, int(torch.argmax(L).item()),
                int(np.random.default_rng(w.seed).integers(0, w.B))]
    prob = host_problem(w, t, rows)
    names = ("k_blocks", "v_blocks") if w.paged else ("k_cache", "v_cache")
    before = {n: t[n].clone() for n in names} if full_cache_check else None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_gpu(w, t, kernel, grid_ctas, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    want = run_oracle(w, prob)
    sel = prob["rows"]
    got = out[torch.tensor(sel, device="cuda")].double().cpu().numpy()
    err = float(np.abs(got - want).max())
    vmax = attended_vmax(prob)
    tol = tolerance(w, vmax)
    assert np.isfinite(got).all()
    guard(path_of(w, kernel), err, vmax)
    # append / addressing: the GPU's post-step storage at the sampled rows
    # equals the oracle's post-step host copies, bit for bit
    if w.paged:
        idx = torch.tensor(prob["blocks"], dtype=torch.long, device="cuda")
        for n in names:
            assert to_np(t[n][idx]).tobytes() == prob[n].tobytes(), f"{n} differs after the append"
    else:
        idx = torch.tensor(prob["cache_rows"], dtype=torch.long, device="cuda")
        for n in names:
            assert to_np(t[n][idx]).tobytes() == prob[n].tobytes(), f"{n} differs after the append"
    if full_cache_check:
        _check_whole_cache(w, t, before)
    return err, tol, out


def _check_whole_cache(w, t, before):
    """Everywhere: post-step storage == pre-step storage with exactly the
    append slots replaced by k_new / v_new (device-side comparison)."""
    B = w.B
    L = t["lengths"].long()
    b = torch.arange(B, device="cuda")
    for name, new in ((0, "k_new"), (1, "v_new")):
        n = ("k_blocks", "v_blocks")[name] if w.paged else ("k_cache", "v_cache")[name]
        exp = before[n]
        if w.paged:
            blk = t["block_table"][b, L // w.block_size].long()
            exp[blk, :, L % w.block_size] = t[new]
        else:
            r = t["slot_ids"].long() if "slot_ids" in t else b
            exp[r, :, L] = t[new]
        assert torch.equal(exp.view(torch.int16) if exp.dtype == torch.bfloat16 else exp.view(torch.int32),
                           t[n].view(torch.int16) if exp.dtype == torch.bfloat16 else t[n].view(torch.int32)), \
            f"{n}: bytes outside the append slots changed, or the append is wrong"
