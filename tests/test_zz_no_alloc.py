"""gqa_decode_step_noalloc: the decode step for callers that cannot allocate.

Some callers cannot hand the library a workspace (a plugin host that gives an
operator no scratch and forbids device allocation while it runs, or a plain C
caller with no device allocator). The no-allocation entry point keeps its
scratch in a fixed array inside the library. These tests call it through the
C ABI and check that two calls in a row give the output of the regular entry
point (which takes a caller-owned workspace) within the float32 / bfloat16
bars the other parity tests use, and that sizes beyond the fixed scratch are
refused before anything runs. The file is named so that pytest collects it
last.
"""
import ctypes

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

F32_TOL, BF16_REL_TOL = 1e-5, 2e-2
DTYPE = {torch.float32: 0, torch.bfloat16: 1}


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _regular(lib, t, w, out, stream):
    need = lib.gqa_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, DTYPE[t["q"].dtype], None)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")   # zero-filled before first use
    return lib.gqa_decode_step(_p(t["q"]), _p(t["k_new"]), _p(t["v_new"]), _p(t["k_cache"]),
                               _p(t["v_cache"]), _p(t["lengths"]), _p(t.get("slot_ids")), _p(out),
                               w.B, w.Hq, w.Hkv, w.D, w.rows, w.Smax, DTYPE[t["q"].dtype],
                               _p(ws), need, None, stream)


def _noalloc(lib, t, w, out, stream):
    return lib.gqa_decode_step_noalloc(_p(t["q"]), _p(t["k_new"]), _p(t["v_new"]), _p(t["k_cache"]),
                                       _p(t["v_cache"]), _p(t["lengths"]), _p(t.get("slot_ids")),
                                       _p(out), w.B, w.Hq, w.Hkv, w.D, w.rows, w.Smax,
                                       DTYPE[t["q"].dtype], None, stream)


CASES = [
    W.small("llama3_8b", B=4, Smax=700, len_lo=0, len_hi=699, seed=200),               # bf16, tensor cores
    W.small("ragged_slots", B=6, R=11, Smax=600, len_lo=1, len_hi=599, seed=201),      # bf16, slot_ids
    W.small("pr1_fp32", B=3, Smax=300, len_lo=0, len_hi=299, seed=202),                # fp32, CUDA cores
]


@pytest.mark.parametrize("w", CASES, ids=[c.name + "_" + c.dtype for c in CASES])
def test_noalloc_matches_regular_entry_point(w):
    import gqa_kv_cache_gb300 as gqa
    lib = gqa._lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t = {k: v.cuda() for k, v in W.generate(w, "cpu").items()}
    ref = torch.empty(w.B, w.Hq, w.D, dtype=torch.float32, device="cuda")
    assert _regular(lib, {k: v.clone() for k, v in t.items()}, w, ref, stream) == 0
    torch.cuda.synchronize()
    vmax = float(t["v_cache"].float().abs().max().item())
    tol = F32_TOL if w.dtype == "f32" else BF16_REL_TOL * vmax
    kc0, vc0 = t["k_cache"].clone(), t["v_cache"].clone()
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _noalloc(lib, t, w, out, stream) == 0
        torch.cuda.synchronize()
        err = (out - ref).abs().max().item()
        assert err <= tol, f"call {call}: max abs error {err} > {tol}"
        if call == 0:
            # a regular call on its own workspace in between leaves the shared scratch alone
            mid = torch.empty_like(ref)
            assert _regular(lib, {k: v.clone() for k, v in t.items()}, w, mid, stream) == 0
            torch.cuda.synchronize()
            assert (mid - ref).abs().max().item() <= tol
    # the append happened in place (one slot per row and head, K and V), as with the regular call
    L = t["lengths"].long()
    rows = t["slot_ids"].long() if "slot_ids" in t else torch.arange(w.B, device="cuda")
    kc0[rows, :, L] = t["k_new"]
    vc0[rows, :, L] = t["v_new"]
    assert torch.equal(kc0, t["k_cache"])
    assert torch.equal(vc0, t["v_cache"])


def test_noalloc_refuses_sizes_beyond_its_scratch():
    import gqa_kv_cache_gb300 as gqa
    lib = gqa._lib.load()
    cap = lib.gqa_noalloc_scratch_bytes()
    assert cap >= 1 << 20
    B = 100000                                           # needs far more than the fixed scratch
    assert lib.gqa_workspace_bytes(B, 64, 8, 128, 1, None) > cap
    dummy = ctypes.c_void_p(256)
    rc = lib.gqa_decode_step_noalloc(dummy, dummy, dummy, dummy, dummy, dummy, None, dummy,
                                     B, 64, 8, 128, B, 16, 1, None, None)
    assert rc == 5
    assert b"noalloc" in lib.gqa_status_string(5)
