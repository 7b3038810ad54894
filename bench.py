#!/usr/bin/env python
"""Benchmark of the GQA decode step over a KV cache on one GB300.

A step is one call of the library's decode step (in-place append, split-S
attention, log-sum-exp combine) over the whole synthetic batch of a workload.

By default every one of the five decode workloads is measured in turn (each
generated, timed and freed before the next):

  pr1_fp32      fp32, B=2, Hq=8, Hkv=2, D=64, Smax=256
  llama3_8b     bf16, B=32, Hq=32, Hkv=8, D=128, Smax=4096
  long_context  bf16, B=4, Hq=64, Hkv=8, D=128, Smax=131072
  ragged_slots  bf16, B=256 of 512 rows, Hq=32, Hkv=4, D=128, Smax=8192
  paged         bf16, B=64, Hq=48, Hkv=8, D=128, 65536 blocks of 16 slots

and ONE JSON line is printed (rank 0) whose headline is `paged`, the largest
workload by KV bytes read per step (2.2 GB), with every workload's own
figures under `per_config`. `--workload NAME` measures that one alone.

Per workload:
  value     KV-cache bytes the step must read (sum_b lengths[b]*Hkv*D*2*es)
            divided by the device time of the step, in GB/s, inputs resident
            in HBM, L2 flushed between timed steps (a 256 MB write and then a
            256 MB read, outside the events, so L2 is cold and holds no dirty
            lines whose write-back would fall inside the next step);
  e2e       the same metric through the public API with the step's inputs
            copied from pinned host memory (one staging buffer, one copy) and
            the output read back, every step;
  roofline  the decode kernel alone (CUDA events around its launches) against
            the measured HBM copy bandwidth, with the per-launch DRAM traffic
            of the committed ncu capture of that kernel and workload;
  cpu_baseline  the float64 CPU oracle on this machine's host cores over a
            bounded sample of the workload's batch rows.
With --impl reference the oracle itself is timed as the reference arm.

--op attend times the read-only attend instead (no append; lengths count the
valid slots; a float32 query over the workload's cache unless --q-dtype cache).
--window W / --kept-prefix P / --sink add the softmax modifiers; the KV bytes
then count only the slots inside the window or the prefix.
--kv e4m3 stores the cache as E4M3 (FP8) bytes with per-head scales (the KV
bytes are then one per element; q, k_new, v_new stay bfloat16).
--q-len N times the multi-token step (N new tokens per row, causal); its KV
bytes count the cached slots once (a row whose tokens span several chunks
streams them once per chunk, which shows in the roofline).

Multi-GPU (torchrun): every rank runs an independent replica with its own
batch (weak scaling, no data-path collective); times are max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV-cache HBM GB/s & fraction of ~8 TB/s peak; µs per GQA decode step"
METRIC_ATTEND = "KV-cache HBM GB/s & fraction of ~8 TB/s peak; µs per GQA read-only attend"
METRIC_MULTI = "KV-cache HBM GB/s & fraction of ~8 TB/s peak; µs per GQA multi-token decode step"
UNIT = "GB/s"
NOMINAL_HBM_GBPS = 8000.0
FALLBACK_HBM_GBPS = 6800.0
L2_FLUSH_BYTES = 256 << 20
SUITE = ["pr1_fp32", "llama3_8b", "long_context", "ragged_slots", "paged"]
HEADLINE = "paged"          # the largest workload by KV bytes read per step
CPU_SAMPLE_KV_BYTES = 192 << 20   # KV bytes of one CPU-baseline pass (bounded sample)
REF_SAMPLE_KV_BYTES = 64 << 20    # KV bytes of one reference-arm step


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="all",
                    help="one workload, or 'all' (default): the five, headline " + HEADLINE)
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "tc", "tc5"])
    ap.add_argument("--op", default="decode", choices=["decode", "attend"],
                    help="decode step (default) or the read-only attend")
    ap.add_argument("--q-dtype", default=None, choices=["cache", "f32"],
                    help="attend only: query dtype (default f32)")
    ap.add_argument("--window", type=int, default=0, help="sliding window W (0: none)")
    ap.add_argument("--kept-prefix", type=int, default=0, help="kept prefix P (with a window)")
    ap.add_argument("--sink", action="store_true", help="a per-head sink logit (seeded N(0,1))")
    ap.add_argument("--q-len", type=int, default=0, help="multi-token step with this many new tokens per row")
    ap.add_argument("--kv", default="native", choices=["native", "e4m3"],
                    help="cache element type: the workload's own or E4M3 bytes with per-head scales")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shrink", type=int, default=1,
                    help="divide the batch (and the cache rows / paged blocks) by this factor: a "
                         "smaller instance of the same shapes and length law, for ncu captures")
    ap.add_argument("--clocks-dir", default=None,
                    help="folder for the raw nvidia-smi samples of the timed region (default: the temp dir)")
    ap.add_argument("--sched-pad", type=int, default=None,
                    help="schedule-only tiles per (row, head); default: the library's")
    ap.add_argument("--l2-flush", default="write_read", choices=["write_read", "write", "none"],
                    help="between timed steps: write 256 MB then read another 256 MB (L2 cold "
                         "and clean), write only (dirty lines left to write back), or nothing")
    return ap.parse_args()


# ------------------------------------------------------------------ ranks --

class Ranks:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------- workload ----

def workload(name, rank, shrink=1):
    """The named workload; rank r > 0 draws its own batch (seed + 1000 r).
    shrink > 1: B, the dense rows and the paged block pool divided by it (the
    same G, D, block size and length law; a paged table still gets distinct
    blocks)."""
    import workloads as W
    from dataclasses import replace
    w = W.WORKLOADS[name]
    if rank:
        w = replace(w, seed=w.seed + 1000 * rank)
    if shrink > 1:
        w = replace(w, B=max(1, w.B // shrink), R=max(1, w.R // shrink) if w.R else 0,
                    num_blocks=max(1, w.num_blocks // shrink) if w.paged else 0,
                    name=f"{w.name}/shrink{shrink}")
    return w


def cached_slots_read(L, attend, window=0, kept_prefix=0):
    """Cached slots each row's step must read: the decode step reads slots
    0..L-1 (slot L = lengths[b] comes from k_new / v_new), the attend slots
    0..L-1 with L = lengths[b]; with a window W only those above L' - W (L' the
    query position) and those below the kept prefix P."""
    import torch
    L = L.to(torch.int64)
    if not window:
        return L
    last = L - 1 if attend else L                      # query position
    lo = torch.clamp(last - window + 1, min=0)
    return (L - lo) + torch.clamp(lo, max=kept_prefix)


def algorithmic_bytes_multi(w, t, kv_es=None) -> dict:
    """Multi-token step: every cached slot read once, the new tokens' K/V
    read (their own dtype) and appended (cache element bytes), q read, out
    written, index reads."""
    import torch
    L = t["lengths"].to(torch.int64)
    es = w.elem_bytes
    kes = es if kv_es is None else kv_es      # cache element bytes (1 for E4M3)
    T = t["q"].shape[0]
    kv = int(L.sum().item()) * w.Hkv * w.D * 2 * kes
    new_read = T * w.Hkv * w.D * es * 2
    new_write = T * w.Hkv * w.D * kes * 2
    q = t["q"].numel() * t["q"].element_size()
    out = T * w.Hq * w.D * 4
    idx = w.B * 4 * (3 if w.slot_ids else 2)
    if w.paged:
        ql = (t["cu_q"][1:] - t["cu_q"][:-1]).to(torch.int64)
        idx += int(((L + ql + w.block_size - 1) // w.block_size).sum().item()) * 4
    return {"kv_read": kv, "append_write": new_write, "new_kv_read": new_read, "q_read": q, "out_write": out,
            "index_read": idx, "total": kv + new_read + new_write + q + out + idx}


def algorithmic_bytes(w, t, attend=False, window=0, kept_prefix=0, kv_es=None) -> dict:
    """Bytes the step must move (no split partials): the KV read, the append
    write, the new K/V, q, out and the index reads. The decode step reads the
    lengths[b] cached slots (slot lengths[b] comes from k_new / v_new); the
    read-only attend reads its lengths[b] valid slots and appends nothing; a
    window and kept prefix cut both to the attended slots."""
    import torch
    L = t["lengths"].to(torch.int64)
    es = w.elem_bytes
    kes = es if kv_es is None else kv_es      # cache element bytes (1 for E4M3)
    kv = int(cached_slots_read(L, attend, window, kept_prefix).sum().item()) * w.Hkv * w.D * 2 * kes
    # the new token's K and V: read (their own dtype) and appended (cache element bytes)
    new_read = 0 if attend else 2 * w.B * w.Hkv * w.D * es
    new_write = 0 if attend else 2 * w.B * w.Hkv * w.D * kes
    new = new_read + new_write
    idx = w.B * 4 * (2 if w.slot_ids else 1)
    if w.paged:
        touched = L if attend else L + 1
        idx += int(((touched + w.block_size - 1) // w.block_size).sum().item()) * 4
    q = t["q"].numel() * t["q"].element_size()
    return {"kv_read": kv, "append_write": new_write, "new_kv_read": new_read,
            "q_read": q, "out_write": w.B * w.Hq * w.D * 4, "index_read": idx,
            "total": kv + new + q + w.B * w.Hq * w.D * 4 + idx}


def step_fn(w, t, kernel, out, sched_pad=None, attend=False, mods=None, max_q=0):
    import gqa_kv_cache_gb300 as gqa
    kw = dict(out=out, kernel=kernel, sched_pad=sched_pad, **(mods or {}))
    if max_q and w.paged:
        def run(tt=t):
            gqa.decode_multi_paged(tt["q"], tt["k_new"], tt["v_new"], tt["k_blocks"], tt["v_blocks"],
                                   tt["block_table"], tt["lengths"], tt["cu_q"], max_q_len=max_q, **kw)
    elif max_q:
        def run(tt=t):
            gqa.decode_multi(tt["q"], tt["k_new"], tt["v_new"], tt["k_cache"], tt["v_cache"], tt["lengths"],
                             tt["cu_q"], tt.get("slot_ids"), max_q_len=max_q, **kw)
    elif attend and w.paged:
        def run(tt=t):
            gqa.attend_paged(tt["q"], tt["k_blocks"], tt["v_blocks"], tt["block_table"], tt["lengths"], **kw)
    elif attend:
        def run(tt=t):
            gqa.attend(tt["q"], tt["k_cache"], tt["v_cache"], tt["lengths"], tt.get("slot_ids"), **kw)
    elif w.paged:
        def run(tt=t):
            gqa.decode_step_paged(tt["q"], tt["k_new"], tt["v_new"], tt["k_blocks"], tt["v_blocks"],
                                  tt["block_table"], tt["lengths"], **kw)
    else:
        def run(tt=t):
            gqa.decode_step(tt["q"], tt["k_new"], tt["v_new"], tt["k_cache"], tt["v_cache"],
                            tt["lengths"], tt.get("slot_ids"), **kw)
    return run


# ---------------------------------------------------------------- clocks ---

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index, log_dir=None, tag=""):
        self.dev = device_index
        self.proc = None
        # the raw samples stay on disk for inspection (--clocks-dir)
        import tempfile
        self.path = os.path.join(log_dir or tempfile.gettempdir(), f"clocks_rank{device_index}{tag}.csv")

    def start(self):
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            sel = ["-i", "GPU-" + uuid if not uuid.startswith("GPU-") else uuid]
        except Exception:
            sel = []
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50", *sel],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons)}


# ---------------------------------------------------------------- oracle ---

def sample_rows(w, t, budget_bytes, kv_es, attend, multi, offset=0):
    """A bounded sample of batch rows for the CPU oracle: rows taken in order
    (starting at `offset`, wrapping) until their cached KV bytes reach
    `budget_bytes` (at least one row)."""
    L = t["lengths"].to("cpu").tolist()
    rows, total = [], 0
    for k in range(w.B):
        b = (offset + k) % w.B
        rows.append(b)
        total += max(int(L[b]), 0) * w.Hkv * w.D * 2 * kv_es
        if total >= budget_bytes:
            break
    return sorted(rows)


def oracle_problem(w, t, rows, mods=None):
    """Host copies of what the oracle needs for batch rows `rows`: the rows'
    cache rows (dense / slot-id caches) or the blocks their tables name (paged,
    renumbered), their queries and new tokens (packed tokens of a multi-token
    step, with new offsets). Returns (callable running the oracle without
    append, cached KV bytes it reads)."""
    import numpy as np
    import torch
    import oracle
    dev = t["q"].device
    sel = torch.tensor(rows, dtype=torch.long, device=dev)

    def host(x):
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16).copy()
        if x.dtype == torch.uint8:
            return x.numpy().copy()
        return x.numpy().copy()

    attend = "k_new" not in t
    multi = "cu_q" in t
    om = {}
    if mods:
        om = {"window": mods.get("window", 0), "kept_prefix": mods.get("kept_prefix", 0)}
        if mods.get("sink") is not None:
            om["sink"] = mods["sink"].cpu().numpy()
    if "k_scale" in t:
        om["k_scale"] = t["k_scale"].cpu().numpy()
        om["v_scale"] = t["v_scale"].cpu().numpy()
    L = host(t["lengths"][sel])
    if multi:
        cu = t["cu_q"].cpu().tolist()
        tok = [i for b in rows for i in range(cu[b], cu[b + 1])]
        tsel = torch.tensor(tok, dtype=torch.long, device=dev)
        qlen = [cu[b + 1] - cu[b] for b in rows]
        cu_s = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
        q, kn, vn = host(t["q"][tsel]), host(t["k_new"][tsel]), host(t["v_new"][tsel])
    else:
        q = host(t["q"][sel])
        if not attend:
            kn, vn = host(t["k_new"][sel]), host(t["v_new"][sel])
    if w.paged:
        bt = t["block_table"][sel].cpu().numpy()
        used = sorted(set(int(x) for x in bt[bt >= 0].tolist()))
        remap = {b: i for i, b in enumerate(used)}
        idx = torch.tensor(used, dtype=torch.long, device=dev)
        kb, vb = host(t["k_blocks"][idx]), host(t["v_blocks"][idx])
        btr = np.vectorize(lambda x: remap.get(int(x), -1))(bt).astype(np.int32)
        if multi:
            run = lambda: oracle.decode_multi_paged(q, kn, vn, kb, vb, btr, L, cu_s, append=False, **om)
        elif attend:
            run = lambda: oracle.attend_paged(q, kb, vb, btr, L, **om)
        else:
            run = lambda: oracle.decode_paged(q, kn, vn, kb, vb, btr, L, append=False, **om)
    else:
        cr = t["slot_ids"][sel].long() if "slot_ids" in t else sel
        kc, vc = host(t["k_cache"][cr]), host(t["v_cache"][cr])
        if multi:
            run = lambda: oracle.decode_multi_dense(q, kn, vn, kc, vc, L, cu_s, append=False, **om)
        elif attend:
            run = lambda: oracle.attend_dense(q, kc, vc, L, **om)
        else:
            run = lambda: oracle.decode_dense(q, kn, vn, kc, vc, L, append=False, **om)
    win, kp = (mods or {}).get("window", 0), (mods or {}).get("kept_prefix", 0)
    n = cached_slots_read(torch.from_numpy(np.asarray(L, dtype=np.int64)), attend, win, kp)
    kv_es = 1 if "k_scale" in t else w.elem_bytes
    kv = int(n.sum().item()) * w.Hkv * w.D * 2 * kv_es
    return run, kv


def oracle_rate(w, t, rows, repeats=3, mods=None):
    """CPU oracle over batch rows `rows` (host copies), timed: returns
    (GB/s of KV processed, seconds per pass, threads)."""
    run, kv = oracle_problem(w, t, rows, mods)
    r = run()                                   # warm-up
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        r = run()
        times.append(time.perf_counter() - t0)
    sec = statistics.median(times)
    return kv / sec / 1e9, sec, r.threads


def make_mods(args, w, dev):
    """The softmax modifiers asked for on the command line (None: none)."""
    import torch
    if not args.window and not args.kept_prefix and not args.sink:
        return None
    m = {"window": args.window, "kept_prefix": args.kept_prefix}
    if args.sink:
        g = torch.Generator().manual_seed(1234)
        m["sink"] = torch.randn(w.Hq, generator=g).to(dev)
    return m


def mods_config(args):
    return {"window": args.window, "kept_prefix": args.kept_prefix, "sink": bool(args.sink),
            "q_len": args.q_len or 1, "kv": args.kv}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBPS, "fallback"


def sources_sha(names):
    """Digest of the kernel sources a profile was taken on."""
    import hashlib
    h = hashlib.sha256()
    for n in names:
        h.update(open(os.path.join(ROOT, "gqa_kv_cache_gb300", "csrc", n), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel_name, key, alg_total):
    """Per-launch DRAM bytes (read + write) of the kernel on this workload and
    operation from the committed ncu summary, if it was taken on the current
    sources of that kernel; else None. A capture of the full launch gives its
    bytes; a capture of a scaled-down instance (fewer rows, the same length
    law) gives its bytes over its own algorithmic bytes, which scales to this
    launch by the slots it processes (`alg_total`)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))[kernel_name][key]
        if sources_sha(d["sources"]) != d["sources_sha"]:
            return None
        if "bytes_per_launch" in d:
            return d["bytes_per_launch"]
        return int(round(d["bytes_over_algorithmic"] * alg_total))
    except Exception:
        return None


def traffic_key(wname, attend, fp8, q_len, mods):
    key = wname + ("/attend" if attend else "") + ("/e4m3" if fp8 else "") + (f"/q{q_len}" if q_len else "")
    if mods:
        key += "/mods"
    return key


def supported(wname, args):
    """Whether the workload takes the options asked for (an E4M3 cache needs
    the tensor-core kernel's D = 128)."""
    import workloads as W
    w = W.WORKLOADS[wname]
    if args.kv == "e4m3" and (w.D != 128 or w.dtype != "bf16" or args.kernel == "simt"):
        return False
    return True


# ------------------------------------------------------------------ arms ---

def run_reference(args, ranks):
    """The reference arm: the float64 CPU oracle (plain loops, as it stands),
    on a bounded sample of the same workload, on this machine's host cores."""
    if ranks.rank != 0:
        return
    import torch
    wname = HEADLINE if args.workload == "all" else args.workload
    w = workload(wname, 0, args.shrink)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    import workloads as W
    attend = args.op == "attend"
    multi = args.q_len > 0
    fp8 = args.kv == "e4m3"
    t = W.generate(w, dev, attend=attend, q_f32=attend and args.q_dtype != "cache",
                   q_lens=[args.q_len] * w.B if multi else None, kv_e4m3=fp8)
    mods = make_mods(args, w, dev)
    kv_es = 1 if fp8 else w.elem_bytes
    rows0 = sample_rows(w, t, REF_SAMPLE_KV_BYTES, kv_es, attend, multi)
    n = len(rows0)
    for i in range(args.warmup):
        oracle_rate(w, t, sample_rows(w, t, REF_SAMPLE_KV_BYTES, kv_es, attend, multi, i * n), repeats=1,
                    mods=mods)
    threads = 1
    kv_total, t_total = 0, 0.0
    for i in range(args.steps):
        rows = sample_rows(w, t, REF_SAMPLE_KV_BYTES, kv_es, attend, multi, (i + args.warmup) * n)
        gbs, sec, threads = oracle_rate(w, t, rows, repeats=1, mods=mods)
        kv_total += gbs * sec * 1e9
        t_total += sec
    value = kv_total / t_total / 1e9
    metric = METRIC_MULTI if multi else (METRIC_ATTEND if attend else METRIC)
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "op": args.op, "B": w.B, "Hq": w.Hq,
                                        "Hkv": w.Hkv, "D": w.D, "sample_rows_per_step": n,
                                        **mods_config(args)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"about {REF_SAMPLE_KV_BYTES >> 20} MB of cached KV per step "
                                   f"({n} of {w.B} batch rows, rotating), float64 loops"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def measure(args, ranks, wname, dev):
    """Times one workload: the step (device time, L2 flushed between steps),
    the decode kernel alone, the end-to-end step through the public API and
    the CPU oracle on a bounded sample. Returns the workload's record."""
    import torch
    import workloads as W
    import gqa_kv_cache_gb300 as gqa

    w = workload(wname, ranks.rank, args.shrink)
    attend = args.op == "attend"
    multi = args.q_len > 0
    fp8 = args.kv == "e4m3"
    t = W.generate(w, dev, attend=attend, q_f32=attend and args.q_dtype != "cache",
                   q_lens=[args.q_len] * w.B if multi else None, kv_e4m3=fp8)
    torch.cuda.synchronize()
    out = torch.empty(t["q"].shape[0], w.Hq, w.D, dtype=torch.float32, device=dev)
    mods = make_mods(args, w, dev)
    call_mods = dict(mods or {})
    if fp8:
        call_mods.update(k_scale=t["k_scale"], v_scale=t["v_scale"])
    step = step_fn(w, t, args.kernel, out, args.sched_pad, attend, call_mods, args.q_len)
    kv_es = 1 if fp8 else None
    alg = algorithmic_bytes_multi(w, t, kv_es) if multi else algorithmic_bytes(w, t, attend, args.window,
                                                                               args.kept_prefix, kv_es)
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def l2_flush(i):
        """Evict the step's data from L2 outside the timed events. Writing a
        buffer larger than L2 leaves L2 full of dirty lines whose write-back
        would land inside the next timed step; reading a second buffer after
        it pushes those write-backs out here and leaves L2 clean and cold."""
        if args.l2_flush == "none":
            return
        flush_w.fill_(i & 0xFF)
        if args.l2_flush == "write_read":
            torch.sum(flush_r, dim=0, out=flush_sink)

    stream = torch.cuda.current_stream()

    for i in range(args.warmup):
        l2_flush(i)
        step()
    torch.cuda.synchronize()

    # ---- timed region: K steps, L2 flushed between them (outside the events)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(ranks.local, args.clocks_dir, "_" + wname)
    clocks.start()
    ranks.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(K):
        l2_flush(i)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ranks.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = ranks.max(sum(step_ms))
    ms_per_step = total_ms / K
    kv_all = ranks.sum(alg["kv_read"])
    value = kv_all * K / (total_ms * 1e-3) / 1e9

    # ---- the decode kernel alone (trace: CUDA events around each launch)
    gqa.trace_enable(True)
    gqa.trace_collect()
    Kr = min(K, 500)
    for i in range(Kr):
        l2_flush(i)
        step()
    torch.cuda.synchronize()
    tr = gqa.trace_collect()
    gqa.trace_enable(False)
    main = max(tr, key=lambda k: tr[k][0])
    n_main, ms_main = tr[main]
    avg_main_s = ms_main / max(n_main, 1) * 1e-3
    hbm_peak, peak_kind = peaks()
    achieved = alg["total"] / avg_main_s / 1e9
    tkey = traffic_key(w.name, attend, fp8, args.q_len, mods)
    traffic = traffic_for(main, tkey, alg["total"]) if args.kernel == "auto" else None

    # ---- end to end through the public API, host buffers, copies inside
    Ke = min(K, 500)
    inputs = ["q", "lengths"] + ([] if attend else ["k_new", "v_new"]) + (["cu_q"] if multi else []) + \
        (["slot_ids"] if "slot_ids" in t else []) + \
        (["block_table"] if "block_table" in t else [])
    # the step's inputs travel in one pinned staging buffer, each at a 256-byte
    # aligned offset, so a step makes one host-to-device copy; the device
    # tensors the API gets are views of one device buffer
    offs, total = {}, 0
    for k in inputs:
        offs[k] = total
        total += (t[k].numel() * t[k].element_size() + 255) // 256 * 256
    host_buf = torch.zeros(total, dtype=torch.uint8, pin_memory=True)
    dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)
    dev_in = {}
    for k in inputs:
        nb = t[k].numel() * t[k].element_size()
        host_buf[offs[k]:offs[k] + nb].copy_(t[k].contiguous().view(torch.uint8).reshape(-1).cpu())
        dev_in[k] = dev_buf[offs[k]:offs[k] + nb].view(t[k].dtype).view(t[k].shape)
    tt = dict(t)
    tt.update(dev_in)
    step_e2e = step_fn(w, tt, args.kernel, out, args.sched_pad, attend, call_mods, args.q_len)
    out_host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = total
    d2h = out.numel() * out.element_size()
    e2e_ms = 0.0
    for i in range(Ke + 3):
        l2_flush(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dev_buf.copy_(host_buf, non_blocking=True)
        step_e2e()
        out_host.copy_(out, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= 3:
            e2e_ms += a.elapsed_time(b)
    e2e_ms = ranks.max(e2e_ms)
    e2e_value = kv_all * Ke / (e2e_ms * 1e-3) / 1e9

    # ---- CPU baseline: the oracle on host cores (bounded sample), rank 0 at N = 1 only
    cpu = None
    if ranks.world == 1 and not args.no_cpu_baseline:
        rows = sample_rows(w, t, CPU_SAMPLE_KV_BYTES, 1 if fp8 else w.elem_bytes, attend, multi)
        gbs, sec, threads = oracle_rate(w, t, rows, repeats=3, mods=mods)
        cpu = {"value": gbs, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{len(rows)} of {w.B} batch rows of one step (about "
                         f"{CPU_SAMPLE_KV_BYTES >> 20} MB of cached KV or all rows; no append), "
                         f"float64 loops, median of 3 after 1 warm-up, {sec:.3f} s per pass"}

    rec = {
        "metric": METRIC_MULTI if multi else (METRIC_ATTEND if attend else METRIC),
        "value": value, "unit": UNIT, "ms_per_step": ms_per_step, "us_per_step": ms_per_step * 1e3,
        "dtype": w.dtype,
        "frac_of_8TBps": value / ranks.world / NOMINAL_HBM_GBPS,
        "frac_of_measured_hbm": value / ranks.world / hbm_peak,
        "config": {"workload": w.name, "op": args.op, "q_dtype": str(t["q"].dtype).replace("torch.", ""),
                   "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "G": w.G, "D": w.D,
                   "Smax": w.Smax, "paged": w.paged, "kernel": main, "kernel_option": args.kernel,
                   "kv_bytes_per_step_per_gpu": alg["kv_read"],
                   "l2": {"write_read": "flushed between timed steps (256 MB write, then 256 MB read: "
                                        "L2 cold and clean; outside the events)",
                          "write": "flushed between timed steps (256 MB write outside the events)",
                          "none": "not flushed; inputs larger than L2"}[args.l2_flush],
                   "parallelism": f"replicas x{ranks.world} (independent batches per GPU)",
                   **mods_config(args),
                   "wall_s_timed_region": wall},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "traffic_key": tkey,
                     "peak_kind": peak_kind + " (STREAM-style copy)",
                     "kernel": main, "avg_launch_us": avg_main_s * 1e6,
                     "algorithmic_bytes_per_launch": alg["total"]},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "us_per_step": e2e_ms / Ke * 1e3},
        "gpu_launches": K,   # one decode kernel per step (the split merge is fused)
        "clocks": clk,
    }
    del t, out, flush_w, flush_r, host_buf, dev_buf, dev_in, tt
    torch.cuda.empty_cache()
    return rec


def run_ours(args, ranks):
    import torch

    torch.cuda.set_device(ranks.local)
    dev = torch.device("cuda", ranks.local)
    if args.q_len > 0 and (args.op == "attend" or args.window or args.kept_prefix):
        raise SystemExit("--q-len times the plain multi-token step (no --op attend / window)")
    names = SUITE if args.workload == "all" else [args.workload]
    head = HEADLINE if args.workload == "all" else args.workload
    if not supported(head, args):
        raise SystemExit(f"{head} does not take these options")
    per = {}
    for name in names:
        if not supported(name, args):
            per[name] = {"skipped": "an E4M3 cache needs the tensor-core kernel (bfloat16 data, D = 128)"}
            continue
        per[name] = measure(args, ranks, name, dev)
    h = per[head]
    line = {
        "metric": h["metric"], "value": h["value"], "unit": UNIT,
        "n_gpus": ranks.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": h["ms_per_step"], "us_per_step": h["us_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": h["dtype"],
        "data": "synthetic",
        "frac_of_8TBps": h["frac_of_8TBps"], "frac_of_measured_hbm": h["frac_of_measured_hbm"],
        "config": dict(h["config"], headline=("largest workload by KV bytes per step"
                                              if args.workload == "all" else "the workload asked for")),
        "roofline": h["roofline"],
        "cpu_baseline": h["cpu_baseline"],
        "e2e": h["e2e"],
        "gpu_launches": h["gpu_launches"],
        "clocks": h["clocks"],
    }
    if len(names) > 1:
        keys = ("value", "us_per_step", "frac_of_8TBps", "frac_of_measured_hbm", "roofline",
                "cpu_baseline", "e2e", "gpu_launches", "clocks", "dtype")
        line["per_config"] = {n: (r if "skipped" in r else
                                  dict({k: r[k] for k in keys}, kernel=r["config"]["kernel"],
                                       kv_bytes_per_step=r["config"]["kv_bytes_per_step_per_gpu"]))
                              for n, r in per.items()}
    if ranks.rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    ranks = Ranks()
    if args.impl == "reference":
        # no GPU collective is needed: rank 0 alone runs the oracle
        run_reference(args, ranks)
        return
    import torch
    ranks.init("nccl" if torch.cuda.is_available() else "gloo")
    try:
        run_ours(args, ranks)
    finally:
        ranks.close()


if __name__ == "__main__":
    main()
