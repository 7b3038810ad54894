"""The C ABI library: it loads, exports every function include/*.h declares,
and its host-side argument checks answer without touching a GPU."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(gqa_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    from gqa_kv_cache_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        from gqa_kv_cache_gb300 import build as b
        b.build()
    return _lib.load()


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("gqa_decode_step", "gqa_decode_step_paged", "gqa_workspace_bytes", "gqa_validate",
              "gqa_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from gqa_kv_cache_gb300 import _lib
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = _declared_functions() - exported
    assert not missing, f"declared but not exported: {missing}"
    for n in _declared_functions():
        getattr(lib, n)          # resolvable through ctypes
        assert n in _lib.SIGNATURES, f"binding lacks a signature for {n}"


def test_status_strings(lib):
    for code in range(6):
        assert lib.gqa_status_string(code)
    assert b"workspace" in lib.gqa_status_string(4)


def test_version(lib):
    assert lib.gqa_version() >= 100


def test_kernel_names_and_choices(lib):
    """Every trace kind has its kernel's name, and the binding's kernel
    choices are the header's enum values."""
    names = [lib.gqa_kernel_name(k).decode() for k in range(4)]
    assert names == ["simt_decode_kernel", "tc_decode_kernel", "unit_decode_kernel", "tc5_multi_kernel"]
    assert lib.gqa_kernel_name(4) == b"unknown"
    import gqa_kv_cache_gb300 as gqa
    text = open(os.path.join(ROOT, "include", "gqa_decode.h")).read()
    enum = {m.group(1).lower(): int(m.group(2)) for m in re.finditer(r"GQA_KERNEL_(\w+) = (\d+)", text)}
    assert gqa.KERNELS == enum


def test_tcgen05_choice_sizes_the_workspace_like_tc(lib):
    """The opt-in tcgen05 form is the tensor-core kernel for every size
    question: the same workspace for the single- and multi-token steps."""
    from gqa_kv_cache_gb300 import _lib
    def opts(kernel):
        o = _lib.GqaOptions()
        o.kernel = kernel
        o.grid_ctas = 304          # no device query (no GPU here)
        return o
    tc, t5 = opts(2), opts(4)
    for B, Hq, Hkv in ((32, 32, 8), (4, 64, 8), (64, 48, 8)):
        a = lib.gqa_workspace_bytes_multi(B, Hq, Hkv, 128, 1, 8, ctypes.byref(tc))
        b = lib.gqa_workspace_bytes_multi(B, Hq, Hkv, 128, 1, 8, ctypes.byref(t5))
        assert a == b and a > 0


def _step(lib, **kw):
    a = dict(q=1, k_new=1, v_new=1, kc=1, vc=1, lengths=1, slot_ids=None, out=1,
             B=2, Hq=8, Hkv=2, D=64, R=2, Smax=16, dt=1, ws=None, ws_bytes=0, status=None)
    a.update(kw)
    P = lambda x: None if x is None else ctypes.c_void_p(x * 256)
    return lib.gqa_decode_step(P(a["q"]), P(a["k_new"]), P(a["v_new"]), P(a["kc"]), P(a["vc"]),
                               P(a["lengths"]), P(a["slot_ids"]), P(a["out"]), a["B"], a["Hq"],
                               a["Hkv"], a["D"], a["R"], a["Smax"], a["dt"], P(a["ws"]),
                               a["ws_bytes"], P(a["status"]), None)


def test_host_argument_checks(lib):
    """Host-visible errors return before any CUDA call (no GPU needed)."""
    assert _step(lib, B=0) == 0                        # empty batch: nothing to do
    assert _step(lib, Hq=6, Hkv=4) == 1                # Hq % Hkv != 0
    assert _step(lib, Hkv=0) == 1
    assert _step(lib, dt=7) == 1                       # unknown dtype
    assert _step(lib, q=None) == 1                     # null pointer
    assert _step(lib, R=1) == 1                        # fewer rows than batch, no slot_ids
    assert _step(lib, Smax=0) == 1
    assert _step(lib, D=96, dt=1) == 2                 # no kernel for D = 96
    assert _step(lib, Hq=32, Hkv=2) == 2               # G = 16 > 8


def test_paged_argument_checks(lib):
    P = lambda x: ctypes.c_void_p(x * 256)
    args = lambda **k: {**dict(B=1, Hq=4, Hkv=1, D=128, nb=4, bs=16, mb=2), **k}
    def call(**k):
        a = args(**k)
        return lib.gqa_decode_step_paged(P(1), P(1), P(1), P(1), P(1), P(1), P(1), P(1), a["B"],
                                         a["Hq"], a["Hkv"], a["D"], a["nb"], a["bs"], a["mb"], 1,
                                         None, 0, None, None)
    assert call(B=0) == 0
    assert call(nb=0) == 1
    assert call(bs=0) == 1
    assert call(mb=0) == 1


def test_workspace_bytes_rejects_bad_sizes(lib):
    assert lib.gqa_workspace_bytes(1, 6, 4, 64, 1, None) == 0
    assert lib.gqa_workspace_bytes(-1, 8, 2, 64, 1, None) == 0


def test_validate_argument_checks(lib):
    assert lib.gqa_validate(ctypes.c_void_p(256), None, None, 2, 1, 16, 0, 0, 0,
                            ctypes.c_void_p(256), None) == 1     # R < B without slot_ids
    assert lib.gqa_validate(ctypes.c_void_p(256), None, None, 2, 2, 16, 0, 0, 0,
                            None, None) == 1                     # no result buffer


def test_binding_raises_without_gpu_tensors():
    import torch
    import gqa_kv_cache_gb300 as gqa
    q = torch.zeros(1, 2, 8)
    with pytest.raises(ValueError):
        gqa.decode_step(q, q[:, :1], q[:, :1], q[None], q[None], torch.zeros(1, dtype=torch.int32))


def test_options_struct_layout_matches_the_header(tmp_path):
    """The binding's gqa_options has the header's size and field offsets."""
    from gqa_kv_cache_gb300 import _lib
    fields = [f[0] for f in _lib.GqaOptions._fields_ if f[0] != "reserved"]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "gqa_decode.h"\nint main(void) {\n'
                   '  printf("%zu\\n", sizeof(gqa_options));\n'
                   + "".join(f'  printf("%zu\\n", offsetof(gqa_options, {f}));\n' for f in fields)
                   + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)])
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert got[0] == ctypes.sizeof(_lib.GqaOptions)
    assert got[1:] == [getattr(_lib.GqaOptions, f).offset for f in fields]


def test_negative_wait_limit_is_refused(lib):
    """A negative consumer wait limit is an argument error, found before any launch."""
    from gqa_kv_cache_gb300 import _lib
    P = lambda x: ctypes.c_void_p(x * 256)
    o = _lib.GqaOptions()
    o.wait_limit_cycles = -1
    code = lib.gqa_decode_step_ex(P(1), P(1), P(1), P(1), P(1), P(1), None, P(1), 2, 8, 2, 128, 2, 16, 1,
                                  None, 0, None, None, ctypes.byref(o))
    assert code == 1
