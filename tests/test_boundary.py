"""The C-ABI boundary without a GPU: libdkv builds for sm_103a, loads, exports
every entry point include/dkv.h declares, and the binding's ctypes structs
match the header's layout (checked by compiling the header with gcc)."""
import os
import re
import subprocess

import pytest

import differentiated_kv_cache_gb300 as dkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dkv.h")


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(dkv_\w+)\s*\(", src, re.M)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(dkv.EXPORTED)


def test_library_builds_and_exports_every_symbol():
    path = dkv.build.build()
    lib = dkv.load()
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    for name in declared_functions():
        assert re.search(rf"\bT {name}$", out, re.M), name
    assert dkv.dkv_strerror(dkv.DKV_ERR_NO_PAGES) == "free page list exhausted"


def test_struct_layouts_match_header(tmp_path):
    import ctypes as C
    prog = tmp_path / "layout.c"
    fields = {
        "dkv_config": [f for f, _ in dkv.dkv_config._fields_],
        "dkv_geometry": [f for f, _ in dkv.dkv_geometry._fields_],
        "dkv_status": [f for f, _ in dkv.dkv_status._fields_],
        "dkv_snapshot": [f for f, _ in dkv.dkv_snapshot._fields_],
    }
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "dkv.h"', "int main(void){"]
    for st, fs in fields.items():
        lines.append(f'printf("{st} %zu\\n", sizeof({st}));')
        for f in fs:
            lines.append(f'printf("{st}.{f} %zu\\n", offsetof({st}, {f}));')
    lines.append("return 0;}")
    prog.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)], check=True)
    got = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True, text=True).stdout.splitlines())
    for st, fs in fields.items():
        cls = getattr(dkv, st)
        assert int(got[st]) == C.sizeof(cls), st
        for f in fs:
            assert int(got[f"{st}.{f}"]) == getattr(cls, f).offset, (st, f)


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "differentiated_kv_cache_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"\boracle\b", text.replace("the oracle", "")), fn


def test_create_without_gpu_fails_cleanly():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    cfg = dkv.make_config(n_layers=1, n_kv_heads=2, group_size=4, n_pages=16, max_requests=2, max_seq_len=64)
    with pytest.raises(dkv.DkvError):
        dkv.dkv_pool_create(cfg, 0)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built library the binding raises; nothing falls back."""
    monkeypatch.setattr(dkv.build, "LIB", str(tmp_path / "absent" / "libdkv.so"))
    monkeypatch.setattr(dkv.dkv, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        dkv.load()
    with pytest.raises(RuntimeError, match="not built"):
        dkv.dkv_pool_create(dkv.make_config(n_layers=1, n_kv_heads=2, group_size=4, n_pages=16, max_requests=2,
                                            max_seq_len=64), 0)
