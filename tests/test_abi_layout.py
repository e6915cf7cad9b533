"""The Python binding and the C header describe the same ABI.

A small C program compiled against include/kvc.h reports the size and field
offsets of the descriptor structs; the ctypes structures must match them, and
every prototype's parameter count must equal the argtypes the binding
registers.  No GPU is needed (the program only evaluates sizeof/offsetof).
"""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

from agent_shared_context_gb300 import kvc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvc.h")

_FIELDS = {
    "kvc_cache_view": ["base", "s_req", "s_layer", "s_head", "s_tok"],
    "kvc_segments": ["R", "T", "L", "H", "d", "S", "max_seg_len", "dtype", "seg_request",
                     "seg_start", "seg_len"],
    "kvc_params": ["rank", "oversample", "power_iters", "n_anchors", "top_k", "energy_frac",
                   "temperature", "tau", "select_mode", "reuse_ratio", "summary_mode", "rank_c",
                   "omega_c"],
}


def _cuda_include():
    for base in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        inc = os.path.join(base, "include")
        if base and os.path.exists(os.path.join(inc, "cuda_runtime_api.h")):
            return inc
    return None


def test_struct_layouts_match_the_header(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    inc = _cuda_include()
    if cc is None or inc is None:
        pytest.skip("needs a C compiler and the CUDA headers")
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "kvc.h"', "int main(void) {"]
    for st, fields in _FIELDS.items():
        lines.append('  printf("%s size %%zu\\n", sizeof(%s));' % (st, st))
        for f in fields:
            lines.append('  printf("%s.%s %%zu\\n", offsetof(%s, %s));' % (st, f, st, f))
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), "-I", inc, str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = dict(line.rsplit(" ", 1) for line in out.strip().splitlines())
    for st, fields in _FIELDS.items():
        cls = getattr(kvc, st)
        assert [f[0] for f in cls._fields_] == fields, st
        assert int(got["%s size" % st]) == ctypes.sizeof(cls), st
        for f in fields:
            assert int(got["%s.%s" % (st, f)]) == getattr(cls, f).offset, (st, f)


def _prototypes():
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    protos = {}
    for m in re.finditer(r"\b(kvc_[a-z_]+)\s*\(([^;{]*?)\)\s*;", src):
        params = m.group(2).strip()
        protos[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return protos


def test_every_prototype_has_matching_argtypes():
    protos = _prototypes()
    assert set(protos) == set(kvc.EXPORTS)
    for name, n in protos.items():
        fn = getattr(kvc.lib, name)
        argtypes = fn.argtypes or []
        assert len(argtypes) == n, (name, len(argtypes), n)
