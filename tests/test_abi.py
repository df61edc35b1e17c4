"""The C-ABI library loads and exports every entry point include/qlin.h declares (CPU only)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "qlin.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qlin_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_match_binding(qlin):
    assert _declared() == sorted(qlin.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(qlin):
    L = ctypes.CDLL(qlin.LIB_PATH)
    for name in _declared():
        assert hasattr(L, name), name
    nm = subprocess.run(["nm", "-D", "--defined-only", qlin.LIB_PATH], capture_output=True, text=True)
    if nm.returncode == 0:
        exported = set(line.split()[-1] for line in nm.stdout.splitlines() if line.strip())
        for name in _declared():
            assert name in exported, name


def test_status_strings(qlin):
    assert qlin.status_string(0) == "ok"
    assert "timed out" in qlin.status_string(qlin.QLIN_ERR_TIMEOUT)
    assert qlin.status_string(99) == "unknown status"


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "qlin.h"\nint main(void){ qlin_layer_info i; (void)i; return QLIN_OK; }\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-c", str(src),
                        "-o", str(tmp_path / "t.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
