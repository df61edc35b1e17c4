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


_C_PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include "qlin.h"

int main(void) {
  const int N = 70, K = 256, G = K / 128;
  float* W = (float*)malloc(sizeof(float) * N * K);
  unsigned s = 12345u;
  for (int i = 0; i < N * K; ++i) {
    s = s * 1103515245u + 12345u;
    W[i] = (float)((int)((s >> 8) % 2001u) - 1000) * 2e-5f;
  }
  qlin_handle h = NULL;
  if (qlin_pack_w4g128(W, N, K, &h) != QLIN_OK || !h) return 1;
  qlin_layer_info info;
  if (qlin_info(h, &info) != QLIN_OK || info.format != QLIN_FMT_W4G128 || info.N != N || info.K != K ||
      info.packed_bytes != (int64_t)N * K / 2 + (int64_t)N * G * 4)
    return 2;
  qlin_canonical c;
  if (qlin_export(h, &c) != QLIN_OK || !c.codes || !c.scale || !c.zero || c.perm || c.codes3 || c.qw) return 3;
  qlin_handle h2 = NULL;
  if (qlin_import(QLIN_FMT_W4G128, N, K, &c, &h2) != QLIN_OK || !h2) return 4;
  qlin_canonical c2;
  if (qlin_export(h2, &c2) != QLIN_OK) return 5;
  if (memcmp(c.codes, c2.codes, (size_t)N * K / 2) || memcmp(c.scale, c2.scale, (size_t)N * G * 2) ||
      memcmp(c.zero, c2.zero, (size_t)N * G * 2))
    return 6;
  size_t wb = 0, ws = 0;
  if (qlin_device_bytes(h2, &wb) != QLIN_OK || wb == 0) return 7;
  if (qlin_workspace_bytes(h2, 16, &ws) != QLIN_OK || ws == 0) return 8;
  /* errors are reported as status codes, never by crashing */
  qlin_handle bad = NULL;
  if (qlin_pack_w4g128(W, N, 200, &bad) != QLIN_ERR_INVALID_ARG || bad) return 9;
  if (qlin_forward(h, NULL, NULL, 1, NULL) != QLIN_ERR_INVALID_ARG) return 10;
  if (qlin_forward(h, (void*)0x1000, (void*)0x2000, 0, NULL) != QLIN_OK) return 11;
  if (qlin_forward(h, (void*)0x1000, (void*)0x2000, 1, NULL) != QLIN_ERR_NOT_BOUND) return 12;
  if (qlin_import(7, N, K, &c, &bad) != QLIN_ERR_INVALID_ARG || bad) return 13;
  if (strcmp(qlin_status_string(QLIN_OK), "ok") != 0) return 14;
  qlin_destroy(h2);
  qlin_destroy(h);
  free(W);
  printf("ok\n");
  return 0;
}
"""


def test_c_program_links_and_runs(tmp_path, qlin):
    """A C99 program built against include/qlin.h and linked to libqlin.so: host-side calls
    (pack, info, export, import, sizes, argument errors) behave as documented, no GPU needed."""
    src = tmp_path / "abi_host.c"
    src.write_text(_C_PROGRAM)
    libdir = os.path.dirname(qlin.LIB_PATH)
    exe = tmp_path / "abi_host"
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                        "-L", libdir, "-lqlin", "-Wl,-rpath," + libdir, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip() == "ok", (run.returncode, run.stdout, run.stderr)
