"""The public header as a C caller sees it (CPU; no GPU call is made).

A C99 program that includes ``include/kd_topk_kl.h`` is compiled with
warnings as errors and linked against ``libkdtopk.so``; it calls the entry
points that need no device (version, build id, status strings, workspace
sizes) and one loss entry point with a NULL input, which must be refused
on the host before anything is launched.  Its answers must equal the ones
the Python binding gets through ctypes.
"""
import os
import shutil
import subprocess

import pytest

import chunked_top_kl_gemm_b300 as kd
from chunked_top_kl_gemm_b300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "chunked_top_kl_gemm_b300")

C_SOURCE = r"""
#include <stdio.h>
#include <string.h>
#include "kd_topk_kl.h"

int main(void) {
  float loss = 0.f;
  kd_status st;
  printf("abi %d\n", kd_abi_version());
  printf("build %s\n", kd_build_id());
  printf("ws %zu\n", kd_topk_kl_workspace_size(32768, 2880, 201088, 100, 2048));
  printf("ws_flags %zu\n", kd_topk_kl_workspace_size_flags(32768, 2880, 201088, 100, 2048,
                                                           KD_FLAG_STORE_LOGITS));
  printf("ws_bad %zu\n", kd_topk_kl_workspace_size(0, 2880, 201088, 100, 2048));
  st = kd_topk_kl_fwd_bwd(NULL, NULL, NULL, NULL, 16, 64, 128, 4, 1.0f, 64, &loss, NULL, NULL);
  printf("null %d %s\n", (int)st, kd_status_string(st));
  printf("ok %s\n", kd_status_string(KD_OK));
  return 0;
}
"""


@pytest.fixture(scope="module")
def c_program(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    _build.build()                        # (re)built from the tree's sources if stale
    kd.lib()
    d = tmp_path_factory.mktemp("c_abi")
    src = d / "caller.c"
    src.write_text(C_SOURCE)
    exe = d / "caller"
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), "-L", PKG, "-lkdtopk", f"-Wl,-rpath,{PKG}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_header_compiles_as_c_and_the_library_links(c_program):
    r = subprocess.run([str(c_program)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    out = dict(line.split(" ", 1) for line in r.stdout.strip().splitlines())
    assert int(out["abi"]) == kd.abi_version()
    assert out["build"] == kd.build_id()
    assert int(out["ws"]) == kd.kd_topk_kl_workspace_size(32768, 2880, 201088, 100, 2048)
    assert int(out["ws_flags"]) == kd.kd_topk_kl_workspace_size_flags(
        32768, 2880, 201088, 100, 2048, kd.KD_FLAG_STORE_LOGITS)
    assert int(out["ws_bad"]) == 0
    code, text = out["null"].split(" ", 1)
    assert int(code) == 1 and text == kd.kd_status_string(1)      # KD_ERR_INVALID_ARG
    assert out["ok"] == kd.kd_status_string(0)
