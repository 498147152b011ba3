"""The C ABI from C: a C99 program that includes only include/gpt2gb.h,
links libgpt2gb.so, and calls the entry points that need no GPU (version,
status strings, size queries, argument checks).  This checks that the header
is plain C (no C++ or CUDA headers needed) and that the library resolves
every symbol such a program uses."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include "gpt2gb.h"

int main(void) {
  gpt2_dims d = {12, 768, 12, 3072, 50257, 1024, 1e-5f, GPT2_BF16, 0u};
  gpt2_dims bad = d;
  gpt2_block_weights w = {0};
  gpt2_block_grads g = {0};
  int site = -1;
  bad.n_head = 10;  /* head_dim 76.8: unsupported */
  printf("abi %d\n", gpt2_abi_version());
  printf("status3 %s\n", gpt2_status_string(GPT2_ERR_WORKSPACE));
  printf("ws %zu\n", gpt2_workspace_bytes(&d, 8, 1024));
  printf("ws_bad %zu\n", gpt2_workspace_bytes(&bad, 8, 1024));
  printf("kv %zu\n", gpt2_kv_cache_bytes(&d, 64, 1087));
  printf("mlp_scratch %zu\n", gpt2_mlp_noalloc_max_scratch_bytes());
  printf("ln_bad %d\n", gpt2_layernorm(0, 0, 0, 0, 10, 770, 1e-5f, GPT2_F32, GPT2_F32, 0));
  printf("block_null %d\n", gpt2_block_forward(&d, &w, 0, 0, 2, 64, 0, 0, 0));
  printf("bwd_bf16 %d\n", gpt2_block_backward(&d, &w, 0, 0, 0, 0, &g, 2, 64, 0, 0, 0));
  d.flags = 4u;
  printf("flags_bad %zu\n", gpt2_workspace_bytes(&d, 8, 1024));
  (void)site;
  return 0;
}
"""


def test_c_program_uses_the_abi(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from gpt_pre_ln_gb300 import build
    lib = build.build()
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(lib)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                        str(exe), "-L", libdir, "-lgpt2gb", f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    out = dict(line.split(" ", 1) for line in r.stdout.strip().splitlines())
    assert out["abi"] == "4"
    assert out["status3"] == "workspace too small"
    M = 8 * 1024
    assert int(out["ws"]) == 2 * M * 768 * 4 + 2 * M * 768 * 2 + M * 3 * 768 * 2 + M * 3072 * 2
    assert int(out["ws_bad"]) == 0 and int(out["flags_bad"]) == 0
    assert int(out["kv"]) == 12 * 2 * 64 * 12 * 1087 * 64 * 2
    assert int(out["mlp_scratch"]) == 16 << 20
    assert out["ln_bad"] == "2"       # D not a multiple of 4
    assert out["block_null"] == "1"   # null weight pointers
    assert out["bwd_bf16"] == "1"     # null weights come first; (F32-only is checked after the pointers)
