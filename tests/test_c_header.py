"""The boundary from C: include/ditattn.h compiles as strict C11.

A generated C program takes the address of every function the header
declares, so the link fails if libditattn.so is missing any of them. It then
calls the status strings and a zero-sized attention, which returns before
anything touches the GPU. No GPU is needed."""

import re
import shutil
import subprocess

import pytest

from diffusion_transformer_attention_dit_gb300 import build

from test_abi import HEADER, ROOT

pytestmark = pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")


def _functions():
    text = HEADER.read_text()
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(dit_\w+)\s*\(", text, flags=re.M)))


PROGRAM = r"""
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "ditattn.h"

static void (*const every_function[])(void) = {
%s
};

int main(void) {
  int64_t st[3] = {0, 0, 0};
  dit_status s;
  if (sizeof(every_function) / sizeof(every_function[0]) != %d) return 2;
  if (strlen(dit_status_string(DIT_OK)) == 0 || strlen(dit_status_string(DIT_ERR_INVALID_ARG)) == 0) return 3;
  /* zero-sized work: DIT_OK without a launch (null buffers are never read) */
  s = dit_attn_fwd(NULL, NULL, NULL, 0, 1, 1, 1, 128, st, st, 0.125f, 0, 1, NULL, DIT_BF16, st, NULL, NULL);
  if (s != DIT_OK) return 4;
  /* a bad head dimension is refused before anything else */
  s = dit_attn_fwd(NULL, NULL, NULL, 1, 1, 1, 1, 96, st, st, 0.125f, 0, 1, NULL, DIT_BF16, st, NULL, NULL);
  if (s == DIT_OK) return 5;
  printf("ok %%s\n", dit_status_string(s));
  return 0;
}
"""


def test_header_compiles_as_c11_and_links_every_function(tmp_path):
    lib = build.build()
    names = _functions()
    assert "dit_attn_fwd" in names and "dit_status_string" in names
    entries = ",\n".join(f"  (void (*)(void)){n}" for n in names)  # any function pointer type converts
    src = tmp_path / "abi_from_c.c"
    src.write_text(PROGRAM % (entries, len(names)))
    exe = tmp_path / "abi_from_c"
    cc = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror",
                         "-I", str(ROOT / "include"), str(src), "-o", str(exe), str(lib),
                         f"-Wl,-rpath,{lib.parent}"], capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0 and run.stdout.startswith("ok "), (run.returncode, run.stdout, run.stderr)
