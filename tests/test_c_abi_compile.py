"""The boundary is a plain C ABI: include/mla.h compiles as C99 with every
warning an error, a C program takes the address of every declared entry
point, links against libmla.so and runs the host-only calls (no GPU
needed).  Nothing here uses torch."""

import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")
LIBDIR = os.path.join(ROOT, "head_latent_attention_28_b300")

pytestmark = pytest.mark.skipif(shutil.which("gcc") is None, reason="needs a C compiler")


def declared():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(mla_\w+)\s*\(", text)))


def test_header_is_c99_and_host_calls_run(tmp_path):
    names = declared()
    src = tmp_path / "abi.c"
    src.write_text("""
#include <stdio.h>
#include <string.h>
#include "mla.h"

typedef void (*entry_point)(void);
static const entry_point entry_points[] = {
%s
};

int main(void) {
  int32_t lens[3] = {64, 1000, 129}, first[3], last[3];
  int64_t pages = 0;
  int ok = 1;
  ok &= mla_version() >= 100;
  ok &= strlen(mla_status_string(MLA_ERR_WORKSPACE)) > 0;
  ok &= mla_prefill_kv_rows(3) == 256;
  ok &= mla_decode_item_cost(1, 128, 512, 64, MLA_BF16) == 5;
  ok &= mla_decode_row_groups(2, 128, 512, 64, MLA_BF16) == 2;
  ok &= mla_decode_path(1, 128, 512, 64, MLA_BF16) == 1;
  ok &= mla_decode_split_plan(lens, 3, 1, 16, 4, 0, first, last, &pages) == MLA_OK;
  ok &= pages == 1 + 16 + 3;
  ok &= first[0] == 0 && last[2] == 3;
  /* host-side argument checks return before any device is touched */
  ok &= mla_decode_paged(NULL, NULL, MLA_BF16, NULL, NULL, 1, 1, 128, 512, 64, MLA_PAGE_SIZE,
                         1, 1, 0.1f, 0, NULL, 0, NULL, NULL, NULL) == MLA_ERR_INVALID_ARG;
  printf("%%s %%d\\n", ok ? "ok" : "FAILED", (int)(sizeof entry_points / sizeof entry_points[0]));
  return ok ? 0 : 1;
}
""" % ",\n".join(f"  (entry_point)&{n}" for n in names))
    exe = tmp_path / "abi"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic-errors",
           "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
           "-L", LIBDIR, "-lmla", "-Wl,-rpath," + LIBDIR]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.split() == ["ok", str(len(names))], r.stdout + r.stderr
