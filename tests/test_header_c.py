"""include/pa.h is a C header: a C11 translation unit that calls every
declared entry point with arguments of the declared types compiles without
warnings (-Wall -Wextra -Werror), and, when the library is built, links
against it with every symbol resolved."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SOURCE = r"""
#include <stddef.h>
#include <stdint.h>
#include "pa.h"

int main(void) {
  pa_shape s = {0};
  s.mode = PA_MODE_DECODE; s.num_q_heads = 32; s.num_kv_heads = 8; s.head_dim = 128;
  s.page_size = 16; s.kv_dtype = PA_KV_BF16; s.max_batch = 4; s.max_pages_per_seq = 8;
  s.num_sms = 152;
  pa_plan_t plan;
  const int32_t lens[4] = {1, 2, 3, 4};
  pa_status st = pa_plan(&s, lens, 4, &plan);
  void* p = NULL;
  const int32_t* ip = NULL;
  const float* fp = NULL;
  float* lse = NULL;
  uint32_t code = 0;
  /* batch 0: every call returns before touching a pointer or the device */
  st = pa_decode(&plan, p, 0, 0, p, p, 0, 0, 0, 0, ip, 0, ip, 0, 1.f, fp, 1.f, 1.f, fp, fp,
                 p, 0, 0, lse, p, plan.scratch_bytes, p);
  st = pa_decode_static_scratch(&plan, p, 0, 0, p, p, 0, 0, 0, 0, ip, 0, ip, 0, 1.f, fp, 1.f, 1.f,
                                p, 0, 0, lse, p);
  st = pa_extend(&plan, p, 0, 0, p, p, 0, 0, 0, 0, ip, 0, ip, ip, 0, 0, 1.f, fp, 1.f, 1.f, fp, fp,
                 p, 0, 0, lse, p, plan.scratch_bytes, p);
  st = pa_append_kv(p, p, 0, 0, p, p, 0, 0, 0, 0, 16, 8, 128, PA_KV_BF16, (const int64_t*)0, 0,
                    1.f, 1.f, p, p);
  st = pa_debug_wait_expiry(p, 0, 0, p);   /* null scratch: refused on the host */
  (void)pa_scratch_init;
  (void)pa_check;
  (void)code;
  const char* msg = pa_status_string(st);
  return (msg != NULL && pa_version() > 0) ? 0 : 1;
}
"""


@pytest.fixture(scope="module")
def cc():
    c = shutil.which("gcc") or shutil.which("cc")
    if c is None:
        pytest.skip("no C compiler")
    return c


def test_header_compiles_as_c11(cc, tmp_path):
    src = tmp_path / "abi.c"
    src.write_text(SOURCE)
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                        "-I" + os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_links_against_the_library(cc, tmp_path):
    lib = os.path.join(ROOT, "paged_kv_gqa_12_gb300", "_lib", "libpa_gb300.so")
    if not os.path.exists(lib):
        pytest.skip("library not built")
    src = tmp_path / "abi.c"
    src.write_text(SOURCE)
    exe = tmp_path / "abi"
    r = subprocess.run([cc, "-std=c11", "-I" + os.path.join(ROOT, "include"), str(src), lib,
                        "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_binding_struct_layouts_match_the_header(cc, tmp_path):
    # the ctypes mirrors of pa_shape and pa_plan_t: size and every field offset
    # as the C compiler lays them out
    import ctypes
    from paged_kv_gqa_12_gb300 import binding as pb
    fields = {"pa_shape": [f[0] for f in pb.PaShape._fields_],
              "pa_plan_t": [f[0] for f in pb.PaPlan._fields_]}
    lines = ["#include <stddef.h>", "#include <stdio.h>", "#include \"pa.h\"", "int main(void) {"]
    for st, names in fields.items():
        lines.append(f'  printf("{st} size %zu\\n", sizeof({st}));')
        for n in names:
            lines.append(f'  printf("{st} {n} %zu\\n", offsetof({st}, {n}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    r = subprocess.run([cc, "-std=c11", "-I" + os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    got = {}
    for line in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines():
        parts = line.split()
        got[(parts[0], parts[1])] = int(parts[2])
    for st, cls in (("pa_shape", pb.PaShape), ("pa_plan_t", pb.PaPlan)):
        assert got[(st, "size")] == ctypes.sizeof(cls), st
        for n in fields[st]:
            assert got[(st, n)] == getattr(cls, n).offset, (st, n)
