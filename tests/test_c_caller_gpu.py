"""A C program that uses only include/pa.h and the CUDA runtime: a window-1
decode (each query attends to its own key only, so every output row must be
that key's value row, bit for bit) planned, run and checked without Python
in the loop."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SOURCE = r"""
#include <stdint.h>
#include <stdio.h>
#include <string.h>
#include <cuda_runtime_api.h>
#include "pa.h"

enum { B = 2, HQ = 8, HKV = 2, D = 64, PS = 16, POOL = 8, W = 4 };

int main(void) {
  static uint16_t q[B * HQ * D], kv[POOL * PS * HKV * D], out[B * HQ * D];
  const int32_t lens[B] = {20, 7};
  const int32_t bt[B * W] = {3, 5, 0, 0, 1, 6, 0, 0};
  uint32_t x = 12345u;
  for (int i = 0; i < POOL * PS * HKV * D; ++i) { x = x * 1664525u + 1013904223u; kv[i] = (uint16_t)(0x3C00u + (x >> 22)); }
  for (int i = 0; i < B * HQ * D; ++i) { x = x * 1664525u + 1013904223u; q[i] = (uint16_t)(0x3E00u + (x >> 23)); }
  pa_shape s;
  memset(&s, 0, sizeof s);
  s.mode = PA_MODE_DECODE; s.num_q_heads = HQ; s.num_kv_heads = HKV; s.head_dim = D; s.page_size = PS;
  s.kv_dtype = PA_KV_BF16; s.max_batch = B; s.max_pages_per_seq = W; s.window = 1; s.num_splits = 2;
  pa_plan_t plan;
  if (pa_plan(&s, NULL, 0, &plan) != PA_OK) { printf("plan failed\n"); return 2; }
  void *dq, *dk, *dv, *dout, *scratch;
  int32_t *dbt, *dlen;
  if (cudaMalloc(&dq, sizeof q) || cudaMalloc(&dk, sizeof kv) || cudaMalloc(&dv, sizeof kv) ||
      cudaMalloc(&dout, sizeof out) || cudaMalloc((void**)&dbt, sizeof bt) || cudaMalloc((void**)&dlen, sizeof lens) ||
      cudaMalloc(&scratch, (size_t)plan.scratch_bytes)) { printf("cudaMalloc failed\n"); return 3; }
  cudaMemcpy(dq, q, sizeof q, cudaMemcpyHostToDevice);
  cudaMemcpy(dk, kv, sizeof kv, cudaMemcpyHostToDevice);   /* K and V share the values here */
  cudaMemcpy(dv, kv, sizeof kv, cudaMemcpyHostToDevice);
  cudaMemcpy(dbt, bt, sizeof bt, cudaMemcpyHostToDevice);
  cudaMemcpy(dlen, lens, sizeof lens, cudaMemcpyHostToDevice);
  if (pa_scratch_init(scratch, NULL) != PA_OK) return 4;
  pa_status st = pa_decode(&plan, dq, HQ * D, D, dk, dv, PS * HKV * D, HKV * D, D, POOL, dbt, W, dlen, B,
                           0.125f, NULL, 1.f, 1.f, NULL, NULL, dout, HQ * D, D, NULL,
                           scratch, plan.scratch_bytes, NULL);
  if (st != PA_OK) { printf("pa_decode: %s\n", pa_status_string(st)); return 5; }
  uint32_t code = 0;
  if (pa_check(scratch, NULL, &code) != PA_OK) { printf("device error %u\n", code); return 6; }
  cudaMemcpy(out, dout, sizeof out, cudaMemcpyDeviceToHost);
  int bad = 0;
  for (int b = 0; b < B; ++b) {
    const int pos = lens[b] - 1, page = bt[b * W + pos / PS], slot = pos % PS;
    for (int h = 0; h < HQ; ++h)
      for (int d = 0; d < D; ++d) {
        const uint16_t want = kv[((page * PS + slot) * HKV + h / (HQ / HKV)) * D + d];
        if (out[(b * HQ + h) * D + d] != want) ++bad;
      }
  }
  printf("version %d, mismatches %d\n", pa_version(), bad);
  return bad == 0 ? 0 : 1;
}
"""


def test_c_program_decodes_through_the_abi(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = os.path.join(ROOT, "paged_kv_gqa_12_gb300", "_lib", "libpa_gb300.so")
    if not os.path.exists(lib):
        pytest.skip("library not built")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    src = tmp_path / "caller.c"
    src.write_text(SOURCE)
    exe = tmp_path / "caller"
    libdirs = [d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "targets", "sbsa-linux", "lib"),
                           os.path.join(cuda, "targets", "x86_64-linux", "lib")) if os.path.isdir(d)]
    cmd = [cc, "-std=c11", "-O1", "-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(cuda, "include"),
           str(src), lib, "-Wl,-rpath," + os.path.dirname(lib)]
    for d in libdirs:
        cmd += ["-L" + d, "-Wl,-rpath," + d]
    cmd += ["-lcudart", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches 0" in r.stdout
