"""The C ABI from plain C: include/m2.h compiles as C99 with warnings as
errors, a C program links against libm2.so, and the host-side refusals work
without a device (no kernel is launched)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "mamba2_ssm_mixer_gb300")

C_SRC = r"""
#include <stdio.h>
#include <string.h>
#include "m2.h"

#define CHECK(cond) do { if (!(cond)) { printf("failed: %s (%s)\n", #cond, m2_last_error()); return 1; } } while (0)

int main(void) {
  m2_config c = {2048, 4096, 64, 64, 8, 128, 4, 256, M2_DTYPE_F32, 1e-5f, 1.0f / 64, 1.0f / 32, M2_ARM_W8A8};
  unsigned char buf[64];
  m2_weights w;
  m2_handle* h = NULL;
  size_t n = 0;
  memset(&w, 0, sizeof w);
  w.in_proj = buf; w.out_proj = buf; w.s_w1 = 0.01f; w.s_w2 = 0.01f;
  w.conv_w = (const uint16_t*)buf; w.A_log = (const float*)buf; w.D = (const float*)buf;
  w.dt_bias = (const float*)buf; w.norm_w = (const uint16_t*)buf; w.layout = M2_LAYOUT_OUT_IN;

  CHECK(m2_create(&c, &w, &h) == M2_ESHAPE && h == NULL);          /* other geometry */
  c.hidden = 2688;
  c.arm = 7;
  CHECK(m2_create(&c, &w, &h) == M2_EINVAL && h == NULL);          /* unknown arm */
  c.arm = M2_ARM_W8A16;
  c.ssm_dtype = 9;
  CHECK(m2_create(&c, &w, &h) == M2_EINVAL && h == NULL);          /* unknown state dtype */
  CHECK(m2_create(NULL, NULL, NULL) == M2_EINVAL);
  CHECK(m2_prefill(NULL, NULL, NULL, 0, NULL, NULL, NULL, NULL, NULL, 0, NULL) == M2_EINVAL);
  CHECK(m2_decode(NULL, NULL, 1, NULL, NULL, 1, NULL, NULL, NULL, 0, NULL) == M2_EINVAL);
  CHECK(m2_mixed(NULL, NULL, 0, NULL, NULL, 0, NULL, NULL, 0, NULL, NULL, NULL, NULL, NULL, 0, NULL) == M2_EINVAL);
  CHECK(fp8_quant(NULL, 16, 1.0f, NULL, NULL) == M2_EINVAL);
  CHECK(fp8_dequant(NULL, 16, 1.0f, NULL, NULL) == M2_EINVAL);
  CHECK(fp8_linear_workspace_size(8, 8, 20, &n) == M2_ESHAPE);
  CHECK(fp8_linear_workspace_size(64, 10304, 2688, &n) == M2_OK && n == 0);
  CHECK(fp8_linear_workspace_size(200, 10304, 2688, &n) == M2_OK && n > 0);
  CHECK(bf16_linear_workspace_size(64, 10304, 2688, &n) == M2_OK && n == 0);
  CHECK(bf16_linear_workspace_size(200, 10304, 2688, &n) == M2_OK && n > 0);
  CHECK(bf16_linear(NULL, NULL, 1.0f, NULL, 4, 4, 24, NULL, 0, NULL) == M2_ESHAPE);
  CHECK(m2_rmsnorm_residual(NULL, NULL, NULL, 1e-5f, NULL, 4, 12, NULL) == M2_ESHAPE);
  CHECK(m2_check(NULL) == M2_EINVAL);
  m2_destroy(NULL);
  printf("ok\n");
  return 0;
}
"""


def test_header_is_c99_and_refusals_work_from_c(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    lib = os.path.join(PKG, "libm2.so")
    if not os.path.exists(lib):
        import __graft_entry__
        __graft_entry__.build()
    src = tmp_path / "abi.c"
    src.write_text(C_SRC)
    exe = tmp_path / "abi"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-L", PKG, "-lm2", f"-Wl,-rpath,{PKG}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
