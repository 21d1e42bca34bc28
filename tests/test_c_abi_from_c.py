"""The C ABI from C: include/moe.h compiles as C99, and a C program linked
against libmoe_gb300.so gets the host-side answers (status strings, router
workspace size, refusals, the empty forward) without touching a device."""
import os
import shutil
import subprocess

import pytest

from moe_ffn_speculative_gb300.build import LIB, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INCLUDE = "/usr/local/cuda/include"

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "moe.h"

#define CHECK(c) do { if (!(c)) { printf("FAIL line %d: %s\n", __LINE__, #c); return 1; } } while (0)

static moe_recipe recipe(int E, int K) {
  moe_recipe r;
  memset(&r, 0, sizeof(r));
  r.num_experts = E; r.top_k = K; r.score_fn = MOE_SCORE_SOFTMAX;
  r.n_group = 1; r.topk_group = 1; r.group_topn = 2;
  r.norm_topk_prob = 1; r.norm_eps = 1e-20f; r.route_scale = 1.0f; r.swiglu_limit = 0.0f;
  return r;
}

int main(void) {
  const moe_recipe ok = recipe(8, 2), bad_k = recipe(8, 9);
  /* plain addresses that no call below dereferences: every one is refused or empty first */
  const moe_bf16* x = (const moe_bf16*)(uintptr_t)(1u << 20);
  const moe_bf16* g = (const moe_bf16*)(uintptr_t)(3u << 20);
  const moe_bf16* wgu = (const moe_bf16*)(uintptr_t)(4u << 20);
  const moe_bf16* wd = (const moe_bf16*)(uintptr_t)(5u << 20);
  void* ws = (void*)(uintptr_t)(6u << 20);
  moe_bf16* y = (moe_bf16*)(uintptr_t)(2u << 20);
  CHECK(strcmp(moe_status_string(MOE_OK), "MOE_OK") == 0);
  CHECK(strcmp(moe_status_string(MOE_ERR_WORKSPACE), "MOE_ERR_WORKSPACE") == 0);
  CHECK(moe_route_workspace_bytes(72, 8) >= 256 + 4 * 72 * 8);
  CHECK(moe_route_workspace_bytes(-1, 8) == 0);
  CHECK(moe_ffn_forward(x, 16, 64, 32, g, NULL, NULL, wgu, wd, NULL, NULL, 0, NULL, &bad_k, ws, 1u << 30, y,
                        NULL, NULL, NULL, (cudaStream_t)0) == MOE_ERR_UNSUPPORTED);
  CHECK(moe_ffn_forward(x, 16, 60, 32, g, NULL, NULL, wgu, wd, NULL, NULL, 0, NULL, &ok, ws, 1u << 30, y,
                        NULL, NULL, NULL, (cudaStream_t)0) == MOE_ERR_UNSUPPORTED);
  CHECK(moe_ffn_forward(x, 16, 64, 32, g, NULL, NULL, wgu, wd, NULL, NULL, 0, NULL, &ok, ws, 1u << 30,
                        (moe_bf16*)x, NULL, NULL, NULL, (cudaStream_t)0) == MOE_ERR_INVALID_ARG);
  CHECK(moe_ffn_forward(x, 0, 64, 32, g, NULL, NULL, wgu, wd, NULL, NULL, 0, NULL, &ok, ws, 1u << 30, y,
                        NULL, NULL, NULL, (cudaStream_t)0) == MOE_OK);
  CHECK(moe_route_from_logits(NULL, 0, NULL, &ok, NULL, NULL, (cudaStream_t)0) == MOE_OK);
  CHECK(moe_set_schedule(7) == MOE_ERR_INVALID_ARG);
  CHECK(moe_set_launch_overlap(2) == MOE_ERR_INVALID_ARG);
  CHECK(moe_set_launch_overlap(1) == MOE_OK);
  printf("c abi ok\n");
  return 0;
}
"""


@pytest.fixture(scope="module")
def lib_path():
    build()
    return LIB


def test_header_compiles_as_c99_and_a_c_program_links_and_runs(lib_path, tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None or not os.path.isdir(CUDA_INCLUDE):
        pytest.skip("no C compiler or CUDA headers")
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(lib_path)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", str(src), "-I", os.path.join(ROOT, "include"),
                        "-I", CUDA_INCLUDE, "-L", libdir, "-l:" + os.path.basename(lib_path),
                        "-Wl,-rpath," + libdir, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0 and "c abi ok" in run.stdout, run.stdout + run.stderr
