"""A plain C99 program against include/moe.h and libmoe_gb300.so (no GPU):
the header compiles as C, the library links and loads without Python or
PyTorch, and the calls that need no device (version, status names, problem
validation, device-free planning) answer from C exactly what the Python
binding answers."""

import os
import shutil
import subprocess

import pytest

from routed_expert_ffn_gemm_gb300 import api, build, inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "routed_expert_ffn_gemm_gb300")

C_SOURCE = r"""
#include <stdio.h>
#include "moe.h"

int main(void) {
  /* Mixtral-shaped layer, 64 tokens, bf16 */
  moe_problem p = {64, 4096, 14336, 8, 2, 0, MOE_BF16, MOE_BF16};
  moe_problem bad = {4, 4096, 14336, 8, 2, 0, MOE_F32, MOE_BF16}; /* mixed dtypes */
  int32_t info[6], launches = 0;
  size_t ws = 0;
  if (moe_abi_version() != MOE_ABI_VERSION) return 10;
  if (moe_plan_info_for(&p, 152, info) != MOE_OK) return 11;
  if (moe_layer_launch_count_for(&p, 152, &launches) != MOE_OK) return 12;
  if (moe_workspace_size_for(&p, 152, &ws) != MOE_OK) return 13;
  if (moe_plan_info_for(&p, 0, info) != MOE_ERR_INVALID_ARG) return 14;
  printf("plan %d %d %d %d %d %d\n", info[0], info[1], info[2], info[3], info[4], info[5]);
  printf("launches %d\n", launches);
  printf("workspace %zu\n", ws);
  printf("bad %d %s\n", moe_workspace_size_for(&bad, 152, &ws),
         moe_status_string(moe_workspace_size_for(&bad, 152, &ws)));
  return 0;
}
"""


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    build.build()
    d = tmp_path_factory.mktemp("c_client")
    src = d / "client.c"
    src.write_text(C_SOURCE)
    exe = d / "client"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", PKG, "-lmoe_gb300", f"-Wl,-rpath,{PKG}"],
                   check=True, capture_output=True, text=True)
    return exe


def test_c_program_answers_as_the_binding(program):
    r = subprocess.run([str(program)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    lines = dict(ln.split(" ", 1) for ln in r.stdout.strip().splitlines())
    shape = inputs.WORKLOADS["mixtral_8x7b"].with_T(64)
    p = api.problem_of(shape)
    pl = api.moe_plan_info_for(p, 152)
    want = [pl["bn_gateup"], pl["bn_down"], pl["splits_down"], pl["grid"], pl["splits_gateup"],
            pl["pair_gateup"] | (pl["pair_down"] << 1)]
    assert [int(v) for v in lines["plan"].split()] == want
    assert int(lines["launches"]) == api.moe_layer_launch_count_for(p, 152)
    assert int(lines["workspace"]) == api.moe_workspace_size_for(p, 152)
    assert lines["bad"] == f"{api.ERR_UNSUPPORTED} MOE_ERR_UNSUPPORTED"
