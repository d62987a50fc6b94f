"""The boundary is a C ABI: a plain C11 program includes include/vcd.h, links
libvcd.so and calls the entry points that need no GPU (the size queries, the
status strings, and the argument checks that run before any CUDA call). CPU
only; needs gcc and the CUDA headers."""
import os
import shutil
import subprocess
import tempfile

import pytest

import varlen_causal_depthwise_gb300 as vcd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = "/usr/local/cuda/include"

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "vcd.h"

static int fails = 0;
#define CHECK(c) do { if (!(c)) { printf("FAILED: %s (line %d)\n", #c, __LINE__); ++fails; } } while (0)

int main(void) {
    size_t fwd = 1, all = 0, bf = 0, fp = 0, call = 0;
    CHECK(conv1d_fwd_workspace_size(65536, 6144, &fwd) == VCD_OK && fwd == 0);
    CHECK(conv1d_bwd_workspace_size(65536, 6144, &all) == VCD_OK && all > 0);
    CHECK(conv1d_bwd_route_workspace_size(65536, 6144, VCD_SILU_GRAD_BF16, &bf) == VCD_OK);
    CHECK(conv1d_bwd_route_workspace_size(65536, 6144, VCD_SILU_GRAD_FP32, &fp) == VCD_OK);
    CHECK(fp > 0 && bf > 0 && all == (bf > fp ? bf : fp));
    CHECK(conv1d_bwd_call_workspace_size(65536, 6144, 20, VCD_SILU_GRAD_BF16, 1, &call) == VCD_OK);
    CHECK(call > 0 && call <= bf && call % 2560 == 0);
    CHECK(conv1d_bwd_workspace_size(64, 12, &all) == VCD_ERR_INVALID_ARG);     /* C % 8 != 0 */
    CHECK(conv1d_bwd_route_workspace_size(64, 8, 7, &bf) == VCD_ERR_INVALID_ARG);
    CHECK(conv1d_bwd_call_workspace_size(64, 8, 0, VCD_SILU_GRAD_BF16, 1, &call) == VCD_ERR_INVALID_ARG);
    CHECK(strcmp(conv1d_status_string(VCD_OK), "ok") == 0);
    CHECK(strcmp(conv1d_status_string(99), "unknown status") == 0);
    /* argument errors are reported before anything touches the GPU */
    CHECK(conv1d_fwd(NULL, 16, 8, NULL, VCD_FP32, NULL, 1, NULL, VCD_FP32, NULL, NULL, 0, 0)
          == VCD_ERR_INVALID_ARG);
    CHECK(conv1d_bwd(NULL, NULL, 16, 12, NULL, VCD_FP32, NULL, 1, NULL, VCD_FP32,
                     VCD_SILU_GRAD_BF16, NULL, NULL, VCD_FP32, NULL, VCD_FP32, NULL, 0, 0)
          == VCD_ERR_INVALID_ARG);
    CHECK(conv1d_bwd_noalloc(NULL, NULL, 16, 8, NULL, VCD_FP32, NULL, 1, NULL, VCD_FP32, 5,
                             NULL, NULL, VCD_FP32, NULL, VCD_FP32, 0) == VCD_ERR_INVALID_ARG);
    printf("%s\n", fails ? "some checks failed" : "all checks passed");
    return fails != 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None or not os.path.isdir(CUDA_INC),
                    reason="gcc or the CUDA headers are missing")
def test_plain_c_program_uses_the_library():
    lib = vcd.library_path()
    if not os.path.exists(lib):
        pytest.skip("libvcd.so is not built")
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "caller.c"), os.path.join(d, "caller")
        with open(src, "w") as f:
            f.write(PROGRAM)
        subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        f"-I{os.path.join(ROOT, 'include')}", f"-I{CUDA_INC}", src,
                        "-o", exe, f"-L{os.path.dirname(lib)}", "-lvcd",
                        f"-Wl,-rpath,{os.path.dirname(lib)}"], check=True,
                       capture_output=True, text=True)
        r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "all checks passed" in r.stdout
