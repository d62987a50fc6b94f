"""The register budgets the launch shapes are chosen by.

The backward picks its launch shape on the host from the route: the wide shape
(12 warps, up to 168 registers) for "bf16"-policy calls with a bias and longer
documents, the deep shape (16 warps, at most 128 registers) otherwise. That
rule rests on the compiled kernels: every wide-shape kernel and every forward
kernel (both batch shapes) keeps its state in registers, and so do the deep
shape's "bf16"-policy kernels without a bias. A source change that makes one of
those spill silently makes its route slower, so this test compiles the kernels
with ptxas' resource report and checks the spill counts. CPU only (nvcc
cross-compiles for sm_103a).
"""
import concurrent.futures
import os
import re
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "varlen_causal_depthwise_gb300", "csrc")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

pytestmark = pytest.mark.skipif(not os.path.exists(NVCC) and shutil.which("nvcc") is None,
                                reason="nvcc not available")


def _resources(src):
    """{mangled kernel name: (registers, spill store bytes, spill load bytes)}."""
    with tempfile.TemporaryDirectory() as d:
        cmd = [NVCC if os.path.exists(NVCC) else "nvcc", "-gencode", "arch=compute_103a,code=sm_103a",
               "-O3", "-std=c++17", f"-I{os.path.join(ROOT, 'include')}", f"-I{CSRC}",
               "-Xptxas", "-v", "-c", os.path.join(CSRC, src), "-o", os.path.join(d, "k.o")]
        out = subprocess.run(cmd, capture_output=True, text=True, check=True).stderr
    res, cur, spill = {}, None, None
    for line in out.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            cur, spill = m.group(1), None
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m:
            spill = (int(m.group(1)), int(m.group(2)))
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and cur:
            res[cur] = (int(m.group(1)),) + (spill or (0, 0))
            cur = None
    return res


@pytest.fixture(scope="module")
def resources():
    with concurrent.futures.ThreadPoolExecutor(2) as ex:
        fwd, bwd = ex.map(_resources, ["vcd_fwd.cu", "vcd_bwd.cu"])
    return fwd, bwd


def _main_kernels(bwd):
    """(shape, weight bf16, bias kind, policy, multi-unit chunks) -> resources."""
    out = {}
    for name, r in bwd.items():
        m = re.search(r"bwd_main_kernelILi(\d)ELb([01])ELi(\d)ELi(\d)ELb([01])E", name)
        if m:
            out[tuple(int(g) for g in m.groups())] = r
    return out


def test_forward_kernels_do_not_spill(resources):
    fwd, _ = resources
    kernels = {n: r for n, r in fwd.items() if "fwd_kernel" in n}
    # per batch shape: 4 routes specialised on their dtypes, 1 taking them at run time
    assert len(kernels) == 10
    for name, (regs, st, ld) in kernels.items():
        assert st == 0 and ld == 0, f"{name}: {regs} registers, spills {st}/{ld} bytes"


def test_backward_shapes_fit_their_register_budgets(resources):
    _, bwd = resources
    k = _main_kernels(bwd)
    # wide shape: "bf16" policy with a bias only, every weight dtype x bias dtype x chunk form
    wide = {key: r for key, r in k.items() if key[0] == 0}
    deep = {key: r for key, r in k.items() if key[0] == 1}
    assert len(wide) == 8 and len(deep) == 24
    assert all(key[3] == 0 and key[2] != 0 for key in wide)
    for key, (regs, st, ld) in wide.items():
        assert regs <= 168 and st == 0 and ld == 0, f"wide {key}: {regs} registers, spills {st}/{ld}"
    for key, (regs, st, ld) in deep.items():
        assert regs <= 128, f"deep {key}: {regs} registers"
    # the deep shape runs mask-free "bf16" calls only where it keeps everything
    # in registers: the routes without a bias (single-unit chunks)
    for wb in (0, 1):
        regs, st, ld = deep[(1, wb, 0, 0, 0)]
        assert st == 0 and ld == 0, f"deep bf16 no-bias (weight bf16={wb}) spills {st}/{ld} bytes"
