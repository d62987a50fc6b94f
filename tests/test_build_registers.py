"""The register budgets the launch shapes are chosen by.

The backward picks its launch shape on the host from the route: the wide shape
(12 warps, up to 168 registers) for "bf16"-policy calls with a bias and longer
documents, the deep shape (16 warps, at most 128 registers) for "bf16"-policy
calls without a bias on longer documents, and the chunked shape (12 warps, up
to 168 registers) for the "fp32" policy and for short documents. That rule
rests on the compiled kernels: every wide-shape and chunked-shape kernel and
every forward kernel (both batch shapes) keeps its state in registers, and so
do the deep shape's kernels (which have no bias). A
source change that makes one of those spill silently makes its route slower,
so this test compiles the kernels with ptxas' resource report and checks the
spill counts. CPU only (nvcc cross-compiles for sm_103a).
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
    """(shape, weight bf16, bias kind, policy, multi-unit chunks, transposed
    narrow column) -> resources, for the routes specialised on their dtypes."""
    out = {}
    for name, r in bwd.items():
        m = re.search(r"bwd_main_kernelILi(\d)ELb([01])ELi(\d)ELi(\d)ELb([01])ELb0ELb([01])E", name)
        if m:
            out[tuple(int(g) for g in m.groups())] = r
    return out


def test_forward_kernels_do_not_spill(resources):
    fwd, _ = resources
    kernels = {n: r for n, r in fwd.items() if "fwd_kernel" in n}
    # per batch shape: 4 routes specialised on their dtypes, 1 taking them at run
    # time; the exactness-guarded shape: the run-time route only
    assert len(kernels) == 11
    for name, (regs, st, ld) in kernels.items():
        if "fwd_kernelILi2E" in name:
            # the exactness-guarded forward: its unrolled loop spills a few
            # words at 128 registers and still runs faster than the rolled
            # loop without spills (measured); bounded here
            assert st <= 64 and ld <= 64, f"{name}: {regs} registers, spills {st}/{ld} bytes"
            continue
        assert st == 0 and ld == 0, f"{name}: {regs} registers, spills {st}/{ld} bytes"


def test_backward_shapes_fit_their_register_budgets(resources):
    _, bwd = resources
    k = _main_kernels(bwd)
    # wide: "bf16" policy with a bias, one unit per chunk; deep: "bf16" policy
    # without a bias, one unit per chunk; chunked: "fp32" policy, both forms,
    # and the "bf16" policy's short-document calls, one unit per chunk
    # the kernels for plans with the transposed narrow column (a separate
    # instantiation of every route: the path it adds costs registers) may
    # spill a few words; the others are held to the shapes' budgets below
    narrow = {key: r for key, r in k.items() if key[5] == 1}
    assert len(narrow) == 24
    for key, (regs, st, ld) in narrow.items():
        assert regs <= (128 if key[0] == 1 else 168), f"narrow {key}: {regs} registers"
        assert st <= 64 and ld <= 96, f"narrow {key}: {regs} registers, spills {st}/{ld}"
    k = {key[:5]: r for key, r in k.items() if key[5] == 0}
    wide = {key: r for key, r in k.items() if key[0] == 0}
    deep = {key: r for key, r in k.items() if key[0] == 1}
    chunked = {key: r for key, r in k.items() if key[0] == 2}
    # the exactness-guarded route: chunked shape, dtypes at run time (not in k,
    # whose pattern matches the specialised routes), without spills
    exact = {n: r for n, r in bwd.items() if "bwd_main_kernel" in n and "Lin1E" in n}
    assert len(exact) == 3
    for name, (regs, st, ld) in exact.items():
        assert regs <= 168 and st == 0 and ld == 0, f"{name}: {regs} registers, spills {st}/{ld}"
    assert len(wide) == 4 and len(deep) == 2 and len(chunked) == 18
    assert all(key[3] == 0 and key[2] != 0 and key[4] == 0 for key in wide)
    assert all(key[3] == 0 and key[2] == 0 and key[4] == 0 for key in deep)
    assert all(key[3] == 1 or key[4] == 0 for key in chunked)
    for key, (regs, st, ld) in list(wide.items()) + list(chunked.items()):
        assert regs <= 168, f"{key}: {regs} registers"
    for key, (regs, st, ld) in wide.items():
        assert st == 0 and ld == 0, f"wide {key}: {regs} registers, spills {st}/{ld}"
    for key, (regs, st, ld) in chunked.items():
        # the multi-unit form every large "fp32" call takes: at most one spilled
        # word (with the packed accurate SiLU' some routes spill 4 bytes, and
        # still run faster than the scalar form without spills, measured)
        if key[4] == 1:
            assert st <= 4 and ld <= 4, f"chunked {key}: {regs} registers, spills {st}/{ld}"
    for key, (regs, st, ld) in deep.items():
        assert regs <= 128, f"deep {key}: {regs} registers"
    # the deep shape runs mask-free "bf16" calls only where it keeps everything
    # in registers: the routes without a bias
    for wb in (0, 1):
        regs, st, ld = deep[(1, wb, 0, 0, 0)]
        assert st == 0 and ld == 0, f"deep bf16 no-bias (weight bf16={wb}) spills {st}/{ld} bytes"
