"""The work decomposition of csrc/vcd_plan.h, checked on the host (CPU only).

A small C++ program includes the plan header and prints every plan field for
many (S, C, policy, launch shape) cases, normal and with the transposed narrow
last column; the test checks what the kernels rely on: the units and chunks
cover the tokens exactly, the "fp32" units stay within 256 tokens and on the
8-token batch grid, a transposed plan's pieces cover each chunk and its
assignments fit one wave of resident warps, and the partial rows stay within
the bound include/vcd.h states. Needs g++."""
import itertools
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "varlen_causal_depthwise_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstdlib>
#include "vcd_plan.h"
using namespace vcd;
int main(int argc, char** argv) {
    for (int i = 1; i + 4 < argc + 1; i += 4) {
        const long S = atol(argv[i]), C = atol(argv[i + 1]);
        const int pol = atoi(argv[i + 2]), shape = atoi(argv[i + 3]);
        for (int t = 0; t < 2; ++t) {
            const BwdPlan p = bwd_plan(S, C, pol, shape, t == 1);
            printf("%ld %ld %d %d %d %ld %ld %ld %ld %ld %ld %ld %ld %ld %ld %ld %ld\n", S, C, pol, shape, t,
                   (long)p.ncols, (long)p.nfull, (long)p.rows, (long)p.L, (long)p.per, (long)p.chunks,
                   (long)p.ng, (long)p.h, (long)p.q, (long)p.nnarrow, (long)p.groups,
                   (long)bwd_workspace_bytes_for(S, C, pol, shape, t == 1));
        }
    }
    return 0;
}
"""

FIELDS = ("S", "C", "pol", "shape", "transpose", "ncols", "nfull", "rows", "L", "per", "chunks",
          "ng", "h", "q", "nnarrow", "groups", "ws")
WARPS = {0: 152 * 12, 1: 152 * 16, 2: 152 * 12}


def _cases():
    rng = np.random.default_rng(11)
    Ss = [1, 7, 16, 63, 300, 4096, 8000, 32768, 65536, 131072, 262144, 1 << 20]
    Cs = [8, 16, 40, 64, 72, 128, 136, 264, 1032, 2056, 6144, 8200]
    out = [(S, C) for S, C in itertools.product(Ss, Cs)]
    out += [(int(rng.integers(1, 1 << 21)), 8 * int(rng.integers(1, 2000))) for _ in range(120)]
    return [(S, C, pol, shape) for S, C in out for pol, shape in ((0, 0), (0, 1), (0, 2), (1, 2))]


@pytest.fixture(scope="module")
def plans():
    if shutil.which("g++") is None:
        pytest.skip("g++ is missing")
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "plan.cpp"), os.path.join(d, "plan")
        with open(src, "w") as f:
            f.write(PROGRAM)
        subprocess.run(["g++", "-O1", "-std=c++17", f"-I{CSRC}", src, "-o", exe], check=True)
        args = [str(v) for case in _cases() for v in case]
        out = subprocess.run([exe, *args], check=True, capture_output=True, text=True).stdout
    return [dict(zip(FIELDS, map(int, line.split()))) for line in out.splitlines()]


def test_units_and_chunks_cover_the_tokens(plans):
    for p in plans:
        S, L, rows, per, chunks = p["S"], p["L"], p["rows"], p["per"], p["chunks"]
        assert rows * L >= S > (rows - 1) * L, p
        assert chunks * per >= rows > (chunks - 1) * per, p
        assert L >= min(S, 16) or rows * L == S, p          # the shortest unit, but for tiny S
        if not p["transpose"] or p["nnarrow"] == 0:          # one wave of warps
            assert p["chunks"] <= max(1, WARPS[p["shape"]] // p["ncols"]), p


def test_fp32_units(plans):
    for p in plans:
        if p["pol"] != 1:
            assert p["per"] == 1, p
            continue
        assert p["L"] <= 256, p                              # FP32 sums of at most 256 terms
        if p["per"] > 1:
            assert p["L"] % 8 == 0, p                         # unit boundaries on the batch grid
            assert p["nfull"] * p["chunks"] + p["nnarrow"] <= WARPS[2], p


def test_transposed_narrow_column(plans):
    for p in plans:
        g = p["groups"] - 32 * (p["ncols"] - 1)
        if not p["transpose"]:
            assert p["nfull"] == p["ncols"] and p["nnarrow"] == 0, p
            continue
        if p["nnarrow"] == 0:
            assert p["nfull"] == p["ncols"], p
            assert g > 16 or p["ncols"] > 3072 or p["per"] > 32 // g, p   # no transposed plan applies
            continue
        m = 32 // g
        assert g <= 16 and p["ng"] == g and p["nfull"] == p["ncols"] - 1, p
        assert p["h"] % p["per"] == 0 and p["q"] == m // p["h"] >= 1, p   # pieces on unit bounds
        P = -(-p["per"] * p["L"] // p["h"])
        assert p["h"] * P >= p["per"] * p["L"], p                         # pieces cover a chunk
        assert p["nnarrow"] * p["q"] >= p["chunks"] > (p["nnarrow"] - 1) * p["q"], p
        assert p["nfull"] * p["chunks"] + p["nnarrow"] <= WARPS[p["shape"]], p
        assert p["chunks"] * p["ncols"] <= 3072, p


def test_partial_rows_and_workspace(plans):
    for p in plans:
        assert p["ws"] == p["chunks"] * p["ncols"] * 2560, p
        assert p["chunks"] * p["ncols"] <= max(3072, p["ncols"]), p


def test_boundary_plans_as_measured(plans):
    """The plans the boundary workload's backward runs (131072 x 1032)."""
    by = {(p["S"], p["C"], p["pol"], p["shape"], p["transpose"]): p for p in plans}
    bf = by[(131072, 1032, 0, 2, 1)]
    assert (bf["nfull"], bf["chunks"], bf["L"], bf["h"], bf["q"], bf["nnarrow"]) == (8, 221, 594, 4, 4, 56)
    fp = by[(131072, 1032, 1, 2, 1)]
    assert (fp["per"], fp["L"], fp["chunks"], fp["h"], fp["q"], fp["nnarrow"]) == (3, 208, 211, 6, 2, 106)
    nt = by[(131072, 1032, 1, 2, 0)]
    assert (nt["per"], nt["L"], nt["chunks"]) == (3, 224, 196)
