"""The C ABI library loads on any host, exports every entry point include/vcd.h
declares, and rejects bad arguments before touching the GPU (CPU only)."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import varlen_causal_depthwise_gb300 as vcd
from varlen_causal_depthwise_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vcd.h")
STREAM_HEADER = os.path.join(ROOT, "include", "vcd_stream.h")


def declared(header=HEADER, prefix="conv1d_"):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    pat = r"^\s*(?:const\s+)?\w+\*?\s+\*?(" + prefix + r"\w+)\s*\("
    return sorted(set(re.findall(pat, text, re.M)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.library_path()):
        from varlen_causal_depthwise_gb300 import build
        build.build()
    return binding.load_library()


def test_header_declares_the_entry_points():
    assert declared() == sorted(binding.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in declared():
        assert hasattr(lib, name), name


def test_stream_header_declares_the_ceiling_kernel(lib):
    assert declared(STREAM_HEADER, "vcd_") == sorted(binding.STREAM_SIGNATURES)
    for name in declared(STREAM_HEADER, "vcd_"):
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert vcd.conv1d_status_string(0) == "ok"
    for s in range(1, 5):
        assert vcd.conv1d_status_string(s) not in ("ok", "unknown status")
    assert vcd.conv1d_status_string(99) == "unknown status"


def test_workspace_queries(lib):
    assert vcd.conv1d_fwd_workspace_size(65536, 6144) == 0
    assert vcd.conv1d_bwd_workspace_size(0, 256) == 0
    n = vcd.conv1d_bwd_workspace_size(65536, 6144)
    assert n > 0 and n % 16 == 0
    for bad in ((-1, 8), (8, 0), (8, 12)):
        with pytest.raises(vcd.VcdError):
            vcd.conv1d_bwd_workspace_size(*bad)
    bf, fp = (vcd.conv1d_bwd_route_workspace_size(65536, 6144, p) for p in ("bf16", "fp32"))
    assert max(bf, fp) == n
    # one FP32 row of 128 channels x 5 values per chunk of a column. "bf16":
    # one warp-sized unit per chunk, the larger of the two launch shapes (16
    # warps per SM: 48 columns x 50 rows = 2400 units)
    assert bf == 48 * 50 * 128 * 5 * 4
    # "fp32": 38 warps per column in the chunked shape, 7 units to a chunk
    # (38 x 7 units of at most 256 tokens cover S), units of 248 tokens (the
    # shortest multiple of 8 that covers S in 38 x 7): 265 units, 38 chunks
    assert fp == 48 * 38 * 128 * 5 * 4
    with pytest.raises(ValueError):
        vcd.conv1d_bwd_route_workspace_size(8, 8, "fp16")


def test_call_workspace_query_follows_the_launch_shape(lib):
    """The per-call query gives the partial rows of the launch shape the call
    takes: 12 warps per SM (1824 target units) for the "bf16" policy with a
    bias and documents of 32 tokens or more on average and for shorter
    documents, 16 warps (2432) without a bias on longer documents; never more
    than the policy's query."""
    S, C, row = 65536, 6144, 128 * 5 * 4
    call = vcd.conv1d_bwd_call_workspace_size
    assert call(S, C, 20, "bf16", True) == 48 * 38 * row           # wide: 1824 units
    assert call(S, C, 20, "bf16", False) == 48 * 50 * row          # deep: 2400 units
    assert call(S, C, S // 32, "bf16", True) == 48 * 38 * row      # short documents: chunked
    assert call(S, C, S // 32 - 1, "bf16", True) == 48 * 38 * row
    assert call(S, C, 20, "fp32", True) == call(S, C, 20, "fp32", False) == 48 * 38 * row  # chunks
    for S_, C_, nd in ((4096, 256, 4), (131072, 1032, 52000), (300, 40, 3), (1, 8, 1)):
        for pol in ("bf16", "fp32"):
            for hb in (True, False):
                assert 0 < call(S_, C_, nd, pol, hb) <= vcd.conv1d_bwd_route_workspace_size(S_, C_, pol)
    assert call(0, 8, 0, "bf16", True) == 0
    with pytest.raises(vcd.VcdError):
        call(8, 8, 0, "bf16", True)          # tokens but no documents
    with pytest.raises(ValueError):
        call(8, 8, 1, "fp16", True)


def _fwd(lib, **kw):
    a = dict(x=16, S=4, C=8, w=16, wd=1, cu=16, nd=1, b=None, bd=1, y=32, ws=None, wsb=0)
    a.update(kw)
    return lib.conv1d_fwd(a["x"], a["S"], a["C"], a["w"], a["wd"], a["cu"], a["nd"], a["b"],
                          a["bd"], a["y"], a["ws"], a["wsb"], None)


def _bwd(lib, **kw):
    a = dict(x=16, dy=48, S=4, C=8, w=16, wd=1, cu=16, nd=1, b=None, bd=1, pol=0, dx=32,
             dw=64, dwd=1, db=None, dbd=1, ws=80, wsb=1 << 20)
    a.update(kw)
    return lib.conv1d_bwd(a["x"], a["dy"], a["S"], a["C"], a["w"], a["wd"], a["cu"], a["nd"],
                          a["b"], a["bd"], a["pol"], a["dx"], a["dw"], a["dwd"], a["db"], a["dbd"],
                          a["ws"], a["wsb"], None)


# Fake, never dereferenced addresses: every case below must fail validation
# before the library reaches the CUDA runtime.
@pytest.mark.parametrize("kw,status", [
    (dict(C=12), binding.VCD_ERR_INVALID_ARG),          # C % 8 != 0
    (dict(C=0), binding.VCD_ERR_INVALID_ARG),
    (dict(S=-1), binding.VCD_ERR_INVALID_ARG),
    (dict(nd=0), binding.VCD_ERR_INVALID_ARG),          # tokens but no documents
    (dict(wd=7), binding.VCD_ERR_INVALID_ARG),
    (dict(x=None), binding.VCD_ERR_INVALID_ARG),
    (dict(y=None), binding.VCD_ERR_INVALID_ARG),
    (dict(y=16), binding.VCD_ERR_INVALID_ARG),          # y aliases x
    (dict(x=18), binding.VCD_ERR_MISALIGNED),
    (dict(w=20), binding.VCD_ERR_MISALIGNED),
    (dict(b=24, bd=0), binding.VCD_ERR_MISALIGNED),
    (dict(y=40), binding.VCD_ERR_MISALIGNED),
])
def test_fwd_rejects(lib, kw, status):
    assert _fwd(lib, **kw) == status


def test_fwd_empty_sequence_launches_nothing(lib):
    assert _fwd(lib, S=0, nd=0, x=None, y=None, cu=16) == binding.VCD_OK
    assert _fwd(lib, S=0, nd=3) == binding.VCD_OK


@pytest.mark.parametrize("kw,status", [
    (dict(C=4), binding.VCD_ERR_INVALID_ARG),
    (dict(pol=2), binding.VCD_ERR_INVALID_ARG),
    (dict(db=96), binding.VCD_ERR_INVALID_ARG),         # dbias without bias
    (dict(dw=None), binding.VCD_ERR_INVALID_ARG),
    (dict(dwd=5), binding.VCD_ERR_INVALID_ARG),
    (dict(dx=16), binding.VCD_ERR_INVALID_ARG),         # dx aliases x
    (dict(dx=48), binding.VCD_ERR_INVALID_ARG),         # dx aliases dy
    (dict(dy=None), binding.VCD_ERR_INVALID_ARG),
    (dict(dy=50), binding.VCD_ERR_MISALIGNED),
    (dict(dw=66), binding.VCD_ERR_MISALIGNED),          # FP32 dweight needs 4 bytes
    (dict(ws=None), binding.VCD_ERR_WORKSPACE_TOO_SMALL),
    (dict(wsb=16), binding.VCD_ERR_WORKSPACE_TOO_SMALL),
    (dict(ws=88), binding.VCD_ERR_MISALIGNED),
])
def test_bwd_rejects(lib, kw, status):
    assert _bwd(lib, **kw) == status


def test_binding_refuses_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "library_path", lambda: str(tmp_path / "libvcd.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        binding.load_library()


def test_binding_rejects_host_tensors_before_any_call():
    """The C ABI takes bare device pointers: the binding must refuse host memory
    itself rather than hand the library a host address."""
    x = torch.zeros(16, 8, dtype=torch.bfloat16)
    w = torch.zeros(8, 4)
    cu = torch.tensor([0, 16], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.conv1d_fwd(x, w, cu)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.conv1d_bwd(x, x, w, cu)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.conv1d_bwd_noalloc(x, x, w, cu)


def test_workspace_queries_are_consistent(lib):
    """Random shapes: the per-call need is a whole number of 2560-byte partial
    rows, never above its policy's need, which is never above the need of every
    route; the "bf16" policy's need is the largest of its launch shapes' needs
    (16 warps without a bias, 12 warps with a bias or on short documents), and
    the "fp32" policy always takes the same (chunked) shape."""
    rng = np.random.default_rng(2024)
    call = vcd.conv1d_bwd_call_workspace_size
    for _ in range(300):
        S = int(rng.integers(1, 1 << 22))
        C = 8 * int(rng.integers(1, 1 << 13))
        nd = int(rng.integers(1, S + 1))
        total = vcd.conv1d_bwd_workspace_size(S, C)
        for pol in ("bf16", "fp32"):
            route = vcd.conv1d_bwd_route_workspace_size(S, C, pol)
            assert route <= total
            for hb in (True, False):
                n = call(S, C, nd, pol, hb)
                assert n % 2560 == 0 and 0 < n <= route
            if pol == "fp32":
                assert call(S, C, nd, pol, True) == call(S, C, 1, pol, False) == route
            elif S > 32:
                assert route == max(call(S, C, 1, pol, True), call(S, C, 1, pol, False),
                                    call(S, C, S, pol, True))
        assert total == max(vcd.conv1d_bwd_route_workspace_size(S, C, p) for p in ("bf16", "fp32"))


NOALLOC_BYTES = 8 << 20      # VCD_NOALLOC_SCRATCH_BYTES in include/vcd.h


def test_noalloc_scratch_size_matches_the_header():
    text = open(HEADER).read()
    m = re.search(r"#define\s+VCD_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == NOALLOC_BYTES


@pytest.mark.parametrize("S,C,policy,fits", [
    (1 << 20, 419328, "bf16", True),    # 3276 columns of one row each
    (1 << 20, 419336, "bf16", False),   # 3277 columns
    (1 << 20, 419328, "fp32", True),
    (1 << 20, 419336, "fp32", False),
    (262144, 311296, "bf16", True),
    (262144, 8192, "fp32", True),       # 64 columns x 28 chunks
    (1 << 20, 8, "bf16", True),         # transposed narrow column: at most 3072 rows
    (1 << 20, 136, "fp32", True),
    (1 << 20, 1032, "bf16", True),
    ((1 << 31) - 128, 6144, "fp32", True),
])
def test_noalloc_limits_stated_in_the_header(lib, S, C, policy, fits):
    """The shapes include/vcd.h names on either side of the fixed scratch's
    limit: the policy's largest need (the size conv1d_bwd_noalloc checks)
    against VCD_NOALLOC_SCRATCH_BYTES."""
    need = vcd.conv1d_bwd_route_workspace_size(S, C, policy)
    assert (need <= NOALLOC_BYTES) == fits, (S, C, policy, need)


def test_workspace_bound_stated_in_the_header(lib):
    """conv1d_bwd_workspace_size never exceeds max(3072, ceil(C / 128)) rows of
    2560 bytes (the bound include/vcd.h states), over shapes with and without
    a narrow last column."""
    rng = np.random.default_rng(5)
    cases = [(S, C) for S in (1, 63, 4096, 131072, 1 << 20, 1 << 24)
             for C in (8, 16, 40, 64, 72, 128, 136, 264, 1032, 2056, 8200, 65544)]
    cases += [(int(rng.integers(1, 1 << 22)), 8 * int(rng.integers(1, 20000))) for _ in range(200)]
    for S, C in cases:
        rows = max(3072, -(-C // 128))
        assert vcd.conv1d_bwd_workspace_size(S, C) <= rows * 2560, (S, C)


def test_exact_workspace_query(lib):
    """The exactness-guarded backward's workspace: its launch shape's partial
    rows, then per chunk a list with room for one in 64 of the chunk's
    elements (at least 64 entries of 8 bytes) and a 4-byte count, each part on
    a 16-byte boundary; 0 for S == 0; errors like the other queries."""
    assert vcd.conv1d_bwd_exact_workspace_size(0, 256) == 0
    for S, C in ((65536, 6144), (4096, 256), (131072, 1032), (7, 8)):
        n = vcd.conv1d_bwd_exact_workspace_size(S, C)
        assert n % 16 == 0
        assert n > max(vcd.conv1d_bwd_call_workspace_size(S, C, 1, p, True) for p in ("bf16", "fp32"))
    # 65536 x 6144 in the chunked shape (1824 target warps): "bf16" 38 chunks
    # of 1725 tokens per column, lists of 1725 * 128 / 64 = 3450 entries;
    # "fp32" 38 chunks of 7 units of 248 tokens, lists of 3472; the larger
    bf = 48 * 38 * (2560 + 3450 * 8 + 4)
    fp = 48 * 38 * (2560 + 3472 * 8 + 4)
    assert abs(vcd.conv1d_bwd_exact_workspace_size(65536, 6144) - max(bf, fp)) <= 32
    with pytest.raises(vcd.VcdError):
        vcd.conv1d_bwd_exact_workspace_size(8, 12)
