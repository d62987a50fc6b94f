"""conv1d_bwd_noalloc -- the backward for callers that cannot give the library
device memory -- must give what conv1d_bwd gives.

Some callers cannot hand the library a workspace: a plugin inside a host
program whose device memory belongs to an allocator it cannot reach, or code
that must not call cudaMalloc/cudaFree while it runs. This entry point keeps its
partial rows in a fixed array inside the library. The test calls it through the
C ABI twice in a row (the second call finds the first call's rows in the shared
array) and compares each result with conv1d_bwd's under the same tolerances as
the parity tests; both run the same fixed-order reduction, so the bits match.

Named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import varlen_causal_depthwise_gb300 as vcd
from varlen_causal_depthwise_gb300 import binding, synth
from _check import REL_L2, bf16_close, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _abi_noalloc(w, policy, dx, dW, dB):
    lib = vcd.load_library()
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    dt = lambda t: binding.VCD_FP32 if t is None or t.dtype == torch.float32 else binding.VCD_BF16
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.conv1d_bwd_noalloc(p(w.x), p(w.dy), w.S, w.C, p(w.weight), dt(w.weight),
                                  p(w.cu_seqlens), w.cu_seqlens.numel() - 1, p(w.bias),
                                  dt(w.bias), binding.POLICIES[policy], p(dx), p(dW), dt(dW),
                                  p(dB), dt(dB), stream)


@pytest.mark.parametrize("name,S,C", [("linattn", 8192, 6144), ("boundary", 4096, 1032),
                                      ("mid", 3000, 264)])
def test_noalloc_matches_workspace_entry_point(name, S, C):
    w = synth.make(name, device=DEV, S=S, C=C)
    for policy in synth.RECIPES[name].policies:
        dB_ref = None if w.bias is None else torch.empty(C, device=DEV)
        ref = vcd.conv1d_bwd(w.x, w.dy, w.weight, w.cu_seqlens, w.bias, policy,
                             dweight=torch.empty(C, 4, device=DEV), dbias=dB_ref)
        torch.cuda.synchronize()
        for call in range(2):
            dx = torch.full_like(w.x, float("nan"))
            dW = torch.full((C, 4), float("nan"), device=DEV)
            dB = None if w.bias is None else torch.full((C,), float("nan"), device=DEV)
            assert _abi_noalloc(w, policy, dx, dW, dB) == binding.VCD_OK
            torch.cuda.synchronize()
            what = f"{name} {policy} call {call}"
            bf16_close(dx.double().cpu().numpy(), ref[0].double().cpu().numpy(), None, what)
            assert rel_l2(dW.double().cpu().numpy(), ref[1].double().cpu().numpy()) <= REL_L2[policy]
            assert torch.equal(dx, ref[0]) and torch.equal(dW, ref[1])
            if dB is not None:
                assert rel_l2(dB.double().cpu().numpy(), ref[2].double().cpu().numpy()) <= REL_L2[policy]
                assert torch.equal(dB, ref[2])


def test_noalloc_refuses_shapes_beyond_its_scratch():
    S, C = 4, 524288          # 4096 channel columns -> 10 MiB of partial rows > 8 MiB
    assert vcd.conv1d_bwd_workspace_size(S, C) > 8 << 20
    w = synth.custom(S, C, [S], seed=0).to(DEV)
    dx = torch.empty_like(w.x)
    dW = torch.empty(C, 4, device=DEV)
    dB = torch.empty(C, device=DEV)
    assert _abi_noalloc(w, "bf16", dx, dW, dB) == binding.VCD_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(vcd.VcdError, match="workspace"):
        vcd.conv1d_bwd_noalloc(w.x, w.dy, w.weight, w.cu_seqlens, w.bias, "bf16")


def test_noalloc_fp32_policy_on_a_chunked_shape():
    """The "fp32" policy at S = 65536, C = 6144: 248-token units folded seven
    to a chunk, 1824 chunk rows of the fixed scratch's 3276."""
    S, C = 65536, 6144
    w = synth.make("linattn", device=DEV, S=S, C=C)
    ref = vcd.conv1d_bwd(w.x, w.dy, w.weight, w.cu_seqlens, w.bias, "fp32",
                         dweight=torch.empty(C, 4, device=DEV), dbias=torch.empty(C, device=DEV))
    for _ in range(2):
        dx = torch.full_like(w.x, float("nan"))
        dW = torch.full((C, 4), float("nan"), device=DEV)
        dB = torch.full((C,), float("nan"), device=DEV)
        assert _abi_noalloc(w, "fp32", dx, dW, dB) == binding.VCD_OK
        torch.cuda.synchronize()
        assert torch.equal(dx, ref[0]) and torch.equal(dW, ref[1]) and torch.equal(dB, ref[2])


def test_noalloc_empty_sequence_gives_zero_gradients():
    w = synth.custom(0, 64, [0, 0], seed=0).to(DEV)
    dx = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    dW = torch.ones(64, 4, device=DEV)
    dB = torch.ones(64, device=DEV)
    assert _abi_noalloc(w, "bf16", dx, dW, dB) == binding.VCD_OK
    torch.cuda.synchronize()
    assert not dW.any() and not dB.any()


def test_noalloc_captured_after_a_first_call_replays_the_same_bits():
    """The supported order: one call outside capture on the device, then calls
    captured into a CUDA graph; every replay gives the eager call's bits."""
    w = synth.make("boundary", device=DEV, S=4096, C=1032)
    C = w.C
    eager = [torch.empty_like(w.x), torch.empty(C, 4, device=DEV), torch.empty(C, device=DEV)]
    assert _abi_noalloc(w, "bf16", *eager) == binding.VCD_OK
    torch.cuda.synchronize()
    out = [torch.zeros_like(t) for t in eager]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            assert _abi_noalloc(w, "bf16", *out) == binding.VCD_OK
    torch.cuda.synchronize()
    for _ in range(2):
        for t in out:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(eager, out):
            assert torch.equal(a, b)
