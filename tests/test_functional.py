"""The torch API with the pages' names: contracts (CPU) and behaviour (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import varlen_causal_depthwise_gb300 as vcd
from varlen_causal_depthwise_gb300 import synth
from _check import bf16_close, rel_l2

F = vcd.cake_causal_conv1d_train_forward
B = vcd.cake_causal_conv1d_train_backward


def _cpu_case():
    x = torch.zeros(16, 8, dtype=torch.bfloat16)
    return x, torch.zeros(8, 4), torch.tensor([0, 16], dtype=torch.int32)


@pytest.mark.parametrize("mutate,exc", [
    (lambda x, w, cu: (x.float(), w, cu), TypeError),                   # x not BF16
    (lambda x, w, cu: (x, torch.zeros(8, 3), cu), ValueError),          # width 3 rejected
    (lambda x, w, cu: (x, torch.zeros(8, 5), cu), ValueError),          # width 5 rejected
    (lambda x, w, cu: (x[:, :4].contiguous(), w[:4], cu), ValueError),  # C % 8 != 0
    (lambda x, w, cu: (x, w, cu.long()), ValueError),                   # cu_seqlens not int32
])
def test_forward_contracts_rejected_before_the_gpu(mutate, exc):
    x, w, cu = mutate(*_cpu_case())
    with pytest.raises(exc):
        F(x, w, cu)


def test_backward_needs_bias_for_dbias():
    x, w, cu = _cpu_case()
    with pytest.raises((ValueError, TypeError)):
        B(x, w, cu, x, dbias=torch.zeros(8))


@pytest.mark.gpu
def test_functional_matches_oracle_and_shapes():
    wc = synth.make("tiny", S=1024, C=64)
    w = wc.to("cuda")
    for shaped in (False, True):
        x = w.x.unsqueeze(0) if shaped else w.x
        dy = w.dy.unsqueeze(0) if shaped else w.dy
        y = F(x, w.weight, w.cu_seqlens, bias=w.bias)
        assert y.shape == x.shape and y.dtype == torch.bfloat16
        ry, ay = oracle.fwd(wc.x, wc.weight, wc.cu_seqlens, wc.bias)
        bf16_close(y.reshape(wc.S, wc.C).double().cpu().numpy(), ry, ay, "functional y")
        dx, dW, dB = B(x, w.weight, w.cu_seqlens, dy, bias=w.bias)
        assert dx.shape == x.shape and dW.dtype == w.weight.dtype and dB.dtype == w.bias.dtype
        rdx, adx, rdw, rdb = oracle.bwd(wc.x, wc.dy, wc.weight, wc.cu_seqlens, wc.bias, "bf16")
        bf16_close(dx.reshape(wc.S, wc.C).double().cpu().numpy(), rdx, adx, "functional dx")
        assert rel_l2(dW.double().cpu().numpy(), rdw) <= 5e-5
        assert rel_l2(dB.double().cpu().numpy(), rdb) <= 5e-5


@pytest.mark.gpu
def test_backward_without_bias_returns_two():
    w = synth.make("mid", S=512, C=64, device="cuda")
    out = B(w.x, w.weight, w.cu_seqlens, w.dy)
    assert len(out) == 2 and out[1].dtype == torch.bfloat16     # mid: BF16 weight


@pytest.mark.gpu
@pytest.mark.parametrize("policy", ["bf16", "fp32"])
def test_autograd_function(policy):
    wc = synth.make("boundary", S=700, C=40)
    w = wc.to("cuda")
    x = w.x.clone().requires_grad_(True)
    W = w.weight.clone().requires_grad_(True)
    b = w.bias.clone().requires_grad_(True)
    y = vcd.causal_conv1d(x, W, w.cu_seqlens, b, policy)
    g = torch.randn(y.shape, device="cuda", dtype=torch.float32)   # FP32 incoming gradient
    y.backward(g.t().contiguous().t())                             # non-contiguous too
    assert x.grad.dtype == torch.bfloat16 and W.grad.dtype == W.dtype and b.grad.dtype == b.dtype
    dy = g.to(torch.bfloat16)
    dx, dW, dB = B(w.x, w.weight, w.cu_seqlens, dy, bias=w.bias, silu_grad_preactivation=policy)
    assert torch.equal(x.grad, dx) and torch.equal(W.grad, dW) and torch.equal(b.grad, dB)


@pytest.mark.gpu
def test_workspace_is_reused_per_stream():
    w = synth.make("tiny", S=2048, C=128, device="cuda")
    B(w.x, w.weight, w.cu_seqlens, w.dy, bias=w.bias)
    from varlen_causal_depthwise_gb300 import functional
    key = functional._stream_key(w.x.device)
    ws = functional._BWD_WS[key]
    B(w.x, w.weight, w.cu_seqlens, w.dy, bias=w.bias)
    assert functional._BWD_WS[key] is ws


@pytest.mark.gpu
def test_two_streams_two_workspaces_run_concurrently():
    """Two backward calls on two streams with their own workspaces give the
    same gradients as one after the other (the pages' concurrency contract)."""
    w1 = synth.make("linattn", S=4096, C=1024, device="cuda")
    w2 = synth.make("linattn", S=4096, C=1024, device="cuda", seed=9)
    ref1 = B(w1.x, w1.weight, w1.cu_seqlens, w1.dy, bias=w1.bias)
    ref2 = B(w2.x, w2.weight, w2.cu_seqlens, w2.dy, bias=w2.bias)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ws1 = vcd.cake_causal_conv1d_train_backward_workspace(4096, 1024)
    ws2 = vcd.cake_causal_conv1d_train_backward_workspace(4096, 1024)
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        with torch.cuda.stream(s1):
            o1 = B(w1.x, w1.weight, w1.cu_seqlens, w1.dy, bias=w1.bias, workspace=ws1)
        with torch.cuda.stream(s2):
            o2 = B(w2.x, w2.weight, w2.cu_seqlens, w2.dy, bias=w2.bias, workspace=ws2)
    torch.cuda.synchronize()
    for a, b in zip(o1, ref1):
        assert torch.equal(a, b)
    for a, b in zip(o2, ref2):
        assert torch.equal(a, b)


@pytest.mark.gpu
def test_graph_capture_of_the_autograd_step():
    """forward + backward through the autograd wrapper, captured in a CUDA graph."""
    w = synth.make("tiny", device="cuda")
    x = w.x.clone().requires_grad_(True)
    W = w.weight.clone().requires_grad_(True)
    b = w.bias.clone().requires_grad_(True)
    g = w.dy

    def step():
        y = vcd.causal_conv1d(x, W, w.cu_seqlens, b)
        y.backward(g)
        return y

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        y0 = step()                       # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    ref = [y0.detach().clone(), x.grad.clone(), W.grad.clone(), b.grad.clone()]
    x.grad = W.grad = b.grad = None
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        yg = step()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(yg, ref[0]) and torch.equal(x.grad, ref[1])
    assert torch.equal(W.grad, ref[2]) and torch.equal(b.grad, ref[3])
