"""The library inside CUDA graphs and on concurrent streams: la_forward (with
its stream-ordered workspace and programmatically dependent launches) and
la_decode_step captured into graphs and replayed, and two forwards running
at once on two streams, all against the fp64 oracle."""
import pytest
import torch

import causal_kernelized_linear_gb300 as cl
import oracle
import workloads as W
from causal_kernelized_linear_gb300 import _binding as B
from helpers import TOL_BF16, assert_parity, to_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    cl.build()
    cl.load()


@pytest.mark.parametrize("fm,m,decay,n", [("elu1", 0, (0.9, 0.999), 3000),
                                          ("performer", 256, None, 3000)])
def test_forward_graph_capture_and_replay(cuda_device, fm, m, decay, n):
    inp = W.make_forward_inputs(2, 4, n, 64, "bf16", fm, m, decay=decay, seed=51,
                                qk_scale=(64 ** -0.25 if fm == "performer" else 1.0))
    g = to_cuda(inp, cuda_device)
    out = torch.empty_like(g["q"])
    torch.cuda.synchronize()                         # inputs were copied on the default stream
    s = torch.cuda.Stream()
    cl.forward(g["q"], g["k"], g["v"], g["a"], fm, g["omega"], True, out=out, stream=s)  # warm-up
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        cl.forward(g["q"], g["k"], g["v"], g["a"], fm, g["omega"], True, out=out, stream=s)
    ref = oracle.forward(inp["q"], inp["k"], inp["v"], inp["a"], fm, inp["omega"], True)
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert_parity(out, ref, TOL_BF16, f"{fm} graph replay")
    # new inputs copied into the captured buffers are picked up by a replay
    inp2 = W.make_forward_inputs(2, 4, n, 64, "bf16", fm, m, decay=decay, seed=52,
                                 qk_scale=(64 ** -0.25 if fm == "performer" else 1.0))
    for key in ("q", "k", "v"):
        g[key].copy_(inp2[key].to(cuda_device))
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    ref2 = oracle.forward(inp2["q"], inp2["k"], inp2["v"], inp["a"], fm, inp["omega"], True)
    assert_parity(out, ref2, TOL_BF16, f"{fm} graph replay, new inputs")
    assert cl.last_device_status() == B.LA_OK


def test_decode_steps_in_one_graph(cuda_device):
    B_, H, d, steps = 4, 8, 128, 8
    pre = W.make_forward_inputs(B_, H, 50, d, "bf16", "elu1", decay=(0.9, 0.99), seed=53)
    g = to_cuda(pre, cuda_device)
    _, mu, nu = cl.forward_with_state(g["q"], g["k"], g["v"], g["a"], "elu1")
    torch.cuda.synchronize()
    _, ref_mu, ref_nu = oracle.forward(pre["q"], pre["k"], pre["v"], pre["a"], "elu1",
                                       return_state=True)
    gen = torch.Generator().manual_seed(54)
    xs = [[torch.randn(B_, H, d, generator=gen).bfloat16() for _ in range(3)] for _ in range(steps)]
    dx = [[t.to(cuda_device) for t in x] for x in xs]
    outs = [torch.empty(B_, H, d, device=cuda_device, dtype=torch.bfloat16) for _ in range(steps)]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for i in range(steps):
            cl.decode_step(mu, nu, dx[i][0], dx[i][1], dx[i][2], g["a"], out=outs[i], stream=s)
    graph.replay()                                   # capture queued nothing: one pass of 8 steps
    torch.cuda.synchronize()
    for i in range(steps):
        ref_o, ref_mu, ref_nu = oracle.decode_step(ref_mu, ref_nu, xs[i][0], xs[i][1], xs[i][2],
                                                   pre["a"])
        assert_parity(outs[i].unsqueeze(2), ref_o[:, :, None], TOL_BF16, f"graph step {i}")
    assert_parity(mu, ref_mu, TOL_BF16, "mu after the graph")


def test_two_streams_concurrently(cuda_device):
    a = W.make_forward_inputs(1, 8, 4096, 128, "bf16", "elu1", decay=(0.95, 0.999), seed=55)
    b = W.make_forward_inputs(2, 4, 2000, 64, "bf16", "performer", 256, seed=56,
                              qk_scale=64 ** -0.25)
    ga, gb = to_cuda(a, cuda_device), to_cuda(b, cuda_device)
    oa, ob = torch.empty_like(ga["q"]), torch.empty_like(gb["q"])
    torch.cuda.synchronize()                         # inputs were copied on the default stream
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        cl.forward(ga["q"], ga["k"], ga["v"], ga["a"], "elu1", None, True, out=oa, stream=s1)
        cl.forward(gb["q"], gb["k"], gb["v"], None, "performer", gb["omega"], False, out=ob,
                   stream=s2)
    torch.cuda.synchronize()
    assert_parity(oa, oracle.forward(a["q"], a["k"], a["v"], a["a"], "elu1", None, True),
                  TOL_BF16, "stream 1")
    assert_parity(ob, oracle.forward(b["q"], b["k"], b["v"], None, "performer", b["omega"], False),
                  TOL_BF16, "stream 2")


def test_token_decay_forward_and_backward_in_graphs(cuda_device):
    """la_forward_token_decay and la_backward, each captured into a graph
    (stream-ordered workspace inside the capture) and replayed."""
    n = 3000
    x = W.make_forward_inputs(2, 4, n, 64, "bf16", "elu1", decay=(0.9, 0.999), seed=57)
    a_tok, b_tok = W.make_token_decay(2, 4, n, seed=57)
    gen = torch.Generator().manual_seed(58)
    go = torch.randn(2, 4, n, 64, generator=gen).bfloat16()
    g = to_cuda(x, cuda_device)
    at, bt, god = a_tok.to(cuda_device), b_tok.to(cuda_device), go.to(cuda_device)
    out = torch.empty_like(g["q"])
    dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    # warm-up outside the capture
    cl.forward_token_decay(g["q"], g["k"], g["v"], at, bt, out=out, stream=s)
    cl.backward(g["q"], g["k"], g["v"], god, g["a"], dq=dq, dk=dk, dv=dv, want_da=False, stream=s)
    s.synchronize()
    g1, g2 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1, stream=s):
        cl.forward_token_decay(g["q"], g["k"], g["v"], at, bt, out=out, stream=s)
    with torch.cuda.graph(g2, stream=s):
        cl.backward(g["q"], g["k"], g["v"], god, g["a"], dq=dq, dk=dk, dv=dv, want_da=False,
                    stream=s)
    ref = oracle.forward_token_decay(x["q"], x["k"], x["v"], a_tok, b_tok, "elu1")
    rq, rk, rv, _ = oracle.backward(x["q"], x["k"], x["v"], go, x["a"], "elu1")
    for _ in range(2):
        out.zero_()
        dq.zero_()
        g1.replay()
        g2.replay()
        torch.cuda.synchronize()
        assert_parity(out, ref, TOL_BF16, "token decay graph replay")
        assert_parity(dq, rq, TOL_BF16, "backward graph replay dq")
        assert_parity(dk, rk, TOL_BF16, "backward graph replay dk")
        assert_parity(dv, rv, TOL_BF16, "backward graph replay dv")
    assert cl.last_device_status() == B.LA_OK
