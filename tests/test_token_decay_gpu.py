"""GPU parity of the per-token decay ("Efficient Transformers II" eq (4) with a
and b indexed by the token: μ_i = a_i μ_{i−1} + b_i k'_iᵀv_i) through the C
ABI against the fp64 oracle on the same seeded inputs.  Error metric: max|Δ|
/ max|ref| per (b, h) head; bars 1e-4 for fp32 inputs and 2e-2 for bf16."""
import numpy as np
import pytest
import torch

import causal_kernelized_linear_gb300 as cl
import oracle
import workloads as W
from helpers import TOL_BF16, TOL_F32, assert_parity, to_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    cl.build()
    cl.load()


def _inputs(B, H, n, d, dtype, fm="elu1", m=0, seed=0, weight=True, resets=0.0,
            rate=(1.0, 16.0)):
    x = W.make_forward_inputs(B, H, n, d, dtype, fm, m, None, seed=seed,
                              qk_scale=(d ** -0.25 if fm == "performer" else 1.0))
    a, b = W.make_token_decay(B, H, n, seed, rate=rate, weight=weight, resets=resets)
    x["a_tok"], x["b_tok"] = a, b
    return x


def _run(x, fm, device, state=False):
    g = to_cuda(x, device)
    r = cl.forward_token_decay(g["q"], g["k"], g["v"], g["a_tok"], g["b_tok"], fm, g["omega"],
                               return_state=state)
    torch.cuda.synchronize()
    return r


def _ref(x, fm, state=False):
    return oracle.forward_token_decay(x["q"], x["k"], x["v"], x["a_tok"], x["b_tok"], fm,
                                      x["omega"], return_state=state)


# (dtype, d, feature map, m, n, with weight, reset fraction): one chunk, ragged
# tails, one and many segments, both maps, both weights, resets
CASES = [
    ("f32", 32, "elu1", 0, 257, True, 0.0),
    ("f32", 64, "elu1", 0, 1000, False, 0.0),
    ("f32", 128, "elu1", 0, 129, True, 0.01),
    ("f32", 32, "performer", 64, 300, True, 0.0),
    ("f32", 64, "performer", 128, 97, False, 0.0),
    ("bf16", 32, "elu1", 0, 33, True, 0.0),
    ("bf16", 64, "elu1", 0, 128, True, 0.0),
    ("bf16", 64, "elu1", 0, 300, False, 0.0),
    ("bf16", 64, "elu1", 0, 4097, True, 0.002),
    ("bf16", 128, "elu1", 0, 129, True, 0.0),
    ("bf16", 128, "elu1", 0, 2560, False, 0.0),
    ("bf16", 128, "elu1", 0, 9000, True, 0.0),
    ("bf16", 64, "performer", 256, 700, True, 0.0),
    ("bf16", 128, "performer", 64, 150, False, 0.0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(str(x) for x in c))
def test_token_decay_sweep(cuda_device, case):
    dtype, d, fm, m, n, weight, resets = case
    x = _inputs(2, 3, n, d, dtype, fm, m, seed=n * 5 + d, weight=weight, resets=resets)
    out = _run(x, fm, cuda_device)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    assert_parity(out, _ref(x, fm), tol, str(case))


@pytest.mark.parametrize("dtype,n,d", [("bf16", 3000, 64), ("bf16", 1500, 128), ("f32", 700, 64),
                                       ("bf16", 100, 64)])
def test_token_decay_state_matches_oracle_state(cuda_device, dtype, n, d):
    x = _inputs(2, 2, n, d, dtype, seed=41 + n)
    out, mu, nu = _run(x, "elu1", cuda_device, state=True)
    ro, rmu, rnu = _ref(x, "elu1", state=True)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    assert_parity(out, ro, tol, "out")
    assert_parity(mu, rmu, tol, "mu")
    assert_parity(nu.unsqueeze(-1), rnu[..., None], tol, "nu")


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("f32", 64)])
def test_constant_token_decay_equals_per_head_forward(cuda_device, dtype, d):
    # a_i = a_h for every token and b_i = 1 − a_h is the per-head decay of
    # eq (10)–(11): the two entry points agree with each other and the oracle
    B, H, n = 2, 3, 1500
    x = W.make_forward_inputs(B, H, n, d, dtype, "elu1", decay=(0.9, 0.999), seed=43)
    g = to_cuda(x, cuda_device)
    a_tok = g["a"][None, :, None].expand(B, H, n).contiguous()
    tok = cl.forward_token_decay(g["q"], g["k"], g["v"], a_tok, None, "elu1")
    head = cl.forward(g["q"], g["k"], g["v"], g["a"], "elu1")
    ref = oracle.forward(x["q"], x["k"], x["v"], x["a"], "elu1")
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    assert_parity(tok, ref, tol, "token decay")
    assert_parity(head, ref, tol, "per-head decay")


def test_zero_decay_restarts_the_sequence(cuda_device):
    # a_r = 0 at r: the outputs from r on are those of the sequence starting at r
    B, H, n, d, r0 = 1, 4, 2000, 64, 777
    x = _inputs(B, H, n, d, "bf16", seed=47)
    x["a_tok"][:, :, r0] = 0.0
    g = to_cuda(x, cuda_device)
    full = cl.forward_token_decay(g["q"], g["k"], g["v"], g["a_tok"], g["b_tok"], "elu1")
    tail = cl.forward_token_decay(g["q"][:, :, r0:].contiguous(), g["k"][:, :, r0:].contiguous(),
                                  g["v"][:, :, r0:].contiguous(),
                                  g["a_tok"][:, :, r0:].contiguous(),
                                  g["b_tok"][:, :, r0:].contiguous(), "elu1")
    ref = _ref(x, "elu1")
    assert_parity(full, ref, TOL_BF16, "full")
    assert_parity(full[:, :, r0:], tail.float(), TOL_BF16, "restart")


def test_token_decay_workload_sampled_heads(cuda_device):
    """The long shape (B=1, H=16, n=65536, d=128) with a per-token decay and
    weight, as the benchmark runs it; the oracle follows 3 seeded-random
    heads over all tokens."""
    w = W.TOKEN_DECAY_LONG
    x = W.token_decay_inputs(w)
    out = _run(x, "elu1", cuda_device).cpu()
    pick = np.sort(np.random.default_rng(321).choice(w.base.H, size=3, replace=False))
    sub = {k: (v[:, pick].contiguous() if isinstance(v, torch.Tensor) and v.dim() >= 2 else v)
           for k, v in x.items() if k != "omega"}
    ref = oracle.forward_token_decay(sub["q"], sub["k"], sub["v"], sub["a_tok"], sub["b_tok"],
                                     "elu1")
    assert_parity(out[:, pick], ref, TOL_BF16, w.name)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("fm,d,m", [("elu1", 32, 0), ("elu1", 64, 0), ("elu1", 128, 0),
                                    ("performer", 64, 256), ("performer", 128, 64)])
def test_token_decay_decode_against_oracle(cuda_device, dtype, fm, d, m):
    B, H, n1, steps = 3, 4, 200, 6
    x = _inputs(B, H, n1 + steps, d, dtype, fm, m, seed=53 + d + m)
    g = to_cuda(x, cuda_device)
    sl = lambda t, a, b: t[:, :, a:b].contiguous()
    _, mu, nu = cl.forward_token_decay(sl(g["q"], 0, n1), sl(g["k"], 0, n1), sl(g["v"], 0, n1),
                                       sl(g["a_tok"], 0, n1), sl(g["b_tok"], 0, n1), fm,
                                       g["omega"], return_state=True)
    ref = _ref(x, fm)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    for j in range(n1, n1 + steps):
        o = cl.decode_step_token_decay(mu, nu, g["q"][:, :, j].contiguous(),
                                       g["k"][:, :, j].contiguous(), g["v"][:, :, j].contiguous(),
                                       g["a_tok"][:, :, j].contiguous(),
                                       g["b_tok"][:, :, j].contiguous(),
                                       feature_map=fm, omega=g["omega"])
        assert_parity(o.unsqueeze(2), ref[:, :, j:j + 1], tol, f"decode token {j}")


def test_token_decay_decode_default_weight(cuda_device):
    # b = None means b = 1 − a at the step as well
    B, H, d = 4, 2, 64
    x = _inputs(B, H, 1, d, "f32", seed=59, weight=False)
    r = torch.Generator().manual_seed(3)
    mu0 = torch.rand(B, H, d, d, generator=r)
    nu0 = torch.rand(B, H, d, generator=r) + 0.5
    g = to_cuda(x, cuda_device)
    mu, nu = mu0.to(cuda_device), nu0.to(cuda_device)
    o = cl.decode_step_token_decay(mu, nu, g["q"][:, :, 0].contiguous(), g["k"][:, :, 0].contiguous(),
                                   g["v"][:, :, 0].contiguous(), g["a_tok"][:, :, 0].contiguous())
    ro, rmu, rnu = oracle.decode_step_token_decay(mu0, nu0, x["q"][:, :, 0], x["k"][:, :, 0],
                                                  x["v"][:, :, 0], x["a_tok"][:, :, 0])
    assert_parity(o.unsqueeze(2), ro[:, :, None], TOL_F32, "out")
    assert_parity(mu, rmu, TOL_F32, "mu")


def test_token_decay_empty_sequence(cuda_device):
    q = torch.empty(1, 2, 0, 64, device=cuda_device, dtype=torch.bfloat16)
    a = torch.empty(1, 2, 0, device=cuda_device)
    out, mu, nu = cl.forward_token_decay(q, q, q, a, None, return_state=True)
    torch.cuda.synchronize()
    assert out.shape == q.shape
    assert float(mu.abs().sum()) == 0.0 and float(nu.abs().sum()) == 0.0
