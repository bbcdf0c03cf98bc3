"""The steps of the sequence-sharded causal forward on one GPU, against the
fp64 oracle ("Efficient Transformers II" §2.2, eq (7)–(11)):

* ``forward_state`` — the state the recurrence reaches from zero, without
  outputs, equals the oracle's final state;
* ``forward_from_state`` — the causal forward continued from a given state
  equals the oracle run with that initial state (one segment per head and
  several, on every kernel family), and its final state the oracle's;
* the whole exchange: a sequence cut into shards whose aggregates are
  gathered and combined by ``shard_entering_state``, each shard then run from
  its entering state, reproduces the oracle's single forward over the whole
  sequence.  The shards run one after another on this GPU, as the ranks of
  one job would run them each on its own device.
"""
import numpy as np
import pytest
import torch

import causal_kernelized_linear_gb300 as cl
import oracle
import workloads as W
from helpers import TOL_BF16, TOL_F32, assert_parity, to_cuda

pytestmark = pytest.mark.gpu


def _inputs(B, H, n, d, dtype, fm, m, decay, seed):
    return W.make_forward_inputs(B, H, n, d, dtype, fm, m, decay, seed=seed,
                                 qk_scale=(d ** -0.25 if fm == "performer" else 1.0))


def _prefix_state(B, H, d, dtype, fm, m, decay, omega, seed, n0=333):
    """A realistic initial state: the oracle's state after a random prefix."""
    pre = W.make_forward_inputs(B, H, n0, d, dtype, fm, m, decay, seed=seed + 7,
                                qk_scale=(d ** -0.25 if fm == "performer" else 1.0))
    _, mu, nu = oracle.forward(pre["q"], pre["k"], pre["v"], pre["a"], fm, omega, True,
                               return_state=True)
    return mu, nu


# (B, H, n, d, dtype, fm, m, decay)
STATE_CASES = [
    (2, 4, 2048, 64, "bf16", "elu1", 0, (0.9, 0.999)),       # tensor cores, several segments
    (1, 2, 20000, 128, "bf16", "elu1", 0, (0.95, 0.9999)),
    (1, 160, 256, 64, "bf16", "elu1", 0, (0.5, 0.99)),       # one segment per head
    (2, 8, 4096, 64, "bf16", "performer", 256, None),        # Performer tensor cores
    (1, 3, 700, 64, "bf16", "performer", 128, (0.9, 0.99)),  # Performer with decay: CUDA cores
    (1, 3, 1000, 32, "f32", "elu1", 0, (0.3, 0.9)),          # fp32 CUDA cores
    (2, 160, 64, 32, "f32", "elu1", 0, None),                # CUDA cores, one segment per head
    (1, 2, 100, 64, "bf16", "elu1", 0, (0.9, 0.99)),         # n < 128: CUDA cores
]


def _ids(c):
    return f"B{c[0]}H{c[1]}n{c[2]}d{c[3]}{c[4]}{c[5]}{c[6] or ''}{'dec' if c[7] else ''}"


@pytest.mark.parametrize("case", STATE_CASES, ids=_ids)
def test_forward_state_is_the_final_state(cuda_device, case):
    B, H, n, d, dtype, fm, m, decay = case
    inp = _inputs(B, H, n, d, dtype, fm, m, decay, seed=n + d)
    g = to_cuda(inp, cuda_device)
    mu, nu = cl.forward_state(g["k"], g["v"], g["a"], fm, g["omega"])
    torch.cuda.synchronize()
    assert cl.last_device_status() == 0
    _, rmu, rnu = oracle.forward(inp["q"], inp["k"], inp["v"], inp["a"], fm, inp["omega"], True,
                                 return_state=True)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    assert_parity(mu, rmu, tol, "μ")
    assert_parity(nu, rnu, tol, "ν")


@pytest.mark.parametrize("case", STATE_CASES, ids=_ids)
def test_forward_from_state_continues_the_recurrence(cuda_device, case):
    B, H, n, d, dtype, fm, m, decay = case
    inp = _inputs(B, H, n, d, dtype, fm, m, decay, seed=2 * n + d)
    mu0, nu0 = _prefix_state(B, H, d, dtype, fm, m, decay, inp["omega"], seed=n)
    g = to_cuda(inp, cuda_device)
    mu0_d = torch.from_numpy(mu0).float().to(cuda_device)
    nu0_d = torch.from_numpy(nu0).float().to(cuda_device)
    out, mu, nu = cl.forward_from_state(g["q"], g["k"], g["v"], mu0_d, nu0_d, g["a"], fm,
                                        g["omega"], return_state=True)
    torch.cuda.synchronize()
    assert cl.last_device_status() == 0
    ref, rmu, rnu = oracle.forward(inp["q"], inp["k"], inp["v"], inp["a"], fm, inp["omega"], True,
                                   mu0=mu0_d.cpu(), nu0=nu0_d.cpu(), return_state=True)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    assert_parity(out, ref, tol, "o")
    assert_parity(mu, rmu, tol, "μ")
    assert_parity(nu, rnu, tol, "ν")


def test_forward_from_state_of_an_empty_sequence_returns_the_initial_state(cuda_device):
    q = torch.zeros(1, 2, 0, 64, device=cuda_device, dtype=torch.bfloat16)
    mu0 = torch.rand(1, 2, 64, 64, device=cuda_device)
    nu0 = torch.rand(1, 2, 64, device=cuda_device)
    out, mu, nu = cl.forward_from_state(q, q, q, mu0, nu0, return_state=True)
    torch.cuda.synchronize()
    assert out.numel() == 0
    assert torch.equal(mu, mu0) and torch.equal(nu, nu0)


def test_zero_initial_state_is_la_forward(cuda_device):
    inp = _inputs(1, 4, 3000, 128, "bf16", "elu1", 0, (0.9, 0.999), seed=9)
    g = to_cuda(inp, cuda_device)
    ref = cl.forward(g["q"], g["k"], g["v"], g["a"])
    zmu = torch.zeros(1, 4, 128, 128, device=cuda_device)
    znu = torch.zeros(1, 4, 128, device=cuda_device)
    out = cl.forward_from_state(g["q"], g["k"], g["v"], zmu, znu, g["a"])
    torch.cuda.synchronize()
    # the same kernels and plan: an initial state of zeros changes nothing
    assert torch.equal(out, ref)


# (B, H, d, dtype, fm, m, decay, shard lengths)
SHARD_CASES = [
    (1, 4, 128, "bf16", "elu1", 0, (0.95, 0.9999), [7000, 5000, 8000]),
    (2, 8, 64, "bf16", "performer", 256, None, [2048, 2048]),
    (1, 3, 32, "f32", "elu1", 0, (0.5, 0.99), [0, 300, 17, 400]),
    (1, 2, 64, "bf16", "performer", 128, (0.9, 0.99), [100, 600, 300]),
]


@pytest.mark.parametrize("case", SHARD_CASES,
                         ids=lambda c: f"d{c[2]}{c[3]}{c[4]}{c[5] or ''}-{len(c[7])}shards")
def test_sharded_sequence_equals_one_forward(cuda_device, case):
    B, H, d, dtype, fm, m, decay, lens = case
    n = sum(lens)
    inp = _inputs(B, H, n, d, dtype, fm, m, decay, seed=n + 5)
    g = to_cuda(inp, cuda_device)
    dp = d if fm == "elu1" else m
    cuts = np.concatenate([[0], np.cumsum(lens)])
    shard = lambda t, r: t[:, :, cuts[r]:cuts[r + 1]].contiguous()  # noqa: E731
    # every rank's aggregate, gathered as the all-gather would lay them out
    rows = []
    for r in range(len(lens)):
        mu, nu = cl.forward_state(shard(g["k"], r), shard(g["v"], r), g["a"], fm, g["omega"])
        rows.append(torch.cat([mu.reshape(-1), nu.reshape(-1)]))
    gathered = torch.stack(rows)
    outs = []
    for r in range(len(lens)):
        mu_in, nu_in = cl.shard_entering_state(gathered, r, lens, B, H, dp, d, g["a"])
        out, mu, nu = cl.forward_from_state(shard(g["q"], r), shard(g["k"], r), shard(g["v"], r),
                                            mu_in, nu_in, g["a"], fm, g["omega"],
                                            return_state=True)
        outs.append(out)
    torch.cuda.synchronize()
    assert cl.last_device_status() == 0
    ref, rmu, rnu = oracle.forward(inp["q"], inp["k"], inp["v"], inp["a"], fm, inp["omega"], True,
                                   return_state=True)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    assert_parity(torch.cat(outs, dim=2), ref, tol, "o over all shards")
    assert_parity(mu, rmu, tol, "final μ (last shard)")
    assert_parity(nu, rnu, tol, "final ν (last shard)")


def test_entering_state_of_the_first_shard_is_zero(cuda_device):
    gathered = torch.rand(3, 2 * (8 * 8 + 8), device=cuda_device)
    mu, nu = cl.shard_entering_state(gathered, 0, [5, 6, 7], 1, 2, 8, 8)
    torch.cuda.synchronize()
    assert not mu.any() and not nu.any()
