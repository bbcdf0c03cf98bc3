"""GPU parity: the CUDA library (through the C ABI) against the fp64 oracle on
the same seeded inputs.  Error metric: max|Δ| / max|ref| per (b, h) head;
bars 1e-4 for fp32 inputs and 2e-2 for bf16 inputs with fp32 state."""
import numpy as np
import pytest
import torch

import causal_kernelized_linear_gb300 as cl
import oracle
import workloads as W
from helpers import TOL_BF16, TOL_F32, assert_parity, head_rel_err, to_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    cl.build()
    cl.load()


def _run(inp, fm, causal, device):
    g = to_cuda(inp, device)
    out = cl.forward(g["q"], g["k"], g["v"], g["a"], fm, g["omega"], causal)
    torch.cuda.synchronize()
    return out


def _ref(inp, fm, causal):
    return oracle.forward(inp["q"], inp["k"], inp["v"], inp["a"], fm, inp["omega"], causal)


# --- the five workloads at full size ----------------------------------------------------

@pytest.mark.parametrize("causal", [True, False])
def test_tiny_fp32_workload(cuda_device, causal):
    w = W.TINY_FP32
    inp = W.forward_inputs(w)
    out = _run(inp, "elu1", causal, cuda_device)
    assert out.dtype == torch.float32
    assert_parity(out, _ref(inp, "elu1", causal), TOL_F32, f"{w.name} causal={causal}")


def test_elu1_decay_workload(cuda_device):
    w = W.ELU1_DECAY
    inp = W.forward_inputs(w)
    out = _run(inp, "elu1", True, cuda_device)
    assert_parity(out, _ref(inp, "elu1", True), TOL_BF16, w.name)


@pytest.mark.parametrize("causal", [False, True])
def test_performer_workload(cuda_device, causal):
    w = W.PERFORMER
    inp = W.forward_inputs(w)
    out = _run(inp, "performer", causal, cuda_device)
    assert_parity(out, _ref(inp, "performer", causal), TOL_BF16, f"{w.name} causal={causal}")


def test_long_workload(cuda_device):
    w = W.LONG
    inp = W.forward_inputs(w)
    out = _run(inp, "elu1", True, cuda_device)
    # every head, every token: the oracle runs one head per core
    assert_parity(out, _ref(inp, "elu1", True), TOL_BF16, w.name)


def test_decode_workload_sampled_heads(cuda_device):
    """Full-size decode (B=256, H=32, d=128): 512-token prefill through
    la_forward_with_state, then 1024 steps of la_decode_step.  The oracle
    follows 64 seeded-random heads through the prefill and every step."""
    w = W.DECODE
    pre = W.decode_prefill_inputs(w)
    g = to_cuda(pre, cuda_device)
    _, mu, nu = cl.forward_with_state(g["q"], g["k"], g["v"], g["a"], "elu1")
    BH = w.B * w.H
    pick = np.sort(np.random.default_rng(123).choice(BH, size=64, replace=False))
    pick_t = torch.from_numpy(pick)
    hsel = pick % w.H

    def sub(x):  # [B,H,...] -> [1, 64, ...]
        return x.reshape(BH, *x.shape[2:])[pick_t].unsqueeze(0)

    a_sub = pre["a"][torch.from_numpy(hsel)]
    _, ref_mu, ref_nu = oracle.forward(sub(pre["q"]), sub(pre["k"]), sub(pre["v"]), a_sub, "elu1",
                                       return_state=True)
    assert_parity(sub(mu.cpu()), ref_mu, TOL_BF16, "prefill state mu")
    assert_parity(sub(nu.cpu()).unsqueeze(-1), ref_nu[..., None], TOL_BF16, "prefill state nu")
    worst = 0.0
    out = torch.empty(w.B, w.H, w.d, device=cuda_device, dtype=torch.bfloat16)
    for step in range(w.steps):
        st = W.decode_step_inputs(w, step)
        gs = to_cuda(st, cuda_device)
        cl.decode_step(mu, nu, gs["q"], gs["k"], gs["v"], g["a"], out=out)
        ref_o, ref_mu, ref_nu = oracle.decode_step(ref_mu, ref_nu, sub(st["q"]), sub(st["k"]),
                                                   sub(st["v"]), a_sub)
        if step in (0, 1, 2, 511) or step % 64 == 63:
            worst = max(worst, assert_parity(sub(out.cpu()).unsqueeze(2), ref_o[:, :, None],
                                             TOL_BF16, f"decode step {step}"))
    torch.cuda.synchronize()
    assert_parity(sub(mu.cpu()), ref_mu, TOL_BF16, "final mu")
    assert_parity(sub(nu.cpu()).unsqueeze(-1), ref_nu[..., None], TOL_BF16, "final nu")


def test_decode_workload_all_heads_at_checked_steps(cuda_device):
    """Full-size decode, every one of the 8192 heads at steps 1, 2, 3, 512 and
    1024: before a checked step the GPU's own state is widened to fp64 and the
    oracle takes the same step from it, so the step's output and new state are
    checked for all heads (the sampled-heads test above follows the whole
    trajectory).  One step from the same state leaves only fp32 rounding in
    the new state, so its bar is the fp32 one."""
    w = W.DECODE
    pre = W.decode_prefill_inputs(w)
    g = to_cuda(pre, cuda_device)
    _, mu, nu = cl.forward_with_state(g["q"], g["k"], g["v"], g["a"], "elu1")
    out = torch.empty(w.B, w.H, w.d, device=cuda_device, dtype=torch.bfloat16)
    checked = {0, 1, 2, 511, w.steps - 1}
    for step in range(w.steps):
        st = W.decode_step_inputs(w, step)
        gs = to_cuda(st, cuda_device)
        if step in checked:
            torch.cuda.synchronize()
            mu0, nu0 = mu.cpu(), nu.cpu()
        cl.decode_step(mu, nu, gs["q"], gs["k"], gs["v"], g["a"], out=out)
        if step in checked:
            ref_o, ref_mu, ref_nu = oracle.decode_step(mu0, nu0, st["q"], st["k"], st["v"],
                                                       pre["a"])
            torch.cuda.synchronize()
            # o is stored in bf16: its rounding is the bf16 bar
            assert_parity(out.cpu(), ref_o, TOL_BF16, f"decode all heads, step {step + 1}: o")
            assert_parity(mu.cpu(), ref_mu, TOL_F32, f"decode all heads, step {step + 1}: mu")
            assert_parity(nu.cpu(), ref_nu, TOL_F32, f"decode all heads, step {step + 1}: nu")


def test_performer_decode_workload_sampled_heads(cuda_device):
    """Full-size Performer decode (B=256, H=32, d=64, m=256): 512-token prefill
    through la_forward_with_state, then all 1024 steps of la_decode_step_fm; the
    oracle follows 32 seeded-random heads through the prefill and every step."""
    w = W.PERFORMER_DECODE
    pre = W.decode_prefill_inputs(w)
    g = to_cuda(pre, cuda_device)
    _, mu, nu = cl.forward_with_state(g["q"], g["k"], g["v"], g["a"], "performer", g["omega"])
    BH = w.B * w.H
    pick = np.sort(np.random.default_rng(321).choice(BH, size=32, replace=False))
    pick_t = torch.from_numpy(pick)
    hsel = pick % w.H

    def sub(x):  # [B,H,...] -> [1, 32, ...]
        return x.reshape(BH, *x.shape[2:])[pick_t].unsqueeze(0)

    a_sub = pre["a"][torch.from_numpy(hsel)]
    _, ref_mu, ref_nu = oracle.forward(sub(pre["q"]), sub(pre["k"]), sub(pre["v"]), a_sub,
                                       "performer", pre["omega"], return_state=True)
    assert_parity(sub(mu.cpu()), ref_mu, TOL_BF16, "performer prefill state mu")
    out = torch.empty(w.B, w.H, w.d, device=cuda_device, dtype=torch.bfloat16)
    for step in range(w.steps):
        st = W.decode_step_inputs(w, step)
        gs = to_cuda(st, cuda_device)
        cl.decode_step(mu, nu, gs["q"], gs["k"], gs["v"], g["a"], out=out,
                       feature_map="performer", omega=g["omega"])
        ref_o, ref_mu, ref_nu = oracle.decode_step(ref_mu, ref_nu, sub(st["q"]), sub(st["k"]),
                                                   sub(st["v"]), a_sub, "performer", pre["omega"])
        if step in (0, 1, 2, 127, 511) or step % 64 == 63:
            assert_parity(sub(out.cpu()).unsqueeze(2), ref_o[:, :, None], TOL_BF16,
                          f"performer decode step {step}")
    torch.cuda.synchronize()
    assert_parity(sub(mu.cpu()), ref_mu, TOL_BF16, "performer final mu")
    assert_parity(sub(nu.cpu()).unsqueeze(-1), ref_nu[..., None], TOL_BF16, "performer final nu")


# --- sweeps over shapes, maps, decays, ragged lengths --------------------------------------

CASES = [
    # (dtype, d, fm, m, decay, n, causal)
    ("bf16", 32, "elu1", 0, None, 1, True),
    ("bf16", 64, "elu1", 0, (0.0, 0.0), 77, True),
    ("bf16", 64, "elu1", 0, (0.5, 0.5), 300, True),
    ("bf16", 128, "elu1", 0, (0.9, 0.999), 1000, True),
    ("bf16", 128, "elu1", 0, (1.0, 1.0), 513, True),
    ("bf16", 32, "elu1", 0, None, 4099, True),
    ("bf16", 64, "elu1", 0, None, 1234, False),
    ("bf16", 64, "performer", 64, None, 333, True),
    ("bf16", 64, "performer", 128, (0.95, 0.99), 700, True),
    ("bf16", 32, "performer", 256, None, 259, False),
    ("bf16", 128, "performer", 256, (0.9, 0.99), 200, True),
    # tensor-core path (bf16, elu+1, causal, d ∈ {64, 128}, n ≥ 128)
    ("bf16", 64, "elu1", 0, (0.0, 0.0), 300, True),
    ("bf16", 128, "elu1", 0, (0.5, 0.9), 128, True),
    ("bf16", 128, "elu1", 0, (0.99, 0.9999), 129, True),
    ("bf16", 64, "elu1", 0, None, 20000, True),
    ("bf16", 128, "elu1", 0, (0.3, 0.7), 4097, True),
    ("bf16", 64, "elu1", 0, (1.0, 1.0), 2560, True),
    # tensor-core Performer path (bf16, d = 64, m ∈ {128, 256}, no decay, n ≥ 128):
    # one chunk, ragged tails, one and many segments, both modes
    ("bf16", 64, "performer", 256, None, 128, True),
    ("bf16", 64, "performer", 256, None, 129, False),
    ("bf16", 64, "performer", 256, None, 1000, True),
    ("bf16", 64, "performer", 128, None, 4097, True),
    ("bf16", 64, "performer", 128, None, 300, False),
    ("bf16", 64, "performer", 256, None, 6000, False),
    # tensor-core non-causal elu+1 (bf16, d ∈ {64, 128}, n ≥ 128): state-only
    # launch over all segments, the scan's total, the tensor-core readout
    ("bf16", 64, "elu1", 0, None, 128, False),
    ("bf16", 128, "elu1", 0, None, 129, False),
    ("bf16", 128, "elu1", 0, None, 1000, False),
    ("bf16", 64, "elu1", 0, None, 4097, False),
    ("bf16", 128, "elu1", 0, None, 20000, False),
    ("f32", 32, "elu1", 0, (0.9, 0.999), 1111, True),
    ("f32", 64, "elu1", 0, None, 517, False),
    ("f32", 128, "elu1", 0, (0.0, 1.0), 129, True),
    ("f32", 64, "performer", 128, None, 130, True),
    ("f32", 32, "performer", 64, None, 70, False),
]


def test_noncausal_elu1_many_heads_one_segment(cuda_device):
    # 160 heads: one segment per head, the readout's CTA count set by the heads
    for d in (64, 128):
        inp = W.make_forward_inputs(2, 80, 700, d, "bf16", "elu1", 0, None, seed=d + 1)
        out = _run(inp, "elu1", False, cuda_device)
        assert_parity(out, _ref(inp, "elu1", False), TOL_BF16, f"non-causal d={d}, 160 heads")


def test_noncausal_elu1_exports_the_totals(cuda_device):
    inp = W.make_forward_inputs(1, 4, 3000, 128, "bf16", "elu1", 0, None, seed=31)
    g = to_cuda(inp, cuda_device)
    out, mu, nu = cl.forward_with_state(g["q"], g["k"], g["v"], None, "elu1", None, False)
    torch.cuda.synchronize()
    ref, rmu, rnu = oracle.forward(inp["q"], inp["k"], inp["v"], None, "elu1", None, False,
                                   return_state=True)
    assert_parity(out, ref, TOL_BF16, "non-causal o")
    assert_parity(mu, rmu, TOL_BF16, "non-causal μ_n")
    assert_parity(nu, rnu, TOL_BF16, "non-causal ν_n")


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(str(x) for x in c))
def test_sweep(cuda_device, case):
    dtype, d, fm, m, decay, n, causal = case
    inp = W.make_forward_inputs(2, 3, n, d, dtype, fm, m, decay, seed=n * 7 + d,
                                qk_scale=(d ** -0.25 if fm == "performer" else 1.0))
    out = _run(inp, fm, causal, cuda_device)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    assert_parity(out, _ref(inp, fm, causal), tol, str(case))


def test_many_heads_short_sequences(cuda_device):
    inp = W.make_forward_inputs(64, 8, 40, 64, "bf16", "elu1", decay=(0.8, 0.99), seed=5)
    out = _run(inp, "elu1", True, cuda_device)
    assert_parity(out, _ref(inp, "elu1", True), TOL_BF16, "B64 H8 n40")


# --- state export and hand-off ------------------------------------------------------------

@pytest.mark.parametrize("dtype,n", [("bf16", 3000), ("f32", 700), ("bf16", 64)])
def test_forward_with_state_matches_oracle_state(cuda_device, dtype, n):
    inp = W.make_forward_inputs(2, 2, n, 64, dtype, "elu1", decay=(0.9, 0.999), seed=11)
    g = to_cuda(inp, cuda_device)
    out, mu, nu = cl.forward_with_state(g["q"], g["k"], g["v"], g["a"], "elu1")
    ref_o, ref_mu, ref_nu = oracle.forward(inp["q"], inp["k"], inp["v"], inp["a"], "elu1",
                                           return_state=True)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    assert_parity(out, ref_o, tol, "out")
    assert_parity(mu, ref_mu, tol, "mu")
    assert_parity(nu.unsqueeze(-1), ref_nu[..., None], tol, "nu")


@pytest.mark.parametrize("causal,n", [(True, 3000), (False, 3000), (True, 200)])
def test_performer_state_matches_oracle_state(cuda_device, causal, n):
    inp = W.make_forward_inputs(2, 2, n, 64, "bf16", "performer", 256, seed=13,
                                qk_scale=64 ** -0.25)
    g = to_cuda(inp, cuda_device)
    out, mu, nu = cl.forward_with_state(g["q"], g["k"], g["v"], None, "performer", g["omega"],
                                        causal=causal)
    ref_o, ref_mu, ref_nu = oracle.forward(inp["q"], inp["k"], inp["v"], None, "performer",
                                           inp["omega"], causal=causal, return_state=True)
    assert_parity(out, ref_o, TOL_BF16, "out")
    assert_parity(mu, ref_mu, TOL_BF16, "mu")
    assert_parity(nu.unsqueeze(-1), ref_nu[..., None], TOL_BF16, "nu")


def test_noncausal_state_is_full_sum(cuda_device):
    inp = W.make_forward_inputs(1, 2, 2000, 64, "bf16", "elu1", seed=12)
    g = to_cuda(inp, cuda_device)
    _, mu, nu = cl.forward_with_state(g["q"], g["k"], g["v"], None, "elu1", causal=False)
    _, ref_mu, ref_nu = oracle.forward(inp["q"], inp["k"], inp["v"], None, "elu1", causal=False,
                                       return_state=True)
    assert_parity(mu, ref_mu, TOL_BF16, "mu")


def test_prefill_then_decode_equals_forward(cuda_device):
    n1, n2 = 300, 20
    inp = W.make_forward_inputs(2, 4, n1 + n2, 128, "bf16", "elu1", decay=(0.9, 0.99), seed=13)
    g = to_cuda(inp, cuda_device)
    full = cl.forward(g["q"], g["k"], g["v"], g["a"], "elu1")
    _, mu, nu = cl.forward_with_state(g["q"][:, :, :n1].contiguous(), g["k"][:, :, :n1].contiguous(),
                                      g["v"][:, :, :n1].contiguous(), g["a"], "elu1")
    ref = oracle.forward(inp["q"], inp["k"], inp["v"], inp["a"], "elu1")
    for j in range(n1, n1 + n2):
        o = cl.decode_step(mu, nu, g["q"][:, :, j].contiguous(), g["k"][:, :, j].contiguous(),
                           g["v"][:, :, j].contiguous(), g["a"])
        assert_parity(o.unsqueeze(2), ref[:, :, j:j + 1], TOL_BF16, f"decode token {j}")
        assert_parity(o.unsqueeze(2), full[:, :, j:j + 1].float(), TOL_BF16, f"vs forward {j}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_small_against_oracle(cuda_device, dtype):
    for d in (32, 64, 128):
        r = torch.Generator().manual_seed(d)
        B, H = 3, 5
        mu = torch.rand(B, H, d, d, generator=r)
        nu = torch.rand(B, H, d, generator=r) + 0.5
        a = torch.rand(H, generator=r)
        a[0] = 1.0
        a[1] = 0.0
        dt = W.torch_dtype(dtype)
        q, k, v = (torch.randn(B, H, d, generator=r).to(dt) for _ in range(3))
        ref_o, ref_mu, ref_nu = oracle.decode_step(mu, nu, q, k, v, a)
        mu_g, nu_g = mu.to(cuda_device), nu.to(cuda_device)
        o = cl.decode_step(mu_g, nu_g, q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                           a.to(cuda_device))
        tol = TOL_F32 if dtype == "f32" else TOL_BF16
        assert_parity(o.unsqueeze(2), ref_o[:, :, None], tol, f"decode out d={d}")
        assert_parity(mu_g, ref_mu, TOL_F32, f"decode mu d={d}")
        assert_parity(nu_g.unsqueeze(-1), ref_nu[..., None], TOL_F32, f"decode nu d={d}")


# --- edge cases and error behaviour --------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d,m", [(32, 64), (32, 256), (64, 128), (64, 256), (128, 64), (128, 256)])
def test_performer_decode_small_against_oracle(cuda_device, dtype, d, m):
    B, H, steps = 3, 4, 5
    inp = W.make_forward_inputs(B, H, 7, d, dtype, "performer", m, decay=(0.7, 0.99),
                                seed=31 + d + m, qk_scale=d ** -0.25)
    g = to_cuda(inp, cuda_device)
    _, mu, nu = cl.forward_with_state(g["q"], g["k"], g["v"], g["a"], "performer", g["omega"])
    _, ref_mu, ref_nu = oracle.forward(inp["q"], inp["k"], inp["v"], inp["a"], "performer",
                                       inp["omega"], return_state=True)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    gen = torch.Generator().manual_seed(77 + d)
    for s in range(steps):
        q, k, v = (torch.randn(B, H, d, generator=gen) for _ in range(3))
        q, k = q * d ** -0.25, k * d ** -0.25
        q, k, v = (x.to(W.torch_dtype(dtype)) for x in (q, k, v))
        o = cl.decode_step(mu, nu, q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                           g["a"], feature_map="performer", omega=g["omega"])
        ref_o, ref_mu, ref_nu = oracle.decode_step(ref_mu, ref_nu, q, k, v, inp["a"],
                                                   "performer", inp["omega"])
        assert_parity(o.unsqueeze(2), ref_o[:, :, None], tol, f"step {s}")
    assert_parity(mu, ref_mu, tol, "mu")
    assert_parity(nu.unsqueeze(-1), ref_nu[..., None], tol, "nu")


def test_performer_prefill_then_decode_equals_forward(cuda_device):
    # forward over n1 tokens with the state, then decode steps, against the
    # forward over all n1 + n2 tokens (tensor-core prefill: no decay)
    n1, n2 = 300, 12
    inp = W.make_forward_inputs(1, 4, n1 + n2, 64, "bf16", "performer", 256, seed=41,
                                qk_scale=64 ** -0.25)
    g = to_cuda(inp, cuda_device)
    full = cl.forward(g["q"], g["k"], g["v"], None, "performer", g["omega"], True)
    _, mu, nu = cl.forward_with_state(g["q"][:, :, :n1].contiguous(), g["k"][:, :, :n1].contiguous(),
                                      g["v"][:, :, :n1].contiguous(), None, "performer", g["omega"])
    outs = []
    for j in range(n1, n1 + n2):
        o = cl.decode_step(mu, nu, g["q"][:, :, j].contiguous(), g["k"][:, :, j].contiguous(),
                           g["v"][:, :, j].contiguous(), None, feature_map="performer",
                           omega=g["omega"])
        outs.append(o.unsqueeze(2))
    dec = torch.cat(outs, dim=2)
    ref = oracle.forward(inp["q"], inp["k"], inp["v"], None, "performer", inp["omega"], True)
    assert_parity(dec, ref[:, :, n1:], TOL_BF16, "decoded tail vs oracle")
    assert_parity(full[:, :, n1:], ref[:, :, n1:], TOL_BF16, "forward tail vs oracle")


def test_empty_sequence_is_a_noop(cuda_device):
    q = torch.empty(2, 3, 0, 64, device=cuda_device, dtype=torch.bfloat16)
    out = cl.forward(q, q, q)
    assert out.shape == q.shape
    _, mu, nu = cl.forward_with_state(q, q, q)
    assert float(mu.abs().max()) == 0.0 and float(nu.abs().max()) == 0.0


def test_invalid_call_queues_nothing(cuda_device):
    q = torch.randn(1, 2, 16, 64, device=cuda_device).bfloat16()
    out = torch.full_like(q, 7.0)
    a = torch.full((2,), 0.5, device=cuda_device)
    with pytest.raises(cl.LinAttnError) as e:
        cl.forward(q, q, q, a, "elu1", None, causal=False, out=out)
    assert e.value.status_name == "LA_ERR_UNSUPPORTED"
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    assert cl.last_device_status() == 0


def test_outputs_are_finite_and_convex(cuda_device):
    # property at any size: each o_j is a convex combination of v_1..v_j
    inp = W.make_forward_inputs(1, 4, 5000, 64, "bf16", "elu1", decay=(0.9, 0.9999), seed=21)
    out = _run(inp, "elu1", True, cuda_device).float().cpu()
    v = inp["v"].float()
    lo = torch.cummin(v, dim=2).values
    hi = torch.cummax(v, dim=2).values
    slack = 0.02 * float(v.abs().max())
    assert torch.isfinite(out).all()
    assert bool((out >= lo - slack).all()) and bool((out <= hi + slack).all())
