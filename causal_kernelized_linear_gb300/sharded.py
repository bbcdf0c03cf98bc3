"""Causal forward of a sequence split across processes, one device each.

Every head's sequence is cut into consecutive shards, shard r held by rank r
of a ``torch.distributed`` group.  Eq (10)–(11) of "Efficient Transformers
II" §2.2, unrolled over a shard of L_j tokens, says what crosses a shard
boundary: only the state.  So the split needs one exchange step:

1. every rank computes its shard's aggregate A_r, the state (μ, ν) its
   tokens reach from zero (``la_forward_state``);
2. the ranks all-gather the aggregates and the shard lengths (one collective
   for each);
3. rank r forms the state entering its shard,
   S_in(r) = Σ_{j<r} a^{L_{j+1} + … + L_{r−1}}·A_j (``la_shard_entering_state``),
   and runs its shard from it (``la_forward_from_state``).

Its outputs are then those of one forward over the whole sequence, and the
last rank's final state is the sequence's.  Arithmetic runs in the library's
kernels; this module only moves tensors between ranks.  Heads stay
independent, so splitting the heads across devices (no exchange at all)
remains the simpler choice whenever there are enough of them.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import _binding


class CudaOps:
    """The per-rank steps, on this process's CUDA device (the library)."""

    @staticmethod
    def forward_state(k, v, decay_a, feature_map, omega, mu_out, nu_out):
        _binding.forward_state(k, v, decay_a, feature_map, omega, mu_out=mu_out, nu_out=nu_out)

    @staticmethod
    def shard_entering_state(gathered, rank, shard_len, B, H, dp, d, decay_a):
        return _binding.shard_entering_state(gathered, rank, shard_len, B, H, dp, d, decay_a)

    @staticmethod
    def forward_from_state(q, k, v, mu0, nu0, decay_a, feature_map, omega, return_state):
        return _binding.forward_from_state(q, k, v, mu0, nu0, decay_a, feature_map, omega,
                                           return_state=return_state)


def forward_sequence_sharded(q, k, v, decay_a=None, feature_map="elu1", omega=None, group=None,
                             return_state=False, ops=CudaOps):
    """Causal forward of this rank's shard of every head's sequence.

    q, k, v: [B, H, n_r, d], this rank's n_r consecutive tokens (shards in rank
    order; lengths may differ and may be zero); decay_a [H] or None and omega
    [d, m] are the same on every rank.  Returns the shard's outputs, or
    (out, μ, ν) with ``return_state``: the state after the shard (on the last
    rank, the final state of the whole sequence).  ``ops`` performs the
    per-rank steps (by default the library's kernels on q's device).
    """
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    Bn, H, n, d = q.shape
    dp = d if feature_map == "elu1" else int(omega.shape[1])
    dev = q.device
    # the length of every shard
    n_t = torch.tensor([n], dtype=torch.int64, device=dev)
    lens = [torch.empty_like(n_t) for _ in range(world)]
    dist.all_gather(lens, n_t, group=group)
    shard_len = [int(t.item()) for t in lens]
    # this shard's aggregate, μ then ν in one buffer, and everyone's
    nmu = Bn * H * dp * d
    flat = torch.empty(nmu + Bn * H * dp, dtype=torch.float32, device=dev)
    ops.forward_state(k, v, decay_a, feature_map, omega, flat[:nmu].view(Bn, H, dp, d),
                      flat[nmu:].view(Bn, H, dp))
    gathered = torch.empty(world, flat.numel(), dtype=torch.float32, device=dev)
    dist.all_gather(list(gathered.unbind(0)), flat, group=group)
    mu_in, nu_in = ops.shard_entering_state(gathered, rank, shard_len, Bn, H, dp, d, decay_a)
    return ops.forward_from_state(q, k, v, mu_in, nu_in, decay_a, feature_map, omega,
                                  return_state)
