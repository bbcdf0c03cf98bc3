"""Causal kernelized linear attention for GB300 (sm_103a).

Python face of liblinattn (C ABI in include/linattn.h).  The method
("Efficient Transformers II" §2.2 eq (6)–(11); "Linear Attention Research
2026", elu+1 and Performer feature maps):

* ``forward`` — o_j = q'_j·μ_j / q'_j·ν_j with μ_j = a·μ_{j−1} + (1−a)·k'_jᵀv_j,
  ν_j = a·ν_{j−1} + (1−a)·k'_jᵀ (plain sums for a = 1), or the non-causal
  D⁻¹(Q'(K'ᵀV)) of eq (6);
* ``forward_host`` — the same on page-locked host buffers (the library copies them
  in and out, overlapping the copies of some heads with the compute of others);
* ``forward_with_state`` — the same, also returning the final (μ, ν);
* ``forward_from_state`` — the causal form continued from a given (μ, ν);
* ``forward_state`` — the (μ, ν) the causal recurrence reaches from zero,
  without outputs;
* ``shard_entering_state`` and ``sharded.forward_sequence_sharded`` — a
  sequence split into consecutive shards across devices: the state entering
  each shard from the gathered aggregates of the shards before it;
* ``decode_step`` — one recurrent token for many heads, state updated in place;
* ``forward_token_decay`` / ``decode_step_token_decay`` — the causal form with
  a decay a_i and input weight b_i per token ("Efficient Transformers II"
  eq (4) with a, b indexed by the token): μ_i = a_i μ_{i−1} + b_i k'_iᵀv_i;
* ``backward`` — ∂L/∂q, ∂L/∂k, ∂L/∂v and ∂L/∂a of the causal forward.

All work runs in the library's CUDA kernels; PyTorch only allocates device
memory and provides the stream.
"""
from ._binding import (EXPORTED, LinAttnError, backward, debug_build, decode_step,
                       decode_step_token_decay, forward, forward_from_state, forward_host,
                       forward_state, forward_token_decay, forward_with_state, last_device_check,
                       last_device_status, launch_count, library_path, load,
                       selftest_device_check, selftest_wait_timeout, shard_entering_state,
                       status_string)
from .build import build

__all__ = ["forward", "forward_host", "forward_with_state", "forward_from_state", "forward_state",
           "shard_entering_state", "decode_step", "forward_token_decay", "backward",
           "decode_step_token_decay", "last_device_status", "status_string",
           "LinAttnError", "build", "load", "library_path", "launch_count",
           "selftest_wait_timeout", "debug_build", "last_device_check", "selftest_device_check",
           "EXPORTED"]
