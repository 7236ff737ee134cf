"""Vocabulary-parallel (tensor-parallel) selected-token log-probabilities.

Each of n ranks (n in {1, 2, 4}) holds one contiguous shard of the vocabulary:
rows [begin, end) of the LM-head weight W (or those columns of the logits),
with (begin, end) = lp_vocab_shard_range(V, rank, n), a whole number of the
four fixed vocabulary quarters.  One call on every rank

  1. computes its shard's per-row quarter states with liblp
     (lp_linear_logprob_partials / lp_logprob_partials_from_logits);
  2. all-gathers the states of every rank, in rank order, into one buffer
     (the only exchange: 32 bytes per row and quarter; byte movement, no
     arithmetic, so the collective's algorithm, protocol or channel count
     cannot change a bit);
  3. merges the four quarter states of every row with lp_merge_partials in
     the fixed order (Q0 + Q1) + (Q2 + Q3) and finalises logp and entropy.

Every rank ends with the logp and entropy of all T rows, bit-identical to the
unsharded single-GPU call on the same inputs: the tp4_equals_tp1 property of
the RL-Kernel logprob prior-art report (report.json, candidates.*.
tp4_equals_tp1), which the Megatron-style all-reduce of partial sums does not
have (candidates.megatron_ce.tp4_equals_tp1 is false).  The pages also ship
their own all-gather kernels for this exchange (the strict R/R trace runbook,
RL-Kernel issue #342, section 3, deterministic_all_gather_kernel); here the
exchange is torch.distributed's all_gather_into_tensor.

Training on the logits path needs nothing more: the forward's merge can also
return each row's log Z (lp_merge_partials_lse), and every element of dL/dz
depends only on its own logit and its row's log Z and entropy, so each rank
takes the gradient of its own columns (lp_logprob_partials_from_logits_backward)
and holds exactly those columns of the single-GPU gradient, with no exchange.

Training on the fused path (vocab_parallel_linear_logprob_lse, then
vocab_parallel_linear_logprob_backward) has one exchange in the backward: each
rank's grad_W rows are G_shard^T H, the rows of the single-GPU grad_W, but
grad_H = G W sums over the whole vocabulary.  liblp sums grad_H over fixed
vocabulary ranges inside each quarter and then adds the quarter sums as
(Q0 + Q1) + (Q2 + Q3), so a rank's partial grad_H
(lp_linear_logprob_partials_backward) is one subtree of that order; the
partials are all-gathered in rank order (4 T d bytes per rank, byte movement
again) and every rank adds them in the same tree (lp_merge_grad_h_partials).
grad_H is then the single-GPU bits on every rank: an all-reduce, whose order
depends on the collective, would not give that.  This needs V % 64 == 0 (the
quarters start on 16-column boundaries).

Collective backends: NCCL gathers the device buffers directly; any other
backend (gloo) gathers host copies, staged through pinned memory.  All compute
runs in liblp's kernels; this module only moves the states.
"""

from __future__ import annotations

import contextlib
from typing import Optional

import torch
import torch.distributed as dist

from . import lp

__all__ = [
    "shard_of_rank",
    "gather_partials",
    "vocab_parallel_linear_logprob",
    "vocab_parallel_linear_logprob_lse",
    "vocab_parallel_linear_logprob_backward",
    "vocab_parallel_logprob_from_logits",
    "vocab_parallel_logprob_from_logits_lse",
    "vocab_parallel_logprob_from_logits_backward",
]


def _group_info(group) -> tuple[int, int]:
    if not dist.is_available() or not dist.is_initialized():
        return 0, 1
    return dist.get_rank(group), dist.get_world_size(group)


def _on(stream):
    """Run on `stream` (a torch.cuda.Stream) when given, else on the current stream."""
    return torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()


def shard_of_rank(vocab_total: int, group=None) -> tuple[int, int, int, int]:
    """(shard_index, n_shards, begin, end) of the calling rank: shard i is
    rank i of the group; the group size must be 1, 2 or 4."""
    rank, n = _group_info(group)
    if n not in (1, 2, 4):
        raise ValueError(f"vocabulary parallelism needs 1, 2 or 4 ranks, not {n}")
    b, e = lp.vocab_shard_range(vocab_total, rank, n)
    return rank, n, b, e


def gather_partials(partials: torch.Tensor, group=None) -> list[torch.Tensor]:
    """All-gather one [T, n_q, k] state tensor per rank; returns the n tensors
    in rank order (views into one contiguous buffer on partials' device)."""
    rank, n = _group_info(group)
    if n == 1:
        return [partials]
    part = partials.contiguous()
    T = part.shape[0]
    backend = dist.get_backend(group)
    if part.is_cuda and backend != "nccl":
        # host-staged: gloo and the other CPU backends gather host tensors
        host = torch.empty(part.shape, dtype=part.dtype, pin_memory=True)
        host.copy_(part)
        out_host = torch.empty((n * T,) + tuple(part.shape[1:]), dtype=part.dtype)
        dist.all_gather_into_tensor(out_host, host, group=group)
        out = out_host.to(part.device, non_blocking=False)
    else:
        out = torch.empty((n * T,) + tuple(part.shape[1:]), dtype=part.dtype, device=part.device)
        dist.all_gather_into_tensor(out, part, group=group)
    return [out[i * T:(i + 1) * T] for i in range(n)]


def vocab_parallel_linear_logprob(H: torch.Tensor, W_shard: torch.Tensor, y: torch.Tensor,
                                  vocab_total: int, group=None, with_entropy: bool = True,
                                  temperature: Optional[float] = None, workspace=None,
                                  stream=None):
    """logp [T] and entropy [T] (or None) of softmax(H W^T), W split by rows
    across the ranks of `group`; every rank passes the same H and y and its own
    W_shard = W[begin:end] (see shard_of_rank)."""
    rank, n, b, e = shard_of_rank(vocab_total, group)
    _check_w_shard(W_shard, rank, b, e)
    with _on(stream):
        parts = lp.linear_logprob_partials(H, W_shard, y, vocab_total, rank, n,
                                           workspace=workspace, temperature=temperature)
        gathered = gather_partials(parts, group)
        return lp.merge_partials(gathered, with_entropy=with_entropy)


def _check_w_shard(W_shard, rank, b, e):
    if W_shard.shape[0] != e - b:
        raise ValueError(f"rank {rank} holds {W_shard.shape[0]} rows of W, its shard has {e - b}")


def vocab_parallel_linear_logprob_lse(H: torch.Tensor, W_shard: torch.Tensor, y: torch.Tensor,
                                      vocab_total: int, group=None, temperature: float = 1.0,
                                      workspace=None, stream=None):
    """(logp, entropy, lse) [T] of softmax(H W^T / tau), W split by rows: the
    forward of vocabulary-parallel training on the fused path; every rank gets
    the same bits (those of lp_linear_logprob_lse on one GPU)."""
    rank, n, b, e = shard_of_rank(vocab_total, group)
    _check_w_shard(W_shard, rank, b, e)
    T = H.shape[0]
    with _on(stream):
        parts = lp.linear_logprob_partials(H, W_shard, y, vocab_total, rank, n,
                                           workspace=workspace, temperature=temperature)
        gathered = gather_partials(parts, group)
        out = [torch.empty(T, dtype=torch.float32, device=H.device) for _ in range(3)]
        lp.lp_merge_partials_lse(gathered, T, out[0], out[1], out[2])
        return tuple(out)


def vocab_parallel_linear_logprob_backward(H: torch.Tensor, W_shard: torch.Tensor,
                                           y: torch.Tensor, vocab_total: int,
                                           saved_lse: torch.Tensor, saved_entropy: torch.Tensor,
                                           grad_logp=None, grad_entropy=None, group=None,
                                           temperature: float = 1.0, with_grad_W: bool = True,
                                           grad_W_dtype=torch.float32, workspace=None,
                                           stream=None, accumulate_into=None):
    """(grad_H [T, d] fp32, grad_W_shard [end - begin, d] or None) from the merged
    rows' log Z and entropy (vocab_parallel_linear_logprob_lse): grad_H is the
    same on every rank and equal to the single-GPU result bit for bit, and
    grad_W_shard is rows begin..end of the single-GPU grad_W (added into
    accumulate_into, this rank's float32 main gradient rows, when given)."""
    rank, n, b, e = shard_of_rank(vocab_total, group)
    _check_w_shard(W_shard, rank, b, e)
    with _on(stream):
        part, gW = lp.linear_logprob_partials_backward(
            H, W_shard, y, vocab_total, rank, n, saved_lse, saved_entropy, grad_logp,
            grad_entropy, temperature=temperature, with_grad_W=with_grad_W,
            grad_W_dtype=grad_W_dtype, workspace=workspace, accumulate_into=accumulate_into)
        gathered = gather_partials(part, group)
        return lp.merge_grad_h_partials(gathered), gW


def vocab_parallel_logprob_from_logits(z_shard: torch.Tensor, y: torch.Tensor, vocab_total: int,
                                       group=None, with_entropy: bool = True,
                                       temperature: Optional[float] = None, stream=None):
    """logp [T] and entropy [T] (or None) of softmax(z), the fp32 logits split
    by columns across the ranks of `group`; z_shard = z[:, begin:end]."""
    rank, n, b, e = shard_of_rank(vocab_total, group)
    if z_shard.shape[1] != e - b:
        raise ValueError(f"rank {rank} holds {z_shard.shape[1]} logit columns, its shard has {e - b}")
    with _on(stream):
        parts = lp.logprob_partials_from_logits(z_shard, y, vocab_total, rank, n,
                                                temperature=temperature)
        gathered = gather_partials(parts, group)
        return lp.merge_partials(gathered, with_entropy=with_entropy)


def vocab_parallel_logprob_from_logits_lse(z_shard: torch.Tensor, y: torch.Tensor,
                                           vocab_total: int, group=None,
                                           temperature: float = 1.0, stream=None):
    """(logp, entropy, lse) [T] of softmax(z / tau) from the column-split logits:
    the forward of vocabulary-parallel training; every rank gets the same bits."""
    rank, n, b, e = shard_of_rank(vocab_total, group)
    if z_shard.shape[1] != e - b:
        raise ValueError(f"rank {rank} holds {z_shard.shape[1]} logit columns, its shard has {e - b}")
    T = z_shard.shape[0]
    with _on(stream):
        parts = lp.logprob_partials_from_logits(z_shard, y, vocab_total, rank, n,
                                                temperature=temperature)
        gathered = gather_partials(parts, group)
        out = [torch.empty(T, dtype=torch.float32, device=z_shard.device) for _ in range(3)]
        lp.lp_merge_partials_lse(gathered, T, out[0], out[1], out[2])
        return tuple(out)


def vocab_parallel_logprob_from_logits_backward(z_shard: torch.Tensor, y: torch.Tensor,
                                                vocab_total: int, saved_lse: torch.Tensor,
                                                saved_entropy: torch.Tensor, grad_logp=None,
                                                grad_entropy=None, group=None,
                                                temperature: float = 1.0,
                                                stream=None) -> torch.Tensor:
    """dL/dz for this rank's columns, from the merged rows' log Z and entropy
    (vocab_parallel_logprob_from_logits_lse): no exchange, and the bits of the
    same columns of the single-GPU gradient."""
    rank, n, b, e = shard_of_rank(vocab_total, group)
    if z_shard.shape[1] != e - b:
        raise ValueError(f"rank {rank} holds {z_shard.shape[1]} logit columns, its shard has {e - b}")
    grad = torch.empty(z_shard.shape, dtype=torch.float32, device=z_shard.device)
    with _on(stream):
        lp.lp_logprob_partials_from_logits_backward(z_shard, y, vocab_total, rank, n, temperature,
                                                    saved_lse, saved_entropy, grad_logp,
                                                    grad_entropy, grad)
    return grad
