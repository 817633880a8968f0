"""The one cross-rank exchange of a ZeRO data-parallel optimizer step.

Between pass 1 and pass 2 every rank holds, in the first 16 bytes of its
zero_state_t, the partial (sum of g^2, found_inf) of its own shard.  The norm
for clipping and the overflow that skips the step are global over all
shards, so the ranks sum these two binary64 values before calling
zero_adam_step ([ZeRO card §方法适配]: each data-parallel rank owns and
updates one partition of the optimizer state; the pages' ZeRO keeps the data
parallel communication volume, and this 16-byte sum is all the update step
itself adds).  On one GPU the same sum is formed by the `accumulate` flag of
zero_grad_norm_overflow instead.
"""
from __future__ import annotations


def exchange_partials(state, group=None) -> None:
    """All-reduce (sum) of the 16-byte partial at the head of a zero_state_t
    held in a uint8 tensor (device tensor with NCCL, CPU tensor with gloo)."""
    import torch
    import torch.distributed as dist
    if state.dtype != torch.uint8 or state.numel() < 16:
        raise ValueError("state must be the uint8 bytes of a zero_state_t")
    head = state[:16].view(torch.float64)
    dist.all_reduce(head, op=dist.ReduceOp.SUM, group=group)
