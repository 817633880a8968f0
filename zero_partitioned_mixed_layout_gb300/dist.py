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

ZeRO stage 2 and stage 3 add one exchange each.  Stage 2 reduces the
gradient replicas to their owners: here an all-to-all hands every rank all
replicas of its own shard and zero_reduce_grads forms their mean in rank
order (fused with pass 1) -- the traffic of a reduce-scatter, with a
summation order that does not depend on the collective's algorithm.  Stage 3
gathers the parameter shards before a layer runs: an all-gather, then
zero_gather_params cuts the tensors out of the shards.

1-bit Adam's compression stage adds two exchanges of signs and scales: after
zero_onebit_worker, chunk j of every worker's signs (and every worker's
scale) to rank j, an all-to-all; after zero_onebit_server, every rank's
chunk signs and scale to every worker, an all-gather.  They move the 1-bit
messages only: the arithmetic stays in the library's calls on each rank.
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


def _flat(t, what):
    if t.dim() != 1:
        raise ValueError(f"{what} must be a 1-D tensor")
    return t.contiguous()


def stage2_exchange_grads(grad, group=None):
    """ZeRO stage 2's gradient exchange (an all-to-all).  grad: this rank's
    gradient over the whole padded flat buffer, n = Nd*S elements (shard j,
    [j*S, (j+1)*S), goes to rank j).  Returns [Nd, S] of grad's type: every
    rank's gradient on this rank's shard, in rank order -- the replicas of
    zero_reduce_grads (one row each)."""
    import torch
    import torch.distributed as dist
    grad = _flat(grad, "grad")
    nd = dist.get_world_size(group)
    if grad.numel() % nd != 0:
        raise ValueError("the gradient must split into one equal shard per rank")
    out = torch.empty_like(grad)
    dist.all_to_all_single(out, grad, group=group)
    return out.view(nd, -1)


def stage3_gather_shards(shard, group=None):
    """ZeRO stage 3's parameter exchange (an all-gather).  shard: this
    rank's S elements.  Returns [Nd, S]: every rank's shard in rank order --
    the shards of zero_gather_params (one row each)."""
    import torch
    import torch.distributed as dist
    shard = _flat(shard, "shard")
    nd = dist.get_world_size(group)
    out = torch.empty(nd * shard.numel(), dtype=shard.dtype, device=shard.device)
    dist.all_gather_into_tensor(out, shard, group=group)
    return out.view(nd, -1)


def _check_words(bits, what):
    import torch
    if bits.dtype != torch.int32 or bits.dim() != 1:
        raise ValueError(f"{what} must be a 1-D int32 tensor of sign words")


def onebit_exchange_worker_signs(bits, scale, group=None):
    """The worker-side exchange of a 1-bit Adam step (an all-to-all).
    bits: this rank's signs, int32[n/32] with n = Nd*S (chunk j, words
    [j*S/32, (j+1)*S/32), goes to rank j); scale: its scale, float32[1].
    Returns (chunk_bits, worker_scales): the Nd workers' signs on this
    rank's chunk, int32[Nd, S/32] in rank order (row i is the worker_bits[i]
    of zero_onebit_server), and every worker's scale, float32[Nd]."""
    import torch
    import torch.distributed as dist
    _check_words(bits, "bits")
    nd = dist.get_world_size(group)
    if bits.numel() % nd != 0:
        raise ValueError("the sign words must split into one equal chunk per rank")
    if scale.dtype != torch.float32 or scale.numel() != 1:
        raise ValueError("scale must be one float32")
    chunk_bits = torch.empty_like(bits)
    dist.all_to_all_single(chunk_bits, bits.contiguous(), group=group)
    worker_scales = torch.empty(nd, dtype=torch.float32, device=scale.device)
    dist.all_gather_into_tensor(worker_scales, scale.reshape(1).contiguous(), group=group)
    return chunk_bits.view(nd, -1), worker_scales


def onebit_exchange_server_signs(chunk_bits, scale, group=None):
    """The server-side exchange of a 1-bit Adam step (an all-gather).
    chunk_bits: this rank's server signs, int32[S/32]; scale: float32[1].
    Returns (bits, server_scales): every rank's chunk signs in rank order,
    int32[Nd*S/32], and every rank's scale, float32[Nd] -- the bits and
    server_scales of zero_onebit_update."""
    import torch
    import torch.distributed as dist
    _check_words(chunk_bits, "chunk_bits")
    if scale.dtype != torch.float32 or scale.numel() != 1:
        raise ValueError("scale must be one float32")
    nd = dist.get_world_size(group)
    bits = torch.empty(nd * chunk_bits.numel(), dtype=torch.int32, device=chunk_bits.device)
    dist.all_gather_into_tensor(bits, chunk_bits.contiguous(), group=group)
    server_scales = torch.empty(nd, dtype=torch.float32, device=scale.device)
    dist.all_gather_into_tensor(server_scales, scale.reshape(1).contiguous(), group=group)
    return bits, server_scales
