"""Expert parallelism: each rank holds a contiguous range of the experts.

The EP path of spark_model/layers/moe/forward_prefill.rs: every rank routes
all tokens over all experts, runs the experts it holds, the bf16 [m, H] outputs
are summed across ranks by one all-reduce, and the shared expert -- which every
rank holds -- is added once, after the all-reduce ("defer shared expert blend
until after all-reduce" on that page, so it is not counted once per rank).

This module is the host orchestration only: the partial forward and the
shared-expert add are the library's kernels (moe_forward on a shard,
moe_shared_expert_add); the sum is torch.distributed's all-reduce (NCCL on
GPUs), taken in fp32 and rounded to bf16 once.
"""
from __future__ import annotations

import torch

ROUTED = ("w1", "w3", "w2", "s1", "s3", "s2", "sb1", "sb3", "sb2")


def shard_range(num_experts: int, world_size: int, rank: int):
    """Contiguous expert range [begin, end) of `rank`: the experts split as
    evenly as possible, the first num_experts % world_size ranks one more."""
    if not 0 <= rank < world_size or world_size > num_experts:
        raise ValueError("need 0 <= rank < world_size <= num_experts")
    base, extra = divmod(num_experts, world_size)
    begin = rank * base + min(rank, extra)
    return begin, begin + base + (1 if rank < extra else 0)


def shard_tensors(tensors: dict, begin: int, end: int) -> dict:
    """The tensors one shard's layer takes: the routed expert tensors sliced
    to experts [begin, end) (contiguous copies); router, bias and the shared
    expert's tensors unchanged."""
    out = {}
    for name, t in tensors.items():
        if name in ROUTED and isinstance(t, torch.Tensor):
            out[name] = t[begin:end].contiguous()
        else:
            out[name] = t
    return out


def expert_parallel_forward(layer, x, router_w, router_bias=None, arm="auto", group=None, has_shared=None):
    """One layer step on this rank.  `layer` is this rank's shard (a
    binding.MoeLayer made with expert_range, or any object with the same
    moe_forward / moe_shared_expert_add methods).  Returns the full layer
    output (bf16 [m, H]), identical on every rank."""
    import torch.distributed as dist

    partial = layer.moe_forward(x, router_w, router_bias, arm=arm)
    acc = partial.float()
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
    out = acc.to(torch.bfloat16)
    if has_shared is None:
        has_shared = bool(getattr(getattr(layer, "shape", None), "shared_inter", 0))
    if has_shared:
        layer.moe_shared_expert_add(x, out, arm=arm)
    return out
