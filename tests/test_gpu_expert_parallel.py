"""Expert parallelism on one GPU: the ranks' shards run one after another.

A layer split into expert-range shards (moe_config expert_begin/expert_end):
each shard's moe_forward gives the routed sum over the pairs whose expert it
holds; the fp32 sum of the shards' partial outputs (what the all-reduce of
forward_prefill.rs's EP block computes) plus moe_shared_expert_add must equal
the whole layer -- the kernels' own output and the oracle's.  A shard's
moe_permute counts only its experts.
"""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_gemv_gb300 import inputs as I
from _parity import TOL, check_ids, forced_routing, rel_l2, to_np, tol

pytestmark = pytest.mark.gpu

SHARED_BF16 = I.LayerShape(hidden=512, num_experts=16, top_k=4, inter=256, shared_inter=256)
SMALL_FP8 = I.LayerShape(hidden=512, num_experts=8, top_k=2, inter=512, shared_inter=512, fp8=True)
NO_SHARED = I.LayerShape(hidden=512, num_experts=16, top_k=4, inter=256)


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_gemv_gb300 import binding
    binding.load_library()
    return torch.device("cuda", 0)


@pytest.mark.parametrize("arm", ["gemv", "gemm"])
@pytest.mark.parametrize("shape,m,world", [(SHARED_BF16, 5, 2), (SHARED_BF16, 300, 2), (SHARED_BF16, 40, 3),
                                           (SMALL_FP8, 6, 2), (SMALL_FP8, 200, 2), (I.SMALL_NVFP4, 24, 2),
                                           (NO_SHARED, 64, 4)])
def test_shards_sum_to_the_whole_layer(cuda, oracle_mod, arm, shape, m, world):
    from mixture_experts_ffn_gemv_gb300 import binding
    from mixture_experts_ffn_gemv_gb300 import expert_parallel as ep
    wl = I.Workload("ep", shape, (m,))
    tensors = I.make_layer(wl, seed=131, device=cuda)
    x = I.make_x(shape, m, seed=131, device=cuda)
    full = binding.MoeLayer(shape, tensors)
    try:
        whole, ids, w = full.moe_forward(x, tensors["router_w"], tensors["router_bias"], arm=arm, return_routing=True)
    except binding.MoeError as e:
        if e.status == binding.MOE_ERR_UNSUPPORTED and arm == "gemm":
            pytest.skip("grouped GEMM arm not available for this shape")
        raise
    acc = torch.zeros(m, shape.hidden, dtype=torch.float32, device=cuda)
    shards = []
    for r in range(world):
        b, e = ep.shard_range(shape.num_experts, world, r)
        layer = binding.MoeLayer(shape, ep.shard_tensors(tensors, b, e), expert_range=(b, e))
        shards.append(layer)
        acc += layer.moe_forward(x, tensors["router_w"], tensors["router_bias"], arm=arm).float()
        assert layer.device_status() == 0  # other shards' pairs are dropped without an error
        off, sp, sl = layer.moe_permute(ids)
        torch.cuda.synchronize()
        mine = ((ids >= b) & (ids < e)).sum().item()
        assert off.shape[0] == e - b + 1 and int(off[-1]) == mine
        assert int((sl >= 0).sum()) == mine
    out = acc.to(torch.bfloat16)
    if shape.shared_inter:
        shards[0].moe_shared_expert_add(x, out, arm=arm)
    else:
        with pytest.raises(binding.MoeError):
            shards[0].moe_shared_expert_add(x, out, arm=arm)
    torch.cuda.synchronize()
    # the whole layer: the kernels' own, then the oracle's (forced ids on near-ties)
    assert rel_l2(to_np(out), to_np(whole)) < 1e-2
    host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in tensors.items()}
    ref = oracle_mod.reference(shape, host, x.cpu())
    swapped, bad = check_ids(to_np(ids), ref["ids"], ref["logits"])
    assert not bad
    f_ids, f_w = forced_routing(oracle_mod, shape, ref["logits"], ref["ids"], ref["w"], to_np(ids), swapped)
    want = oracle_mod.moe_forward(shape, host, x.cpu(), f_ids, f_w)
    assert rel_l2(to_np(out), want) < tol(shape)


def test_shard_range_is_checked(cuda):
    from mixture_experts_ffn_gemv_gb300 import binding
    shape = NO_SHARED
    tensors = I.make_layer(I.Workload("ep", shape, (4,)), seed=5, device=cuda)
    for rng in [(4, 4), (-1, 3), (3, 17), (5, 2)]:
        with pytest.raises(binding.MoeError):
            binding.MoeLayer(shape, tensors, expert_range=rng)
