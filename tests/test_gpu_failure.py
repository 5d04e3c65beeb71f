"""Failure handling on the GPU, without a GPU fault.

Every mbarrier wait in the grouped-GEMM kernels is bounded.  Here a wait is
made to run out on purpose -- the tensor-core issuer first waits on a barrier
that no thread ever completes (moe_layer_stall_test) under a short wait limit,
on the one-CTA kernel and on the CTA-pair gate/up kernel -- and the call must
come back with the device error word set to DEV_ERR_TIMEOUT, the context
usable, and the next call clean and equal to the oracle.  (forward_prefill.rs reports failures through Rust's Result; the
bounded wait is this library's device-side counterpart.)
"""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_gemv_gb300 import inputs as I
from _parity import TOL, check_ids, forced_routing, rel_l2, to_np

pytestmark = pytest.mark.gpu

DEV_ERR_TIMEOUT = 2
SHAPE = I.LayerShape(hidden=1024, num_experts=8, top_k=2, inter=256)


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_gemv_gb300 import binding
    binding.load_library()
    return torch.device("cuda", 0)


# 400 routed rows over 8 experts: the one-CTA grouped GEMM; 600 rows over 2
# experts: gate/up on CTA pairs
PAIR_SHAPE = I.LayerShape(hidden=1024, num_experts=2, top_k=1, inter=256)


@pytest.mark.parametrize("shape,m", [(SHAPE, 200), (PAIR_SHAPE, 600)])
def test_stalled_gemm_times_out_and_the_next_call_is_clean(cuda, oracle_mod, shape, m):
    from mixture_experts_ffn_gemv_gb300 import binding
    wl = I.Workload("stall", shape, (m,))
    tensors = I.make_layer(wl, seed=61, device=cuda)
    x = I.make_x(shape, m, seed=61, device=cuda)
    layer = binding.MoeLayer(shape, tensors)
    assert layer.select_arm(m) == binding.MOE_ARM_GEMM

    layer.set_wait_limit(200_000)  # 200 us
    layer.stall_test(True)
    for _ in range(2):  # twice: the abort path leaves nothing behind
        layer.moe_forward(x, tensors["router_w"], arm="gemm")
        assert layer.device_status() == DEV_ERR_TIMEOUT

    layer.stall_test(False)
    layer.set_wait_limit(0)  # back to the default limit
    out, ids, w = layer.moe_forward(x, tensors["router_w"], arm="gemm", return_routing=True)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in tensors.items()}
    ref = oracle_mod.reference(shape, host, x.cpu())
    swapped, bad = check_ids(to_np(ids), ref["ids"], ref["logits"])
    assert not bad, bad[:5]
    f_ids, f_w = forced_routing(oracle_mod, shape, ref["logits"], ref["ids"], ref["w"], to_np(ids), swapped)
    want = oracle_mod.moe_forward(shape, host, x.cpu(), f_ids, f_w)
    assert rel_l2(to_np(out), want) < TOL[False]


def test_wait_limit_arguments(cuda):
    from mixture_experts_ffn_gemv_gb300 import binding
    lib = binding.load_library()
    assert lib.moe_layer_set_wait_limit(None, 1000) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_stall_test(None, 1) == binding.MOE_ERR_INVALID_ARG
