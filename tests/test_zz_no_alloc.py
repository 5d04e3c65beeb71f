"""moe_permute_noalloc -- the permute for callers that cannot allocate device
memory (inside CUDA graph capture, allocator-free serving loops, runtimes
without a device allocator) -- must give exactly what the workspace-based
moe_permute gives.  It runs its kernels on a fixed scratch array inside the
library, so two calls in a row also check that the second call is not
disturbed by what the first one left there.

This file sorts last so that a run stopping at the first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _ids(m, k, E, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.permutation(E)[:k] for _ in range(m)]).astype(np.int32)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_permute_matches_workspace_permute():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_gemv_gb300 import binding
    from mixture_experts_ffn_gemv_gb300 import inputs as I

    lib = binding.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    # two calls in a row with different sizes (the second one smaller, so it
    # would read stale histograms if the scratch were not handled correctly),
    # then the first one again
    for m, k, E, seed in [(700, 8, 128, 1), (64, 4, 40, 2), (700, 8, 128, 3)]:
        ids = torch.from_numpy(_ids(m, k, E, seed)).to(dev)
        P = m * k
        shape = I.LayerShape(hidden=256, num_experts=E, top_k=k, inter=128)
        zeros = {n: torch.zeros(E, 128, 256, dtype=torch.bfloat16, device=dev) for n in ("w1", "w3")}
        zeros["w2"] = torch.zeros(E, 256, 128, dtype=torch.bfloat16, device=dev)
        ref_off, ref_sp, ref_sl = binding.MoeLayer(shape, zeros).moe_permute(ids)

        off = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
        sp = torch.full((P,), -7, dtype=torch.int32, device=dev)
        sl = torch.full((P,), -7, dtype=torch.int32, device=dev)
        rc = lib.moe_permute_noalloc(_ptr(ids), m, k, E, _ptr(off), _ptr(sp), _ptr(sl), stream)
        assert rc == binding.MOE_OK, binding.status_string(rc)
        torch.cuda.synchronize(dev)
        assert torch.equal(off, ref_off)
        assert torch.equal(sp, ref_sp)
        assert torch.equal(sl, ref_sl)

    # an out-of-range id: both entry points drop that pair the same way, and
    # expert_offsets[E] (the count of valid pairs) is how this caller sees it
    m, k, E = 50, 4, 16
    bad = _ids(m, k, E, 4)
    bad[7, 2] = E + 3
    ids = torch.from_numpy(bad).to(dev)
    shape = I.LayerShape(hidden=256, num_experts=E, top_k=k, inter=128)
    zeros = {n: torch.zeros(E, 128, 256, dtype=torch.bfloat16, device=dev) for n in ("w1", "w3")}
    zeros["w2"] = torch.zeros(E, 256, 128, dtype=torch.bfloat16, device=dev)
    ref_layer = binding.MoeLayer(shape, zeros)
    ref_off, ref_sp, ref_sl = ref_layer.moe_permute(ids)
    assert ref_layer.device_status() == 1  # the workspace path reports DEV_ERR_BAD_ID
    off = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    sp = torch.full((m * k,), -7, dtype=torch.int32, device=dev)
    sl = torch.full((m * k,), -7, dtype=torch.int32, device=dev)
    rc = lib.moe_permute_noalloc(_ptr(ids), m, k, E, _ptr(off), _ptr(sp), _ptr(sl), stream)
    assert rc == binding.MOE_OK
    torch.cuda.synchronize(dev)
    assert int(off[E]) == m * k - 1 and torch.equal(off, ref_off)
    assert int(sl[7 * k + 2]) == -1 and torch.equal(sl, ref_sl)
    assert torch.equal(sp, ref_sp) and int(sp[-1]) == -1

    # a call whose histograms would not fit in the fixed scratch is refused
    big = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = lib.moe_permute_noalloc(_ptr(big), 32768, 8, 1024, _ptr(big), _ptr(big), _ptr(big), stream)
    assert rc == binding.MOE_ERR_UNSUPPORTED
