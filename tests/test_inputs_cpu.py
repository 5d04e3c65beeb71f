"""The seeded input generators and the benchmark's byte accounting (CPU only).

The generators draw every tensor from its own (seed, name, expert) stream, so
one expert can be regenerated alone and sampled oracle checks at full size see
exactly the weights the device holds; the benchmark's algorithmic bytes are
the storage sizes of what a launch must read and write.
"""
import os
import sys

import pytest
import torch

from mixture_experts_ffn_gemv_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SHAPES = {
    "bf16": I.LayerShape(hidden=256, num_experts=6, top_k=2, inter=128, shared_inter=128),
    "fp8": I.LayerShape(hidden=256, num_experts=6, top_k=2, inter=256, shared_inter=256, fp8=True),
    "nvfp4": I.LayerShape(hidden=256, num_experts=6, top_k=2, inter=256, shared_inter=256, nvfp4=True),
}


@pytest.mark.parametrize("fmt", sorted(SHAPES))
def test_one_expert_regenerates_alone(fmt):
    shape = SHAPES[fmt]
    full = I.make_experts(shape, seed=3)
    part = I.make_experts(shape, seed=3, experts=[4])
    for name, t in full.items():
        if t.dim() >= 1 and t.shape[0] == shape.num_experts and name in part:
            assert torch.equal(part[name][4], t[4]), name
            assert not part[name][0].any(), name  # the others are left zero
        else:
            assert torch.equal(part[name], t), name  # the shared expert is always drawn


@pytest.mark.parametrize("fmt", sorted(SHAPES))
def test_generators_are_deterministic_and_seed_dependent(fmt):
    shape = SHAPES[fmt]
    a = I.make_experts(shape, seed=1)
    b = I.make_experts(shape, seed=1)
    c = I.make_experts(shape, seed=2)
    assert all(torch.equal(a[n], b[n]) for n in a)
    assert any(not torch.equal(a[n], c[n]) for n in ("w1", "w3", "w2"))
    assert torch.equal(I.make_x(shape, 5, seed=1), I.make_x(shape, 5, seed=1))


def test_nvfp4_storage_layout():
    shape = SHAPES["nvfp4"]
    t = I.make_experts(shape, seed=0)
    E, H, Iw = shape.num_experts, shape.hidden, shape.inter
    assert t["w1"].shape == (E, Iw, H // 2) and t["w1"].dtype == torch.uint8
    assert t["w2"].shape == (E, H, Iw // 2)
    assert t["sb1"].shape == (E, Iw, H // 16) and t["sb2"].shape == (E, H, Iw // 16)
    assert t["s1"].shape == (E,) and t["s1"].dtype == torch.float32
    assert t["ws1"].shape == (Iw, H // 2) and t["ssb2"].shape == (H, Iw // 16) and t["ss3"].shape == (1,)
    # block-scale codes stay in the e4m3 codes of [0.5, 4): positive, finite, normal
    for n in ("sb1", "sb3", "sb2", "ssb1", "ssb3", "ssb2"):
        assert int(t[n].min()) >= 0x30 and int(t[n].max()) <= 0x47, n


def test_bench_byte_accounting():
    sys.path.insert(0, ROOT)
    import bench
    q = I.QWEN3_30B_A3B
    assert bench.expert_bytes(q) == 3 * 2048 * 768 * 2
    d = I.DEEPSEEK_V3
    assert bench.expert_bytes(d) == 3 * 7168 * 2048 + 3 * (7168 // 128) * (2048 // 128) * 4
    n = I.QWEN3_NVFP4
    assert bench.expert_bytes(n) == 3 * 2048 * 768 // 2 + 3 * 2048 * 768 // 16 + 12
    # a GEMV launch reads each active expert's matrices once
    U, m = 80, 16
    g = bench.kernel_alg_bytes("gemv_gateup", q, m, U)
    assert g == U * 2 * 768 * 2048 * 2 + m * 2048 * 2 + m * 8 * 768 * 2
    gn = bench.kernel_alg_bytes("gemv_gateup", n, m, U)
    assert gn < g / 3  # NVFP4 weights take 0.5625 bytes per element against 2
    # W4A4: activations count at NVFP4 size too (codes + block scales + a row scale)
    xa, ha = 2048 * bench.NVFP4_B + 4, 768 * bench.NVFP4_B + 4
    assert gn == int(U * 2 * 768 * 2048 * bench.NVFP4_B + m * xa + m * 8 * ha)
    gm = bench.kernel_alg_bytes("gemm_gateup", n, 4096, 128)
    assert gm == int(128 * 2 * 768 * 2048 * bench.NVFP4_B + 4096 * 8 * (xa + ha))
    assert bench._dtype(n) == "nvfp4_e2m1" and bench._dtype(d) == "fp8_e4m3" and bench._dtype(q) == "bf16"
