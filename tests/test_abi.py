"""The C-ABI library builds, loads and exports every entry point include/*.h
declares; host-side argument checks work without a GPU (no compute calls)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names |= set(re.findall(r"MOE_API[^;{]*?\b(moe_\w+)\s*\(", text, flags=re.S))
    return names


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_ffn_gemv_gb300 import binding
    return binding.load_library()


def test_header_declares_the_pages_entry_points():
    names = _declared()
    for n in ("moe_route", "moe_permute", "moe_forward", "moe_experts", "moe_layer_create"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from mixture_experts_ffn_gemv_gb300 import binding
    names = _declared()
    assert names, "no MOE_API declarations found"
    for n in names:
        assert hasattr(lib, n), n
    assert set(binding.EXPORTED) == names


def test_status_strings(lib):
    assert lib.moe_status_string(0) == b"ok"
    assert lib.moe_status_string(3) == b"workspace too small"
    assert lib.moe_status_string(99) == b"unknown status"


def _cfg(**kw):
    from mixture_experts_ffn_gemv_gb300.binding import MoeConfig
    c = dict(hidden=256, num_experts=8, top_k=2, inter=128, shared_inter=0, weights=0)
    c.update(kw)
    return MoeConfig(**c)


def _weights(fp8=False, nvfp4=False):
    from mixture_experts_ffn_gemv_gb300.binding import MoeExpertWeights
    fake = 0x10000  # never dereferenced: creation fails or stops before any device access
    sc = fake if (fp8 or nvfp4) else None
    sb = fake if nvfp4 else None
    return MoeExpertWeights(fake, fake, fake, sc, sc, sc, None, sb, sb, sb)


@pytest.mark.parametrize("kw,want", [
    (dict(hidden=200), 2),              # H not a multiple of 128
    (dict(inter=100), 2),               # I not a multiple of 128
    (dict(num_experts=2048, top_k=2), 2),  # more experts than the top-k kernel covers
    (dict(top_k=40, num_experts=64), 2),   # k > 32
    (dict(top_k=9, num_experts=8), 1),     # k > E
    (dict(weights=7), 1),
    (dict(shared_inter=256), 2),        # shared expert of another width
    (dict(weights=1, inter=384), 2),    # fp8 needs I % 512 == 0
    (dict(weights=1, inter=512, hidden=384), 2),  # ... and H % 512 == 0
    (dict(weights=2, inter=384), 2),    # NVFP4 needs I % 256 == 0
    (dict(weights=2, inter=256, hidden=384), 2),  # ... and H % 256 == 0
    (dict(scoring=2), 1),                          # no such scoring
    (dict(scoring=1, routed_scaling_factor=0.0), 1),  # sigmoid scoring needs a positive scaling factor
    (dict(scoring=1, routed_scaling_factor=float("inf")), 1),
    (dict(scoring=1, routed_scaling_factor=2.5, norm_topk_prob=3), 1),
])
def test_create_rejects_unsupported_shapes(lib, kw, want):
    from mixture_experts_ffn_gemv_gb300.binding import MoeExpertWeights
    cfg = _cfg(**kw)
    w = _weights(fp8=cfg.weights == 1, nvfp4=cfg.weights == 2)
    shared = MoeExpertWeights(0x10000, 0x10000, 0x10000) if cfg.shared_inter else None
    out = ctypes.c_void_p()
    rc = lib.moe_layer_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(shared) if shared else None,
                              ctypes.byref(out))
    assert rc == want
    assert not out.value


def test_create_rejects_null_and_misaligned(lib):
    from mixture_experts_ffn_gemv_gb300.binding import MoeExpertWeights
    out = ctypes.c_void_p()
    assert lib.moe_layer_create(None, None, None, ctypes.byref(out)) == 1
    cfg = _cfg()
    bad = MoeExpertWeights(0x10001, 0x10000, 0x10000)
    assert lib.moe_layer_create(ctypes.byref(cfg), ctypes.byref(bad), None, ctypes.byref(out)) == 1
    missing_scales = _weights(fp8=False)
    cfg8 = _cfg(weights=1, inter=512, hidden=512)
    assert lib.moe_layer_create(ctypes.byref(cfg8), ctypes.byref(missing_scales), None, ctypes.byref(out)) == 1


def test_create_checks_nvfp4_block_scales(lib):
    from mixture_experts_ffn_gemv_gb300.binding import MoeExpertWeights
    out = ctypes.c_void_p()
    cfg4 = _cfg(weights=2, inter=256, hidden=512)
    f = 0x10000
    no_blocks = MoeExpertWeights(f, f, f, f, f, f)                       # NVFP4 without block scales
    assert lib.moe_layer_create(ctypes.byref(cfg4), ctypes.byref(no_blocks), None, ctypes.byref(out)) == 1
    no_tensor = MoeExpertWeights(f, f, f, None, None, None, None, f, f, f)  # ... or without tensor scales
    assert lib.moe_layer_create(ctypes.byref(cfg4), ctypes.byref(no_tensor), None, ctypes.byref(out)) == 1
    odd = MoeExpertWeights(f, f, f, f, f, f, None, f, f + 2, f)          # misaligned block scales
    assert lib.moe_layer_create(ctypes.byref(cfg4), ctypes.byref(odd), None, ctypes.byref(out)) == 1
    bf16_with_blocks = MoeExpertWeights(f, f, f, None, None, None, None, f, f, f)
    assert lib.moe_layer_create(ctypes.byref(_cfg()), ctypes.byref(bf16_with_blocks), None,
                                ctypes.byref(out)) == 1
    assert not out.value


def test_gate_only_on_the_shared_expert(lib):
    from mixture_experts_ffn_gemv_gb300.binding import MoeExpertWeights
    out = ctypes.c_void_p()
    cfg = _cfg()
    gated_routed = MoeExpertWeights(0x10000, 0x10000, 0x10000, None, None, None, 0x10000)
    assert lib.moe_layer_create(ctypes.byref(cfg), ctypes.byref(gated_routed), None, ctypes.byref(out)) == 1
    cfg_s = _cfg(shared_inter=128)
    misaligned_gate = MoeExpertWeights(0x10000, 0x10000, 0x10000, None, None, None, 0x10004)
    assert lib.moe_layer_create(ctypes.byref(cfg_s), ctypes.byref(_weights()), ctypes.byref(misaligned_gate),
                                ctypes.byref(out)) == 1
    assert not out.value


def test_null_layer_calls_are_rejected(lib):
    assert lib.moe_forward(None, None, 4, None, None, None, None, None, 0, None, 0, None) == 1
    assert lib.moe_route(None, None, 1, None, None, None, None, None, None, 0, None) == 1
    assert lib.moe_permute(None, None, 1, None, None, None, None, 0, None) == 1
    assert lib.moe_select_arm(None, 4) == 1
    assert lib.moe_last_launch_count(None) == -1
    assert lib.moe_act_quant_fp8(None, 4, 100, None, None, None) == 1  # n % 128 != 0
    assert lib.moe_act_quant_fp8(None, 0, 128, None, None, None) == 0  # nothing to do
    assert lib.moe_act_quant_nvfp4(None, 4, 100, None, None, None, None) == 1  # n % 16 != 0
    assert lib.moe_act_quant_nvfp4(None, 0, 128, None, None, None, None) == 0
    assert lib.moe_act_quant_nvfp4(None, 4, 128, None, None, None, None) == 1  # null pointers
    assert lib.moe_act_quant_nvfp4_f32(None, 4, 100, None, None, None, None) == 1
    assert lib.moe_act_quant_nvfp4_f32(None, 0, 128, None, None, None, None) == 0
    assert lib.moe_act_quant_nvfp4_f32(None, 4, 128, None, None, None, None) == 1
