"""Seeded synthetic inputs for one MoE FFN layer.

This module only draws numbers: token activations, router weights (with an
optional popularity bias) and stacked expert weights in the storage formats the
layer consumes.  It holds none of the layer's arithmetic, so both the CUDA path
and the CPU oracle can be fed from it without sharing any computation.

Storage formats (the layout the C-ABI documents):
  x         bf16  [m, H]
  router_w  fp32  [E, H]            router_bias fp32 [E] or None
  w1, w3    [E, I, H]   w2 [E, H, I]   (out, in) rows, stacked per expert
            bf16, or e4m3 codes (uint8) with fp32 scales per 128x128 block:
  s1, s3    fp32 [E, I/128, H/128]     s2 fp32 [E, H/128, I/128]
            or NVFP4: e2m1 codes packed two per byte (element 2j in the low
            nibble of byte j), w1, w3 uint8 [E, I, H/2], w2 uint8 [E, H, I/2],
            e4m3 block-scale codes per 16 inputs sb1, sb3 uint8 [E, I, H/16],
            sb2 uint8 [E, H, I/16], and one fp32 scale per expert matrix
            s1, s3, s2 fp32 [E]
  shared expert (optional): ws1, ws3 [Is, H], ws2 [H, Is] (+ ss1, ss3, ss2,
            and ssb1, ssb3, ssb2 for NVFP4; its ss* are then fp32 [1])
  shared_gate fp32 [H] (optional: the shared expert's sigmoid gate)

Every tensor has its own generator seeded from (seed, name, expert), so any one
expert can be regenerated alone and the draws do not depend on the device
order of generation.  fp8 weights are encoded with torch's own float8 cast
after scaling each 128x128 block by amax/448 (the block-scaled checkpoint
format); this is input preparation, not part of the layer's forward.  NVFP4
weights are drawn directly as codes: every 4-bit code uniform over its 16
values, block scales uniform over the e4m3 codes of [0.5, 4), and a per-matrix
scale of 0.02/6 times U(0.75, 1.25), so that the weights come out with a
standard deviation near 0.02.
"""
from __future__ import annotations

import dataclasses
import math

import torch

WEIGHT_STD = 0.02


@dataclasses.dataclass(frozen=True)
class LayerShape:
    hidden: int
    num_experts: int
    top_k: int
    inter: int
    shared_inter: int = 0
    fp8: bool = False
    # routing: "softmax" (renormalised over the k picks; a router bias is added
    # to the logits) or "sigmoid" (scores sigmoid(L); the bias is a correction
    # that only selects; weights are the picked scores, renormalised when
    # norm_topk_prob, times routed_scaling)
    scoring: str = "softmax"
    norm_topk_prob: bool = True
    routed_scaling: float = 1.0
    shared_gate: bool = False  # shared expert scaled by sigmoid(x . gate), gate fp32 [H]
    nvfp4: bool = False  # NVFP4 weights and activations (W4A4); exclusive with fp8

    @property
    def name(self) -> str:
        return (f"H{self.hidden}_E{self.num_experts}_k{self.top_k}_I{self.inter}"
                + (f"_S{self.shared_inter}" if self.shared_inter else "")
                + ("_fp8" if self.fp8 else ("_nvfp4" if self.nvfp4 else "_bf16"))
                + ("_sigmoid" if self.scoring == "sigmoid" else "")
                + ("_gated" if self.shared_gate else ""))


TINY = LayerShape(hidden=256, num_experts=8, top_k=2, inter=128)
QWEN3_30B_A3B = LayerShape(hidden=2048, num_experts=128, top_k=8, inter=768)
DEEPSEEK_V3 = LayerShape(hidden=7168, num_experts=256, top_k=8, inter=2048, shared_inter=2048, fp8=True)
# the same layer with its own router: sigmoid scores + correction bias, weights renormalised and scaled by 2.5
DEEPSEEK_V3_SIGMOID = dataclasses.replace(DEEPSEEK_V3, scoring="sigmoid", routed_scaling=2.5)
# a small layer whose shared expert is blended through a sigmoid gate
GATED_SHARED = LayerShape(hidden=512, num_experts=16, top_k=4, inter=256, shared_inter=256, shared_gate=True)
# the Qwen3 layer with NVFP4 experts, and a small NVFP4 layer with a shared expert
QWEN3_NVFP4 = dataclasses.replace(QWEN3_30B_A3B, nvfp4=True)
SMALL_NVFP4 = LayerShape(hidden=512, num_experts=16, top_k=4, inter=256, shared_inter=256, nvfp4=True)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: LayerShape
    ms: tuple
    router: str = "normal"  # "normal": N(0, 0.02); "uniform": U(-a, a) with std 0.02
    zipf_s: float = 0.0     # > 0: router bias making expert popularity Zipf(s)
    correction_std: float = 0.0  # > 0: sigmoid routing's correction bias ~ N(0, correction_std)


WORKLOADS = {
    "tiny": Workload("tiny", TINY, (16,)),
    "qwen3_decode": Workload("qwen3_decode", QWEN3_30B_A3B, (1, 4, 16, 64)),
    "qwen3_prefill": Workload("qwen3_prefill", QWEN3_30B_A3B, (512, 4096, 16384), router="uniform"),
    "deepseek_v3_fp8": Workload("deepseek_v3_fp8", DEEPSEEK_V3, (1, 16, 4096)),
    "qwen3_zipf": Workload("qwen3_zipf", QWEN3_30B_A3B, (8192,), zipf_s=1.2),
    "deepseek_v3_sigmoid": Workload("deepseek_v3_sigmoid", DEEPSEEK_V3_SIGMOID, (1, 16, 512), correction_std=0.01),
    "gated_shared": Workload("gated_shared", GATED_SHARED, (16, 512)),
    "qwen3_nvfp4": Workload("qwen3_nvfp4", QWEN3_NVFP4, (1, 16, 64)),
    "qwen3_nvfp4_prefill": Workload("qwen3_nvfp4_prefill", QWEN3_NVFP4, (512, 4096, 16384), router="uniform"),
    "small_nvfp4": Workload("small_nvfp4", SMALL_NVFP4, (16, 512)),
}


def _mix(*parts) -> int:
    """A stable 63-bit seed from ints and strings (FNV-1a over their bytes)."""
    h = 0xCBF29CE484222325
    for p in parts:
        data = p.encode() if isinstance(p, str) else int(p).to_bytes(8, "little", signed=True)
        for b in data + b"|":
            h ^= b
            h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h & 0x7FFFFFFFFFFFFFFF


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_mix(*parts))
    return g


def make_x(shape: LayerShape, m: int, seed: int = 0, device="cpu", stream_id: int = 0) -> torch.Tensor:
    """Token activations x ~ N(0, 1), bf16 [m, H]."""
    g = _gen(device, seed, "x", stream_id, m)
    return torch.randn(m, shape.hidden, generator=g, device=device).to(torch.bfloat16)


def make_router(shape: LayerShape, seed: int = 0, device="cpu", kind: str = "normal", zipf_s: float = 0.0,
                correction_std: float = 0.0):
    """Router weights fp32 [E, H] and an optional bias fp32 [E].

    kind "normal": N(0, 0.02).  kind "uniform": U(-sqrt(3)*0.02, +sqrt(3)*0.02),
    the uniform law with the same 0.02 standard deviation.  zipf_s > 0 adds
    bias[e] = -zipf_s * ln(rank[e]) with rank a seeded permutation of 1..E, so
    that softmax popularity falls off as rank^-s.  correction_std > 0 gives the
    sigmoid router's correction bias, bias[e] ~ N(0, correction_std).
    """
    E, H = shape.num_experts, shape.hidden
    g = _gen(device, seed, "router", kind)
    if kind == "normal":
        wr = torch.randn(E, H, generator=g, device=device) * WEIGHT_STD
    elif kind == "uniform":
        a = math.sqrt(3.0) * WEIGHT_STD
        wr = (torch.rand(E, H, generator=g, device=device) * 2.0 - 1.0) * a
    else:
        raise ValueError(f"unknown router kind {kind!r}")
    bias = None
    if correction_std > 0:
        gb = _gen(device, seed, "correction_bias")
        bias = (torch.randn(E, generator=gb, device=device) * correction_std).contiguous()
    if zipf_s > 0:
        gp = _gen("cpu", seed, "zipf_rank")
        rank = torch.randperm(E, generator=gp).to(torch.float64) + 1.0
        bias = (-zipf_s * torch.log(rank)).to(torch.float32).to(device)
    return wr.contiguous(), bias


def _encode_fp8_blocks(w: torch.Tensor):
    """Weight [R, C] fp32 -> (e4m3 codes uint8 [R, C], scales fp32 [R/128, C/128])."""
    R, C = w.shape
    rb, cb = (R + 127) // 128, (C + 127) // 128
    pad = torch.zeros(rb * 128, cb * 128, device=w.device, dtype=torch.float32)
    pad[:R, :C] = w
    blocks = pad.view(rb, 128, cb, 128)
    amax = blocks.abs().amax(dim=(1, 3))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (blocks / scale[:, None, :, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    return q.reshape(rb * 128, cb * 128)[:R, :C].contiguous(), scale.contiguous()


def _weight(shape: LayerShape, R: int, C: int, device, *parts):
    g = _gen(device, *parts)
    w = torch.randn(R, C, generator=g, device=device) * WEIGHT_STD
    if shape.fp8:
        return _encode_fp8_blocks(w)
    return w.to(torch.bfloat16), None


def _nvfp4_weight(R: int, C: int, device, *parts):
    """Random NVFP4 matrix [R, C] -> (packed codes uint8 [R, C/2], block-scale
    codes uint8 [R, C/16], matrix scale fp32 [1])."""
    g = _gen(device, *parts)
    q = torch.randint(0, 256, (R, C // 2), generator=g, device=device, dtype=torch.int32).to(torch.uint8)
    # e4m3 codes 0x30..0x47: exponent fields 6..8, the values [0.5, 4)
    sb = torch.randint(0x30, 0x48, (R, C // 16), generator=g, device=device, dtype=torch.int32).to(torch.uint8)
    u = torch.rand(1, generator=g, device=device)
    return q, sb, (WEIGHT_STD / 6.0) * (0.75 + 0.5 * u)


def make_experts(shape: LayerShape, seed: int = 0, device="cpu", experts=None) -> dict:
    """Stacked expert weights (and the shared expert's, when the shape has one).

    experts: optional iterable of expert ids to generate; the others are left
    zero (used to build only what a sampled oracle check needs).
    """
    E, H, I = shape.num_experts, shape.hidden, shape.inter
    if shape.nvfp4:
        return _make_experts_nvfp4(shape, seed, device, experts)
    wdt = torch.uint8 if shape.fp8 else torch.bfloat16
    out = {
        "w1": torch.zeros(E, I, H, dtype=wdt, device=device),
        "w3": torch.zeros(E, I, H, dtype=wdt, device=device),
        "w2": torch.zeros(E, H, I, dtype=wdt, device=device),
    }
    if shape.fp8:
        ib, hb = (I + 127) // 128, (H + 127) // 128
        out["s1"] = torch.zeros(E, ib, hb, dtype=torch.float32, device=device)
        out["s3"] = torch.zeros(E, ib, hb, dtype=torch.float32, device=device)
        out["s2"] = torch.zeros(E, hb, ib, dtype=torch.float32, device=device)
    todo = range(E) if experts is None else sorted(set(int(e) for e in experts))
    for e in todo:
        for name, (R, C) in (("w1", (I, H)), ("w3", (I, H)), ("w2", (H, I))):
            q, s = _weight(shape, R, C, device, seed, name, e)
            out[name][e].copy_(q)
            if s is not None:
                out["s" + name[1]][e].copy_(s)
    if shape.shared_inter:
        Is = shape.shared_inter
        for name, (R, C) in (("ws1", (Is, H)), ("ws3", (Is, H)), ("ws2", (H, Is))):
            q, s = _weight(shape, R, C, device, seed, name, -1)
            out[name] = q.contiguous()
            if s is not None:
                out["ss" + name[2]] = s
    if shape.shared_gate:
        g = _gen(device, seed, "shared_gate")
        out["shared_gate"] = (torch.randn(H, generator=g, device=device) * WEIGHT_STD).contiguous()
    return out


def _make_experts_nvfp4(shape: LayerShape, seed: int, device, experts) -> dict:
    E, H, I = shape.num_experts, shape.hidden, shape.inter
    u8, f32 = torch.uint8, torch.float32
    out = {
        "w1": torch.zeros(E, I, H // 2, dtype=u8, device=device),
        "w3": torch.zeros(E, I, H // 2, dtype=u8, device=device),
        "w2": torch.zeros(E, H, I // 2, dtype=u8, device=device),
        "sb1": torch.zeros(E, I, H // 16, dtype=u8, device=device),
        "sb3": torch.zeros(E, I, H // 16, dtype=u8, device=device),
        "sb2": torch.zeros(E, H, I // 16, dtype=u8, device=device),
        "s1": torch.zeros(E, dtype=f32, device=device),
        "s3": torch.zeros(E, dtype=f32, device=device),
        "s2": torch.zeros(E, dtype=f32, device=device),
    }
    todo = range(E) if experts is None else sorted(set(int(e) for e in experts))
    for e in todo:
        for name, (R, C) in (("w1", (I, H)), ("w3", (I, H)), ("w2", (H, I))):
            q, sb, sc = _nvfp4_weight(R, C, device, seed, name, e)
            out[name][e].copy_(q)
            out["sb" + name[1]][e].copy_(sb)
            out["s" + name[1]][e:e + 1].copy_(sc)
    if shape.shared_inter:
        Is = shape.shared_inter
        for name, (R, C) in (("ws1", (Is, H)), ("ws3", (Is, H)), ("ws2", (H, Is))):
            q, sb, sc = _nvfp4_weight(R, C, device, seed, name, -1)
            out[name] = q.contiguous()
            out["ssb" + name[2]] = sb.contiguous()
            out["ss" + name[2]] = sc.contiguous()
    if shape.shared_gate:
        g = _gen(device, seed, "shared_gate")
        out["shared_gate"] = (torch.randn(H, generator=g, device=device) * WEIGHT_STD).contiguous()
    return out


def make_layer(workload: Workload, seed: int = 0, device="cpu", experts=None) -> dict:
    """Router + experts for a workload, as one dict of tensors."""
    wr, bias = make_router(workload.shape, seed, device, workload.router, workload.zipf_s, workload.correction_std)
    layer = make_experts(workload.shape, seed, device, experts)
    layer["router_w"] = wr
    layer["router_bias"] = bias
    return layer
