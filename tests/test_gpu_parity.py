"""GPU parity: the CUDA path (through the C-ABI) against the CPU oracle.

Integer work (permute, e4m3 activation codes) is compared bit-exactly;
expert ids exactly except at oracle near-ties (margin 1e-4); routing weights
to 2e-5; layer outputs by relative L2 over [rows, H]: 1e-2 for bf16 weights,
2e-2 for fp8 and NVFP4 block-scaled weights (the oracle emulates their
activation quantisation, so the remaining gap is accumulation order).  Full-size workloads run in the launch
configuration the benchmark times, with the oracle evaluated on sampled rows.
"""
import dataclasses

import numpy as np
import pytest
import torch

from mixture_experts_ffn_gemv_gb300 import inputs as I
from _parity import (TOL, check_ids, forced_routing, max_swapped, oracle_rows, rel_l2, selection_keys,
                     to_np, tol)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_gemv_gb300 import binding
    binding.load_library()
    return torch.device("cuda", 0)


_CACHE = {}


def layer_for(workload, device, seed=0):
    """Device tensors of a workload's layer (one big layer cached at a time)."""
    key = (workload.name, workload.shape, seed)
    if key not in _CACHE:
        _CACHE.clear()
        torch.cuda.empty_cache()
        from mixture_experts_ffn_gemv_gb300 import binding
        tensors = I.make_layer(workload, seed=seed, device=device)
        _CACHE[key] = (tensors, binding.MoeLayer(workload.shape, tensors))
    return _CACHE[key]


def oracle_route(oracle_mod, shape, tensors, x):
    host = {"router_w": tensors["router_w"].cpu(),
            "router_bias": None if tensors["router_bias"] is None else tensors["router_bias"].cpu()}
    return oracle_mod.route(shape, host, x.cpu())


def sample_rows(m, n=48, seed=0):
    if m <= n:
        return np.arange(m)
    rng = np.random.default_rng(seed)
    pick = rng.choice(np.arange(1, m - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, m - 1], pick]))


SMALL_FP8 = I.LayerShape(hidden=512, num_experts=8, top_k=2, inter=512, shared_inter=512, fp8=True)
MEDIUM_BF16 = I.LayerShape(hidden=512, num_experts=16, top_k=4, inter=256)
ODD_E = I.LayerShape(hidden=256, num_experts=40, top_k=3, inter=128)


# ------------------------------------------------------------------ activations

@pytest.mark.parametrize("H", [384, 512, 7168])
def test_act_quant_fp8_bitwise(cuda, oracle_mod, H):
    """Rows of 3 blocks (one warp per block) and of 4 and 56 (four blocks per warp)."""
    from mixture_experts_ffn_gemv_gb300 import binding
    x = I.make_x(dataclasses.replace(SMALL_FP8, hidden=H), 37, seed=21, device=cuda)
    x[3, 128:256] = 0            # an all-zero block
    x[5, :128] *= 1e-3           # small magnitudes (subnormal codes)
    x[6, 7] = -0.0
    x[7, 0] = 3e4                # one large value dominating its block
    codes, scales = binding.moe_act_quant_fp8(x)
    torch.cuda.synchronize()
    xc = x.cpu()
    for r in range(x.shape[0]):
        q, s, _ = oracle_mod.act_quant(xc[r].float().numpy())
        assert np.array_equal(codes[r].cpu().numpy(), q), f"row {r}"
        assert np.array_equal(scales[r].cpu().numpy(), s), f"row {r}"


def test_act_quant_fp8_midpoints(cuda, oracle_mod):
    """Blocks whose amax is 448 * 2^j (a power-of-two scale), so every
    quotient is exact: values on e4m3 rounding midpoints (ties to even,
    normal and subnormal codes) and next to them, bit for bit."""
    from mixture_experts_ffn_gemv_gb300 import binding
    rng = np.random.default_rng(31)
    e4 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    pos = np.sort(np.unique(e4[np.isfinite(e4) & (e4 > 0)]))
    vals = np.concatenate([[0.0], pos])
    mids = (vals[:-1] + vals[1:]) / 2                       # every midpoint below 448
    rows, H = 16, 1024
    x = np.zeros((rows, H), np.float32)
    for r in range(rows):
        for b in range(H // 128):
            j = int(rng.integers(-4, 4))
            blk = rng.choice(mids, 128) * rng.choice([-1.0, 1.0], 128)
            blk[rng.integers(0, 128)] = 448.0                  # the block's amax
            x[r, 128 * b:128 * b + 128] = blk * 2.0 ** j
    xb = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(xb.float().numpy(), x)           # the midpoints are exact in bf16
    codes, scales = binding.moe_act_quant_fp8(xb.to(cuda))
    torch.cuda.synchronize()
    for r in range(rows):
        q, sc, _ = oracle_mod.act_quant(x[r])
        assert np.array_equal(codes[r].cpu().numpy(), q), f"row {r}"
        assert np.array_equal(scales[r].cpu().numpy(), sc), f"row {r}"


@pytest.mark.parametrize("n,rows", [(768, 23), (2048, 23), (7168, 23), (768, 1100), (2048, 1100), (256, 1100),
                                    (512, 1100), (1536, 1100), (7168, 1100)])
def test_act_quant_nvfp4_bitwise(cuda, oracle_mod, n, rows):
    """Both launch shapes: four warps per row (few rows), one warp per row
    (many), over row lengths of 16 to 448 blocks."""
    from mixture_experts_ffn_gemv_gb300 import binding
    shape = I.LayerShape(hidden=n, num_experts=1, top_k=1, inter=256)
    x = I.make_x(shape, rows, seed=22, device=cuda)
    x[1] = 0                     # an all-zero row: g = 1, codes and scales 0
    x[2, 16:32] = 0              # an all-zero block
    x[3, :n // 2] *= 1e-4        # blocks far below the row's amax (small / zero scales)
    x[4, 5] = 3e4                # one value sets the row scale
    x[5, 9] = -0.0
    x[6] = 1.0                   # every block at the row's amax
    codes, sb, g = binding.moe_act_quant_nvfp4(x)
    torch.cuda.synchronize()
    q, r_sb, r_g, _ = oracle_mod.nvfp4_quant(x.cpu().float().numpy())
    assert np.array_equal(g.cpu().numpy(), r_g)
    assert np.array_equal(sb.cpu().numpy(), r_sb)
    assert np.array_equal(codes.cpu().numpy(), q)


def _midpoint_rows(n, rows, seed):
    """fp32 rows whose quotients v / scale land on e2m1 rounding midpoints
    (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5) and one float either side of them,
    for power-of-two scales (exact ties) and arbitrary ones (near ties).  The
    scale a block gets is worked out with the quantisation's own fp32 steps
    (round-to-nearest numpy float32 arithmetic) so that the constructed
    values hit the intended quotients."""
    rng = np.random.default_rng(seed)
    f32 = np.float32
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], f32)
    e4m3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    e4m3_pos = np.sort(np.unique(e4m3[np.isfinite(e4m3) & (e4m3 > 0)]))

    def e4m3_round(x):  # nearest positive e4m3 value (ties are not hit here)
        return e4m3_pos[np.argmin(np.abs(e4m3_pos.astype(np.float64) - float(x)))]

    out = np.zeros((rows, n), f32)
    for r in range(rows):
        amax = f32(2688.0) if r % 2 == 0 else f32(rng.uniform(0.5, 4000.0))
        gs = f32(amax / f32(2688.0))
        out[r, 0] = amax
        for b in range(1, n // 16):
            bmax = f32(6.0 * 2.0 ** rng.integers(-3, 3)) if r % 2 == 0 else f32(rng.uniform(0.01, 1.0) * amax)
            sc = e4m3_round(f32(bmax / f32(f32(6.0) * gs)))
            scale = f32(f32(sc) * gs)
            t = mids[rng.integers(0, len(mids), 15)] * rng.choice([f32(-1), f32(1)], 15)
            v = (t * scale).astype(f32)
            step = rng.integers(-1, 2, 15)
            v = np.where(step < 0, np.nextafter(v, f32(-np.inf)), np.where(step > 0, np.nextafter(v, f32(np.inf)), v))
            blk = np.concatenate([[bmax], v]).astype(f32)
            out[r, 16 * b:16 * b + 16] = blk[rng.permutation(16)]
    return out


@pytest.mark.parametrize("n,rows", [(256, 40), (768, 1100)])
def test_act_quant_nvfp4_f32_bitwise(cuda, oracle_mod, n, rows):
    """The fp32 quantiser (the down projection's input) against the oracle,
    bit for bit, on random rows and on rows built to put quotients on and
    next to the e2m1 rounding midpoints."""
    from mixture_experts_ffn_gemv_gb300 import binding
    rng = np.random.default_rng(23)
    x = rng.standard_normal((rows, n)).astype(np.float32) * rng.uniform(0.1, 10.0, (rows, 1)).astype(np.float32)
    x[1] = 0
    x[2, 16:32] = 0
    x[3, :n // 2] *= 1e-5
    x[5, 9] = -0.0
    x[6] = 1.0
    x[7] = 0                     # subnormal row scale; the second block's scale is subnormal
    x[7, :16] = 1e-36            # too, so its reciprocal overflows and every quotient is divided
    x[7, 16:32] = rng.uniform(-1, 1, 16).astype(np.float32) * np.float32(1e-36 / 256)
    x[8:24] = _midpoint_rows(n, 16, seed=n)
    xd = torch.from_numpy(x).to(cuda)
    codes, sb, g = binding.moe_act_quant_nvfp4(xd)
    torch.cuda.synchronize()
    q, r_sb, r_g, _ = oracle_mod.nvfp4_quant(x)
    assert np.array_equal(g.cpu().numpy(), r_g)
    assert np.array_equal(sb.cpu().numpy(), r_sb)
    bad = np.nonzero(codes.cpu().numpy() != q)
    assert bad[0].size == 0, f"{bad[0].size} code bytes differ, first at row {bad[0][0]} byte {bad[1][0]}"


def test_act_quant_nvfp4_bf16_midpoints(cuda, oracle_mod):
    """bf16 rows on exact e2m1 rounding midpoints (power-of-two scales)."""
    from mixture_experts_ffn_gemv_gb300 import binding
    x = _midpoint_rows(512, 32, seed=5)[::2]          # the power-of-two rows: exact in bf16
    xb = torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)
    codes, sb, g = binding.moe_act_quant_nvfp4(xb.to(cuda))
    torch.cuda.synchronize()
    q, r_sb, r_g, _ = oracle_mod.nvfp4_quant(xb.float().numpy())
    assert np.array_equal(g.cpu().numpy(), r_g)
    assert np.array_equal(sb.cpu().numpy(), r_sb)
    assert np.array_equal(codes.cpu().numpy(), q)


# ------------------------------------------------------------------ permute

@pytest.mark.parametrize("m,k,E,kind", [
    (1, 8, 128, "random"), (16, 2, 8, "random"), (700, 8, 128, "random"),   # 2 chunks + ragged tail
    (600, 8, 40, "random"), (300, 4, 256, "one_expert"), (4096, 8, 256, "random"),
    (16384, 8, 128, "skewed"),
])
def test_permute_exact(cuda, oracle_mod, m, k, E, kind):
    from mixture_experts_ffn_gemv_gb300 import binding
    rng = np.random.default_rng(m * 7 + E)
    if kind == "random":
        ids = np.stack([rng.permutation(E)[:k] for _ in range(m)])
    elif kind == "one_expert":  # expert 3 in every token's slot 0
        ids = np.stack([np.concatenate([[3], rng.permutation([e for e in range(E) if e != 3])[:k - 1]])
                        for _ in range(m)])
    else:  # Zipf-like popularity
        p = 1.0 / np.arange(1, E + 1) ** 1.2
        p /= p.sum()
        ids = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(m)])
    ids = ids.astype(np.int32)
    shape = I.LayerShape(hidden=256, num_experts=E, top_k=k, inter=128)
    # a layer handle of the right E / k over zero weights (only the permute runs)
    dummy = {n: torch.zeros(E, 128, 256, dtype=torch.bfloat16, device=cuda) for n in ("w1", "w3")}
    dummy["w2"] = torch.zeros(E, 256, 128, dtype=torch.bfloat16, device=cuda)
    layer = binding.MoeLayer(shape, dummy)
    off, sp, sl = layer.moe_permute(torch.from_numpy(ids).to(cuda))
    torch.cuda.synchronize()
    r_off, r_sp, r_sl = oracle_mod.permute(ids, E)
    assert np.array_equal(off.cpu().numpy(), r_off)
    assert np.array_equal(sp.cpu().numpy(), r_sp)
    assert np.array_equal(sl.cpu().numpy(), r_sl)
    assert layer.device_status() == 0


# ------------------------------------------------------------------ routing

ROUTE_CASES = [("tiny", 16), ("qwen3_decode", 1), ("qwen3_decode", 64), ("qwen3_prefill", 4096),
               ("deepseek_v3_fp8", 16), ("qwen3_zipf", 8192)]


@pytest.mark.parametrize("wl_name,m", ROUTE_CASES)
def test_route_parity(cuda, oracle_mod, wl_name, m):
    wl = I.WORKLOADS[wl_name]
    tensors, layer = layer_for(wl, cuda)
    x = I.make_x(wl.shape, m, device=cuda)
    ids, w, logits = layer.moe_route(x, tensors["router_w"], tensors["router_bias"], logits=True)
    torch.cuda.synchronize()
    L, r_ids, r_w, margin = oracle_route(oracle_mod, wl.shape, tensors, x)
    scale = np.abs(L).max()
    assert np.abs(to_np(logits) - L).max() <= 1e-5 * max(scale, 1.0)
    swapped, bad = check_ids(to_np(ids), r_ids, L)
    assert not bad, bad[:5]
    same = np.ones(m, bool)
    same[swapped] = False
    assert np.abs(to_np(w)[same] - r_w[same]).max() < 2e-5
    assert np.abs(to_np(w).astype(np.float64).sum(1) - 1).max() < 1e-5
    assert len(swapped) <= max(2, m // 200)


@pytest.mark.parametrize("m", [1, 16, 100, 512])
def test_route_parity_sigmoid_correction_bias(cuda, oracle_mod, m):
    """The sigmoid + correction-bias router (DeepSeek-V3 shape, routed scaling
    2.5): raw logits, ids by score + bias (margin rule on those keys), weights
    the renormalised pre-bias scores times 2.5.  m = 1, 16 take the fused
    decode kernel, 100 and 512 the router + top-k kernels."""
    wl = I.WORKLOADS["deepseek_v3_sigmoid"]
    shape = wl.shape
    x = I.make_x(shape, m, seed=91, device=cuda)
    wr, bias = I.make_router(shape, seed=91, device=cuda, correction_std=wl.correction_std)
    from mixture_experts_ffn_gemv_gb300 import binding
    small = dataclasses.replace(shape, inter=512, shared_inter=0)  # only the router matters here
    zeros = {"w1": torch.zeros(shape.num_experts, 512, shape.hidden, dtype=torch.uint8, device=cuda),
             "w3": torch.zeros(shape.num_experts, 512, shape.hidden, dtype=torch.uint8, device=cuda),
             "w2": torch.zeros(shape.num_experts, shape.hidden, 512, dtype=torch.uint8, device=cuda)}
    for n, (r, c) in (("s1", (4, shape.hidden // 128)), ("s3", (4, shape.hidden // 128)), ("s2", (shape.hidden // 128, 4))):
        zeros[n] = torch.ones(shape.num_experts, r, c, dtype=torch.float32, device=cuda)
    layer = binding.MoeLayer(small, zeros)
    ids, w, logits = layer.moe_route(x, wr, bias, logits=True)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    L, r_ids, r_w, _ = oracle_mod.route(small, {"router_w": wr.cpu(), "router_bias": bias.cpu()}, x.cpu())
    assert np.abs(to_np(logits) - L).max() <= 1e-5 * max(np.abs(L).max(), 1.0)  # no bias in the logits
    swapped, bad = check_ids(to_np(ids), r_ids, selection_keys(small, L, bias))
    assert not bad, bad[:5]
    same = np.ones(m, bool)
    same[swapped] = False
    assert np.abs(to_np(w)[same] - r_w[same]).max() < 2e-5 * shape.routed_scaling
    assert np.abs(to_np(w).astype(np.float64).sum(1) - shape.routed_scaling).max() < 1e-5 * shape.routed_scaling


@pytest.mark.parametrize("arm", ["gemv", "gemm"])
@pytest.mark.parametrize("m", [5, 16, 300])
def test_whole_layer_gated_shared_expert(cuda, oracle_mod, arm, m):
    """The shared expert blended through its sigmoid gate (forward_prefill step
    8), through moe_forward on both arms, against the oracle."""
    from mixture_experts_ffn_gemv_gb300 import binding
    shape = I.GATED_SHARED
    tensors, x = _small_case(shape, m, seed=93, device=cuda)
    host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in tensors.items()}
    ref = oracle_mod.reference(shape, host, x.cpu())
    layer = binding.MoeLayer(shape, tensors)
    out, ids, w = layer.moe_forward(x, tensors["router_w"], arm=arm, return_routing=True)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    swapped, bad = check_ids(to_np(ids), ref["ids"], ref["logits"])
    assert not bad, bad[:5]
    assert len(swapped) <= max_swapped(m)
    f_ids, f_w = forced_routing(oracle_mod, shape, ref["logits"], ref["ids"], ref["w"], to_np(ids), swapped)
    want = oracle_mod.moe_forward(shape, host, x.cpu(), f_ids, f_w)
    assert rel_l2(to_np(out), want) < TOL[False]


def _bf16_np(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("arm", ["gemv", "gemm"])
@pytest.mark.parametrize("shape,m", [(MEDIUM_BF16, 16), (MEDIUM_BF16, 300), (SMALL_FP8, 24), (SMALL_FP8, 200),
                                     (I.GATED_SHARED, 40)])
def test_forward_residual_rmsnorm_tail(cuda, oracle_mod, arm, shape, m):
    """The layer tail in the combine: with a zero residual the new residual is
    moe_forward's output bit for bit (the same fp32 sum rounded once); with a
    random one it is that sum added in fp32 and rounded; norm_out equals the
    oracle's RMSNorm of the new residual to the last bf16 bit (rare ties)."""
    from mixture_experts_ffn_gemv_gb300 import binding
    tensors, x = _small_case(shape, m, seed=97, device=cuda)
    layer = binding.MoeLayer(shape, tensors)
    g = torch.Generator(device=cuda).manual_seed(97)
    norm_w = (torch.randn(shape.hidden, generator=g, device=cuda) * 0.2 + 1.0).contiguous()
    eps = 1e-6
    try:
        out = layer.moe_forward(x, tensors["router_w"], tensors["router_bias"], arm=arm)
    except binding.MoeError as e:
        if e.status == binding.MOE_ERR_UNSUPPORTED and arm == "gemm":
            pytest.skip("grouped GEMM arm not available for this shape")
        raise
    res0 = torch.zeros(m, shape.hidden, dtype=torch.bfloat16, device=cuda)
    n0 = layer.moe_forward_residual_rmsnorm(x, tensors["router_w"], res0, norm_w, eps, tensors["router_bias"], arm=arm)
    res1_in = torch.randn(m, shape.hidden, generator=g, device=cuda).to(torch.bfloat16)
    res1 = res1_in.clone()
    n1 = layer.moe_forward_residual_rmsnorm(x, tensors["router_w"], res1, norm_w, eps, tensors["router_bias"], arm=arm)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    assert np.array_equal(_bf16_np(res0), _bf16_np(out))
    want1 = res1_in.float() + out.float()  # out is the same sum rounded: within half a bf16 ulp of it
    assert ((res1.float() - want1).abs() <= 2.0 ** -8 * (want1.abs() + out.float().abs()) + 1e-30).all()
    for res, normed in ((res0, n0), (res1, n1)):
        _, ref = oracle_mod.residual_rmsnorm(np.zeros((m, shape.hidden), np.float32), _bf16_np(res),
                                             norm_w.cpu().numpy(), eps, fp64=True)
        got = normed.float().cpu()
        exp = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float()
        rel = ((got - exp).abs() / exp.abs().clamp_min(1e-30))
        assert rel.max().item() <= 2.0 ** -7
        assert (got != exp).float().mean().item() < 0.01


@pytest.mark.parametrize("shape,m", [(I.TINY, 300), (ODD_E, 500), (MEDIUM_BF16, 129)])
def test_route_tensor_core_path_odd_shapes(cuda, oracle_mod, shape, m):
    """m > 64 takes the tensor-core router (bf16 x3 split of the fp32 weight);
    E of 8, 40 and 16 exercise the padded N of its MMA."""
    from mixture_experts_ffn_gemv_gb300 import binding
    tensors, x = _small_case(shape, m, seed=61, device=cuda)
    layer = binding.MoeLayer(shape, tensors)
    ids, w, logits = layer.moe_route(x, tensors["router_w"], logits=True)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    L, r_ids, r_w, _ = oracle_route(oracle_mod, shape, tensors, x)
    assert np.abs(to_np(logits) - L).max() <= 1e-5 * max(np.abs(L).max(), 1.0)
    swapped, bad = check_ids(to_np(ids), r_ids, L)
    assert not bad, bad[:5]


# ------------------------------------------------------------------ experts (given routing)

def _small_case(shape, m, seed, device):
    wl = I.Workload("t", shape, (m,))
    tensors = I.make_layer(wl, seed=seed, device=device)
    x = I.make_x(shape, m, seed=seed, device=device)
    return tensors, x


@pytest.mark.parametrize("arm", ["gemv", "gemm"])
@pytest.mark.parametrize("shape,m", [(I.TINY, 16), (I.TINY, 1), (MEDIUM_BF16, 300), (ODD_E, 77),
                                     (SMALL_FP8, 24), (SMALL_FP8, 1), (SMALL_FP8, 200),
                                     (I.SMALL_NVFP4, 1), (I.SMALL_NVFP4, 24), (I.SMALL_NVFP4, 200)])
def test_experts_given_oracle_routing(cuda, oracle_mod, arm, shape, m):
    from mixture_experts_ffn_gemv_gb300 import binding
    tensors, x = _small_case(shape, m, seed=31, device=cuda)
    host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in tensors.items()}
    ref = oracle_mod.reference(shape, host, x.cpu())
    layer = binding.MoeLayer(shape, tensors)
    try:
        out = layer.moe_experts(x, torch.from_numpy(ref["ids"]).to(cuda), torch.from_numpy(ref["w"]).to(cuda),
                                arm=arm)
    except binding.MoeError as e:
        if e.status == binding.MOE_ERR_UNSUPPORTED and arm == "gemm":
            pytest.skip("grouped GEMM arm not available for this shape")
        raise
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    err = rel_l2(to_np(out), ref["out"])
    assert err < tol(shape), err


# few experts, many rows each: the bf16 gate/up GEMM runs on CTA pairs
# (256-row tiles over two SMs) once the rows average 256 per group
PAIR_BF16 = I.LayerShape(hidden=512, num_experts=4, top_k=2, inter=256)
PAIR_SHARED = I.LayerShape(hidden=512, num_experts=4, top_k=1, inter=256, shared_inter=256)


@pytest.mark.parametrize("shape,m", [(PAIR_BF16, 600), (PAIR_BF16, 1000), (PAIR_SHARED, 900)])
def test_gateup_on_cta_pairs(cuda, oracle_mod, shape, m):
    """Groups of 300-500 rows: two or three 128-row m-tiles per pair tile, so
    some pairs have a peer CTA with no rows; every row against the oracle."""
    from mixture_experts_ffn_gemv_gb300 import binding
    tensors, x = _small_case(shape, m, seed=141, device=cuda)
    host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in tensors.items()}
    ref = oracle_mod.reference(shape, host, x.cpu())
    layer = binding.MoeLayer(shape, tensors)
    out, ids, w = layer.moe_forward(x, tensors["router_w"], arm="gemm", return_routing=True)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    swapped, bad = check_ids(to_np(ids), ref["ids"], ref["logits"])
    assert not bad, bad[:5]
    assert len(swapped) <= max_swapped(m)
    f_ids, f_w = forced_routing(oracle_mod, shape, ref["logits"], ref["ids"], ref["w"], to_np(ids), swapped)
    want = oracle_mod.moe_forward(shape, host, x.cpu(), f_ids, f_w)
    assert rel_l2(to_np(out), want) < TOL[False]


# Rows per expert chosen to cover every way a group's rows fill the CTA-pair
# tiles (256 rows over two CTAs):
# - 1, 17 and 128 rows: one pair tile whose peer CTA has no row;
# - 129: the peer has one row;
# - 257 and 770: full pairs, then a tile with 1 or 2 rows;
# - 384 and 385: a full pair, then a tile with 128 or 129 rows.
# The shared expert's 2071 rows end in a 23-row tile.  bf16: I = 384 is an odd
# count of 128-column n-tiles; NVFP4 (K in blocks of 256): I = 512.
PAIR_EDGES = I.LayerShape(hidden=512, num_experts=8, top_k=1, inter=384, shared_inter=384)
PAIR_EDGES_NVFP4 = I.LayerShape(hidden=512, num_experts=8, top_k=1, inter=512, shared_inter=512, nvfp4=True)
PAIR_EDGES_COUNTS = (1, 17, 128, 129, 257, 384, 385, 770)


@pytest.mark.parametrize("shape", [PAIR_EDGES, PAIR_EDGES_NVFP4], ids=["bf16", "nvfp4"])
def test_gateup_pair_group_edges(cuda, oracle_mod, shape):
    """Every row of a layer whose groups end in each kind of pair tile, with
    caller-given routing, against the oracle row by row (the bf16 GEMMs run on
    CTA pairs at these row counts; the NVFP4 case covers the same ragged
    groups on its one-CTA tiles)."""
    from mixture_experts_ffn_gemv_gb300 import binding
    m = sum(PAIR_EDGES_COUNTS)
    tensors, x = _small_case(shape, m, seed=143, device=cuda)
    gen = np.random.default_rng(143)
    ids = gen.permutation(np.repeat(np.arange(8, dtype=np.int32), PAIR_EDGES_COUNTS)).reshape(m, 1)
    w = gen.uniform(0.5, 1.0, (m, 1)).astype(np.float32)
    layer = binding.MoeLayer(shape, tensors)
    out = layer.moe_experts(x, torch.from_numpy(ids).to(cuda), torch.from_numpy(w).to(cuda), arm="gemm")
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in tensors.items()}
    want = oracle_mod.moe_forward(shape, host, x.cpu(), ids, w)
    got = to_np(out).astype(np.float64)
    row_err = np.linalg.norm(got - want, axis=1) / np.maximum(np.linalg.norm(want, axis=1), 1e-30)
    assert rel_l2(got, want) < tol(shape)
    assert row_err.max() < 3 * tol(shape), (int(row_err.argmax()), float(row_err.max()))


SHARED_BF16 = I.LayerShape(hidden=512, num_experts=16, top_k=4, inter=256, shared_inter=256)
TOP1 = I.LayerShape(hidden=256, num_experts=12, top_k=1, inter=128)


@pytest.mark.parametrize("arm", ["gemv", "gemm"])
@pytest.mark.parametrize("shape,m", [(SHARED_BF16, 5), (SHARED_BF16, 260), (TOP1, 37), (TOP1, 400)])
def test_whole_layer_shared_bf16_and_top1(cuda, oracle_mod, arm, shape, m):
    """A bf16 layer with a shared expert (group E of every kernel) and a top-1
    layer, through moe_forward on both arms, against the oracle."""
    from mixture_experts_ffn_gemv_gb300 import binding
    tensors, x = _small_case(shape, m, seed=71, device=cuda)
    host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in tensors.items()}
    ref = oracle_mod.reference(shape, host, x.cpu())
    layer = binding.MoeLayer(shape, tensors)
    out, ids, w = layer.moe_forward(x, tensors["router_w"], arm=arm, return_routing=True)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    swapped, bad = check_ids(to_np(ids), ref["ids"], ref["logits"])
    assert not bad, bad[:5]
    assert len(swapped) <= max_swapped(m)
    f_ids, f_w = forced_routing(oracle_mod, shape, ref["logits"], ref["ids"], ref["w"], to_np(ids), swapped)
    want = oracle_mod.moe_forward(shape, host, x.cpu(), f_ids, f_w)
    assert rel_l2(to_np(out), want) < TOL[False]


@pytest.mark.parametrize("m", [1, 50, 200])
def test_route_and_permute_at_the_largest_expert_count(cuda, oracle_mod, m):
    """E = 1024 experts and top_k = 32: the widest top-k lanes (32 logits per
    lane) and the permute's largest per-warp tables."""
    from mixture_experts_ffn_gemv_gb300 import binding
    shape = I.LayerShape(hidden=256, num_experts=1024, top_k=32, inter=128)
    x = I.make_x(shape, m, seed=81, device=cuda)
    wr, _ = I.make_router(shape, seed=81, device=cuda)
    zeros = {n: torch.zeros(1024, 128, 256, dtype=torch.bfloat16, device=cuda) for n in ("w1", "w3")}
    zeros["w2"] = torch.zeros(1024, 256, 128, dtype=torch.bfloat16, device=cuda)
    layer = binding.MoeLayer(shape, zeros)
    ids, w, logits = layer.moe_route(x, wr, logits=True)
    L, r_ids, r_w, _ = oracle_mod.route(shape, {"router_w": wr.cpu(), "router_bias": None}, x.cpu())
    off, sp, sl = layer.moe_permute(torch.from_numpy(r_ids).to(cuda))  # both sides permute the oracle's ids
    torch.cuda.synchronize()
    swapped, bad = check_ids(to_np(ids), r_ids, L)
    assert not bad, bad[:5]
    r_off, r_sp, r_sl = oracle_mod.permute(r_ids, 1024)
    assert np.array_equal(off.cpu().numpy(), r_off)
    assert np.array_equal(sp.cpu().numpy(), r_sp)
    assert np.array_equal(sl.cpu().numpy(), r_sl)
    assert np.abs(to_np(w).astype(np.float64).sum(1) - 1).max() < 1e-5


def test_prepared_router_weight(cuda):
    """moe_router_prepare splits the router weight once; calls passing that
    pointer skip the split and give identical results, a weight rewritten in
    place needs (and gets) a new preparation, and forgetting it restores the
    per-call split."""
    from mixture_experts_ffn_gemv_gb300 import binding
    shape = MEDIUM_BF16
    tensors, x = _small_case(shape, 300, seed=151, device=cuda)  # m > 64: the tensor-core router
    layer = binding.MoeLayer(shape, tensors)
    wr = tensors["router_w"]
    out0, ids0, w0 = layer.moe_forward(x, wr, return_routing=True)
    n0 = layer.last_launch_count()
    layer.prepare_router(wr)
    out1, ids1, w1 = layer.moe_forward(x, wr, return_routing=True)
    assert layer.last_launch_count() == n0 - 1  # no split
    assert torch.equal(out0, out1) and torch.equal(ids0, ids1) and torch.equal(w0, w1)
    wr.mul_(1.5)  # rewritten in place: prepare again
    layer.prepare_router(wr)
    out2 = layer.moe_forward(x, wr)
    fresh = binding.MoeLayer(shape, tensors).moe_forward(x, wr)
    assert torch.equal(out2, fresh)
    other = wr.clone()  # another pointer: split per call
    assert torch.equal(layer.moe_forward(x, other), fresh)
    layer.prepare_router(None)
    assert torch.equal(layer.moe_forward(x, wr), fresh)
    assert layer.device_status() == 0


# ------------------------------------------------------------------ whole layer, full sizes

FULL_CASES = [("tiny", 16)] + [("qwen3_decode", m) for m in (1, 2, 4, 16, 64)] + \
             [("qwen3_prefill", m) for m in (512, 4096, 16384)] + \
             [("deepseek_v3_fp8", m) for m in (1, 16, 4096)] + [("qwen3_zipf", 8192)] + \
             [("deepseek_v3_sigmoid", m) for m in (1, 16, 512)] + [("gated_shared", m) for m in (16, 512)] + \
             [("qwen3_nvfp4", m) for m in (1, 16, 64)] + [("small_nvfp4", m) for m in (16, 512)] + \
             [("qwen3_nvfp4_prefill", m) for m in (512, 4096, 16384)]


@pytest.mark.parametrize("wl_name,m", FULL_CASES)
def test_forward_full_size(cuda, oracle_mod, wl_name, m):
    from mixture_experts_ffn_gemv_gb300 import binding
    wl = I.WORKLOADS[wl_name]
    tensors, layer = layer_for(wl, cuda)
    x = I.make_x(wl.shape, m, device=cuda)
    try:
        out, ids, w = layer.moe_forward(x, tensors["router_w"], tensors["router_bias"], return_routing=True)
    except binding.MoeError as e:
        if e.status == binding.MOE_ERR_UNSUPPORTED:
            pytest.skip("grouped GEMM arm not available")
        raise
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    L, r_ids, r_w, margin = oracle_route(oracle_mod, wl.shape, tensors, x)
    swapped, bad = check_ids(to_np(ids), r_ids, selection_keys(wl.shape, L, tensors["router_bias"]))
    assert not bad, bad[:5]
    assert len(swapped) <= max_swapped(m), len(swapped)
    # sampled rows plus every near-tie token, the latter under the GPU's ids
    rows = np.union1d(sample_rows(m), np.asarray(swapped, np.int64)).astype(np.int64)
    f_ids, f_w = forced_routing(oracle_mod, wl.shape, L, r_ids, r_w, to_np(ids), swapped)
    ref = oracle_rows(oracle_mod, wl.shape, tensors, x, f_ids, f_w, rows)
    err = rel_l2(to_np(out)[rows], ref)
    assert err < tol(wl.shape), err
    if len(swapped):
        pos = np.searchsorted(rows, swapped)
        assert rel_l2(to_np(out)[swapped], ref[pos]) < tol(wl.shape)


# ------------------------------------------------------------------ edge cases

def test_zero_tokens_launch_nothing(cuda):
    wl = I.WORKLOADS["tiny"]
    tensors, layer = layer_for(wl, cuda)
    x = torch.empty(0, wl.shape.hidden, dtype=torch.bfloat16, device=cuda)
    out = layer.moe_forward(x, tensors["router_w"])
    assert out.shape == (0, wl.shape.hidden)
    assert layer.last_launch_count() == 0


def test_zero_router_ties_pick_lowest_indices(cuda, oracle_mod):
    wl = I.WORKLOADS["tiny"]
    tensors, layer = layer_for(wl, cuda)
    x = I.make_x(wl.shape, 9, seed=5, device=cuda)
    zero = torch.zeros_like(tensors["router_w"])
    out, ids, w = layer.moe_forward(x, zero, return_routing=True)
    torch.cuda.synchronize()
    k = wl.shape.top_k
    assert np.array_equal(to_np(ids), np.tile(np.arange(k), (9, 1)))
    assert np.all(to_np(w) == np.float32(1.0 / k))
    host = {n: tensors[n].cpu() for n in ("w1", "w3", "w2")}
    ref = oracle_mod.moe_forward(wl.shape, host, x.cpu(), to_np(ids).astype(np.int32),
                                 np.full((9, k), 1.0 / k, np.float32))
    assert rel_l2(to_np(out), ref) < TOL[False]


@pytest.mark.parametrize("arm", ["gemv", "gemm"])
def test_all_tokens_on_one_expert(cuda, oracle_mod, arm):
    from mixture_experts_ffn_gemv_gb300 import binding
    shape = MEDIUM_BF16
    tensors, x = _small_case(shape, 260, seed=41, device=cuda)
    bias = torch.zeros(shape.num_experts, device=cuda)
    bias[5] = 100.0  # expert 5 is every token's first choice: 260 rows, 3 m-tiles with a ragged end
    host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in tensors.items()}
    host["router_bias"] = bias.cpu()
    ref = oracle_mod.reference(shape, host, x.cpu())
    assert np.all(ref["ids"][:, 0] == 5)
    layer = binding.MoeLayer(shape, tensors)
    try:
        out, ids, w = layer.moe_forward(x, tensors["router_w"], bias, arm=arm, return_routing=True)
    except binding.MoeError as e:
        if e.status == binding.MOE_ERR_UNSUPPORTED and arm == "gemm":
            pytest.skip("grouped GEMM arm not available")
        raise
    torch.cuda.synchronize()
    swapped, bad = check_ids(to_np(ids), ref["ids"], ref["logits"])
    assert not bad
    assert len(swapped) <= max_swapped(260)
    f_ids, f_w = forced_routing(oracle_mod, shape, ref["logits"], ref["ids"], ref["w"], to_np(ids), swapped)
    want = oracle_mod.moe_forward(shape, host, x.cpu(), f_ids, f_w)
    assert rel_l2(to_np(out), want) < TOL[False]


def test_single_expert_top1_is_dense_mlp(cuda, oracle_mod):
    from mixture_experts_ffn_gemv_gb300 import binding
    shape = I.LayerShape(hidden=256, num_experts=1, top_k=1, inter=256)
    tensors, x = _small_case(shape, 33, seed=51, device=cuda)
    layer = binding.MoeLayer(shape, tensors)
    out, ids, w = layer.moe_forward(x, tensors["router_w"], return_routing=True)
    torch.cuda.synchronize()
    assert np.all(to_np(ids) == 0) and np.all(to_np(w) == 1.0)
    x64 = x.double()
    g = x64 @ tensors["w1"][0].double().T
    u = x64 @ tensors["w3"][0].double().T
    dense = (torch.nn.functional.silu(g) * u) @ tensors["w2"][0].double().T
    assert rel_l2(to_np(out), dense.cpu().numpy()) < TOL[False]


@pytest.mark.parametrize("arm", ["gemv", "gemm"])
def test_bad_expert_id_sets_device_flag(cuda, oracle_mod, arm):
    """Out-of-range ids set the device flag and their pairs are dropped on
    both arms (the grouped-GEMM arm's gather skips the sorted slots they
    leave empty); the other pairs still give the oracle's sum."""
    wl = I.WORKLOADS["tiny"]
    tensors, layer = layer_for(wl, cuda)
    x = I.make_x(wl.shape, 4, device=cuda)
    ids = torch.tensor([[0, 1], [2, 8], [3, 4], [5, -1]], dtype=torch.int32, device=cuda)
    w = torch.full((4, 2), 0.5, device=cuda)
    out = layer.moe_experts(x, ids, w, arm=arm)
    assert layer.device_status() == 1  # DEV_ERR_BAD_ID
    host = {n: tensors[n].cpu() for n in ("w1", "w3", "w2")}
    keep = np.array([[0.5, 0.5], [0.5, 0.0], [0.5, 0.5], [0.5, 0.0]], np.float32)
    ref = oracle_mod.moe_forward(wl.shape, host, x.cpu(), to_np(ids.clamp(0, 7)).astype(np.int32), keep)
    assert rel_l2(to_np(out), ref) < TOL[False]
    layer.moe_experts(x, ids.clamp(0, 7), w, arm=arm)
    assert layer.device_status() == 0  # the next call starts clean


# The grouped-GEMM arm's gather places a chunk's pairs of one expert in the
# order of shared-memory atomics, so its sorted rows may differ from call to
# call; the bf16 (qwen3_prefill) and fp8 (deepseek_v3_fp8 at m = 256) cases
# check that the output does not.
@pytest.mark.parametrize("wl_name,m", [("tiny", 16), ("qwen3_decode", 16), ("qwen3_decode", 1),
                                       ("deepseek_v3_fp8", 1), ("qwen3_nvfp4", 16), ("qwen3_prefill", 4096),
                                       ("deepseek_v3_fp8", 256)])
def test_deterministic_and_graph_capturable(cuda, wl_name, m):
    wl = I.WORKLOADS[wl_name]
    tensors, layer = layer_for(wl, cuda)
    x = I.make_x(wl.shape, m, device=cuda)
    a = layer.moe_forward(x, tensors["router_w"], tensors["router_bias"])
    b = layer.moe_forward(x, tensors["router_w"], tensors["router_bias"])
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    layer.workspace(m)
    out = torch.empty_like(a)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            layer.moe_forward(x, tensors["router_w"], tensors["router_bias"], out=out, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, a)
