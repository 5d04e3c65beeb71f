#!/usr/bin/env python3
"""Benchmark of the MoE FFN layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload qwen3_prefill] [--tokens 4096] [--no-sweep]
                    [--sweep-out FILE]

One step = one forward of the whole layer (router, top-k, permute, experts,
combine) over one batch of m synthetic tokens.  The default workload is the
Qwen3-30B-A3B-shaped layer at prefill, m = 4096 tokens, bf16.  Steps rotate
over R layer replicas (different seeds) whose weights together exceed L2
several times, so no step finds its experts in L2.

Output: the LAST line of stdout is the one headline JSON object (rank 0).
The per-size sweep over every workload and the layer-tail comparison go to
stderr as one compact JSON object per line (and to --sweep-out when given),
so the headline stays short and last.

Under torchrun (N > 1) every rank runs its own replica set on its own GPU
with its own tokens (token-parallel, no data-path collective) and the
whole-job throughput is the tokens of all ranks over the slowest rank's time.

--impl reference times the CPU oracle (the plain per-token loops) on the
host cores on the same workload: every step is one oracle forward of a
bounded sample of the batch (its first tokens; tokens are independent, so
those rows are exactly the full batch's); under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mixture_experts_ffn_gemv_gb300 import inputs as I  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "MoE layer tokens/s; % of HBM roofline (decode) / tensor peak (prefill)"

# ----------------------------------------------------------------- helpers


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws):
    if ws <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, v: float, device) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [int(r[1]) for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": int(rows[0][2]), "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit()) if rows else None,
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------- algorithmic bytes / flops


NVFP4_B = 0.5 + 1.0 / 16  # bytes per NVFP4 element: a 4-bit code + an e4m3 scale per 16


def _dtype(shape) -> str:
    """The arithmetic type of the expert path."""
    if getattr(shape, "nvfp4", False):
        return "nvfp4_e2m1"
    return "fp8_e4m3" if shape.fp8 else "bf16"


def expert_bytes(shape):
    """Bytes of one expert's three matrices (+ fp8 block scales, or NVFP4
    block scales and per-matrix scales)."""
    H, I_ = shape.hidden, shape.inter
    if getattr(shape, "nvfp4", False):
        return int(3 * H * I_ * NVFP4_B) + 3 * 4
    wb = 1 if shape.fp8 else 2
    b = 3 * H * I_ * wb
    if shape.fp8:
        b += 3 * (H // 128) * (I_ // 128) * 4
    return b


def kernel_alg_bytes(kernel, shape, m, U, gemm_arm=None):
    """Algorithmic bytes one launch of `kernel` must move: each weight and
    activation it needs read once, each output written once.  U = active
    expert groups (distinct routed experts + the shared expert).  gemm_arm:
    whether the expert kernels were the grouped GEMMs (their y rows are bf16;
    the GEMV arm's are fp32)."""
    H, I_, E, k = shape.hidden, shape.inter, shape.num_experts, shape.top_k
    P = m * k
    rows = P + (m if shape.shared_inter else 0)
    if getattr(shape, "nvfp4", False):
        # W4A4: weights and activations both count as NVFP4 (a half-byte code
        # + an e4m3 scale per 16 + an fp32 scale per row); the kernels' own
        # wider intermediates (f16 A rows, fp32 h) are implementation choices
        # and are not counted as algorithmic bytes.
        xa = H * NVFP4_B + 4    # one quantised x row
        ha = I_ * NVFP4_B + 4   # one quantised h row
        if kernel == "gemv_gateup":
            return int(U * 2 * I_ * H * NVFP4_B + m * xa + rows * ha)
        if kernel == "gemv_down":
            return int(U * H * I_ * NVFP4_B + rows * ha + rows * H * 2)
        if kernel == "gemm_gateup":
            return int(U * 2 * I_ * H * NVFP4_B + rows * xa + rows * ha)
        if kernel == "gemm_down":
            return int(U * H * I_ * NVFP4_B + rows * ha + rows * H * 2)
        if kernel == "act_quant_nvfp4":
            return int(m * H * 2 + m * (H * NVFP4_B + 4))
        if kernel == "h_quant_nvfp4":
            return int(rows * I_ * 4 + rows * (I_ * NVFP4_B + 4))
    wb = 1 if shape.fp8 else 2
    ab = 1 if shape.fp8 else 2
    sc = 4 * (H // 128) * (I_ // 128) if shape.fp8 else 0
    if kernel in ("gemv_gateup", "gemm_gateup"):
        x_in = (m if kernel == "gemv_gateup" else rows) * H * ab
        return U * (2 * I_ * H * wb + 2 * sc) + x_in + rows * I_ * ab
    if kernel == "gemv_down":
        return U * (H * I_ * wb + sc) + rows * I_ * ab + rows * H * 4
    if kernel == "gemm_down":
        return U * (H * I_ * wb + sc) + rows * I_ * ab + rows * H * 2
    if kernel == "router":
        return E * H * 4 + m * H * 2 + m * E * 4
    if kernel == "combine":
        return rows * H * (2 if gemm_arm else 4) + m * H * 2 + P * 8
    if kernel == "gather_rows":
        return m * H * ab + rows * H * ab
    if kernel == "router_split":
        return E * H * 4 + 3 * E * H * 2
    if kernel == "topk_softmax":
        return m * E * 4 + P * 8
    if kernel == "act_quant_fp8":
        return m * H * 2 + m * H + m * (H // 128) * 4
    if kernel in ("permute_count", "permute_scatter"):
        return P * 4 * (1 if kernel == "permute_count" else 3)
    return None


def layer_alg(shape, m, U):
    """(bytes, flops) of one layer forward: weights of the U active groups,
    router, x in, out; flops of the routed pairs and the shared expert."""
    H, I_, E, k = shape.hidden, shape.inter, shape.num_experts, shape.top_k
    byt = U * expert_bytes(shape) + E * H * 4 + 2 * m * H * 2
    flops = 2 * m * k * 3 * H * I_ + (2 * m * 3 * H * shape.shared_inter if shape.shared_inter else 0)
    return byt, flops


def tensor_ratio(shape):
    """Dense tensor-core rate of the layer's MMA type over bf16's, the nominal
    ratio (fp8 4.5 / 2.25, NVFP4 13.5 / 2.25 PFLOP/s), applied to the measured
    bf16 peak.  (The block-scaled NVFP4 MMA measured 4x the bf16 MMA rate on
    GB300, so against the nominal ratio an NVFP4 GEMM reads at most 0.67.)"""
    if getattr(shape, "nvfp4", False):
        return 6.0
    return 2.0 if shape.fp8 else 1.0


def kernel_flops(kernel, shape, m):
    H, I_, k = shape.hidden, shape.inter, shape.top_k
    rows = m * k + (m if shape.shared_inter else 0)
    if kernel in ("gemm_gateup", "gemv_gateup"):
        return 2 * rows * 2 * H * I_
    if kernel in ("gemm_down", "gemv_down"):
        return 2 * rows * H * I_
    return None


def active_groups(ids_list, shape):
    s = shape.shared_inter > 0
    return [len(np.unique(ids.cpu().numpy())) + (1 if s else 0) for ids in ids_list]


def source_digest(kernel):
    """Digest of the CUDA source a kernel is built from (to tell stale counters)."""
    fname = {"gemv_gateup": "gemv.cu", "gemv_down": "gemv.cu", "gemm_gateup": "gemm.cu",
             "gemm_down": "gemm.cu", "router": "route.cu", "topk_softmax": "route.cu",
             "combine": "combine.cu", "permute_count": "permute.cu", "permute_scatter": "permute.cu",
             "gather_rows": "permute.cu", "act_quant_fp8": "permute.cu"}.get(kernel)
    if fname is None:
        return None
    h = hashlib.sha256()
    for f in (fname, "common.cuh"):
        with open(os.path.join(ROOT, "mixture_experts_ffn_gemv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload, m):
    """dram read+write bytes per launch from the committed ncu summary, when it
    was taken on the current source of that kernel; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(f"{kernel}@{workload}_m{m}")
    if not rec or rec.get("source_digest") != source_digest(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


# ----------------------------------------------------------------- our arm


def build_replicas(wl, m, device, seed_base, max_bytes=48e9, replicas=0):
    from mixture_experts_ffn_gemv_gb300 import binding
    shape = wl.shape
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    full = shape.num_experts * expert_bytes(shape)
    # expected touched bytes per step: distinct experts among m*k draws
    exp_u = shape.num_experts * (1 - (1 - shape.top_k / shape.num_experts) ** m)
    touched = max(exp_u * expert_bytes(shape), 1)
    R = max(2, math.ceil(4 * l2 / touched))
    R = int(max(1, min(R, 16, max_bytes // max(full, 1))))
    if replicas > 0:
        R = replicas
    reps = []
    ws = None
    for r in range(R):
        tensors = I.make_layer(wl, seed=seed_base + r, device=device)
        layer = binding.MoeLayer(shape, tensors)
        layer.prepare_router(tensors["router_w"])  # load-time split of the router weight
        if ws is None:
            ws = layer.workspace(m)
        layer._ws = ws
        x = I.make_x(shape, m, seed=seed_base + r, device=device)
        out = torch.empty(m, shape.hidden, dtype=torch.bfloat16, device=device)
        reps.append({"tensors": tensors, "layer": layer, "x": x, "out": out})
    return reps, R, R * full


def run_steps(reps, n, arm="auto", routing=None):
    launches = 0
    for i in range(n):
        r = reps[i % len(reps)]
        t = r["tensors"]
        if routing is not None:
            out, ids, w = r["layer"].moe_forward(r["x"], t["router_w"], t["router_bias"], arm=arm, out=r["out"],
                                                 return_routing=True)
            routing.append(ids)
        else:
            r["layer"].moe_forward(r["x"], t["router_w"], t["router_bias"], arm=arm, out=r["out"])
        launches += r["layer"].last_launch_count()
    return launches


def time_steps(reps, n, device, dist):
    stream = torch.cuda.current_stream(device)
    barrier(dist, device)
    torch.cuda.synchronize(device)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    launches = run_steps(reps, n)
    b.record(stream)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    return a.elapsed_time(b), launches


def kernel_profile(reps, n, wl, m):
    """Per-kernel device time over n steps (a second pass with event timing on)."""
    for r in reps:
        r["layer"].kernel_timing(True)
    routing = []
    run_steps(reps, n, routing=routing)
    totals = {}
    for r in reps:
        for name, (ms, cnt) in r["layer"].kernel_times().items():
            t = totals.setdefault(name, [0.0, 0])
            t[0] += ms
            t[1] += cnt
        r["layer"].kernel_timing(False)
    U = active_groups(routing, wl.shape)
    return totals, U


def e2e_steps(reps, n, device, dist, m, shape):
    """The same forward through the C-ABI with every step's input copied in
    from pinned host memory and its output copied back, all inside the timed
    region.  The copies run on a second stream and are pipelined with the
    forwards (two device slots): step i+1's input uploads while step i
    computes, and step i's output downloads while step i+1 computes, as a
    serving loop would overlap them."""
    compute = torch.cuda.current_stream(device)
    copy = torch.cuda.Stream(device)
    R = len(reps)
    xh = [r["x"].cpu().pin_memory() for r in reps]
    oh = [torch.empty(m, shape.hidden, dtype=torch.bfloat16).pin_memory() for _ in range(R)]
    xd = [torch.empty_like(reps[0]["x"]) for _ in range(2)]
    od = [torch.empty(m, shape.hidden, dtype=torch.bfloat16, device=device) for _ in range(2)]
    ev = lambda: torch.cuda.Event()  # noqa: E731
    h2d = [ev() for _ in range(n)]
    fwd = [ev() for _ in range(n)]
    d2h = [ev() for _ in range(n)]
    barrier(dist, device)
    torch.cuda.synchronize(device)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(compute)
    copy.wait_stream(compute)
    with torch.cuda.stream(copy):
        xd[0].copy_(xh[0], non_blocking=True)
        h2d[0].record(copy)
    for i in range(n):
        s = i % 2
        r = reps[i % R]
        t = r["tensors"]
        compute.wait_event(h2d[i])
        if i >= 2:
            compute.wait_event(d2h[i - 2])  # this slot's previous output has been read back
        r["layer"].moe_forward(xd[s], t["router_w"], t["router_bias"], out=od[s], stream=compute)
        fwd[i].record(compute)
        with torch.cuda.stream(copy):
            if i + 1 < n:
                if i >= 1:
                    copy.wait_event(fwd[i - 1])  # the other slot's input is no longer read
                xd[1 - s].copy_(xh[(i + 1) % R], non_blocking=True)
                h2d[i + 1].record(copy)
            copy.wait_event(fwd[i])
            oh[i % R].copy_(od[s], non_blocking=True)
            d2h[i].record(copy)
    compute.wait_stream(copy)
    b.record(compute)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    bytes_in = m * shape.hidden * 2
    return a.elapsed_time(b), bytes_in, m * shape.hidden * 2


def oracle_sample_tokens(shape, m, target_flop=12e9):
    """Tokens of the bounded oracle sample: about target_flop of expert work
    (roughly a second on the GPU machine's host cores), at least one, at most m."""
    per_tok = 2 * 3 * shape.hidden * shape.inter * shape.top_k
    if shape.shared_inter:
        per_tok += 2 * 3 * shape.hidden * shape.shared_inter
    return int(max(1, min(m, round(target_flop / per_tok))))


def cpu_baseline(wl, m, reps_host, budget_s=12.0):
    """The oracle, as it stands, on the host cores: whole-layer forwards of a
    bounded sample of the m-token batch (its first tokens, routed and summed
    exactly as in the full batch, since tokens are independent), repeated
    until ~budget_s of wall time."""
    import oracle
    cores = oracle.set_threads(os.cpu_count() or 1)
    tensors, x = reps_host
    ns = oracle_sample_tokens(wl.shape, m)
    xs = x[:ns].contiguous()
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.reference(wl.shape, tensors, xs)
        n += 1
        if time.perf_counter() - t0 >= budget_s or n >= 1000:
            break
    dt = time.perf_counter() - t0
    return {"value": n * ns / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} oracle forwards of the first {ns} of the {m} tokens, {dt:.1f} s"}


def host_copy(tensors):
    return {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in tensors.items()}


def sweep(device, steps, warmup, emit):
    """tokens/s and layer roofline fraction of every workload size (N=1);
    emit(row) receives each row as soon as it is measured."""
    pk, _ = peaks()
    bw = pk["hbm_gbs"] * 1e9
    tc = pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]) * 1e12
    res = []
    for name in ("qwen3_decode", "qwen3_prefill", "deepseek_v3_fp8", "qwen3_zipf", "deepseek_v3_sigmoid",
                 "gated_shared", "qwen3_nvfp4", "qwen3_nvfp4_prefill"):
        wl = I.WORKLOADS[name]
        for m in wl.ms:
            try:
                reps, R, _ = build_replicas(wl, m, device, seed_base=0, max_bytes=32e9)
                run_steps(reps, warmup)
                n = max(4, min(steps, 50))
                ms, _ = time_steps(reps, n, device, None)
                routing = []
                run_steps(reps, min(n, len(reps)), routing=routing)
                U = float(np.mean(active_groups(routing, wl.shape)))
                byt, flops = layer_alg(wl.shape, m, U)
                per = ms / n / 1e3
                tc_peak = tc * tensor_ratio(wl.shape)
                t_roof = max(byt / bw, flops / tc_peak)
                arm = reps[0]["layer"].select_arm(m)
                totals, _ = kernel_profile(reps, n, wl, m)
                kern = {}
                for kname, (kms, kcnt) in sorted(totals.items(), key=lambda kv: -kv[1][0]):
                    avg = kms / kcnt / 1e3
                    ent = {"avg_us": avg * 1e6}
                    kb = kernel_alg_bytes(kname, wl.shape, m, U, gemm_arm=arm == 2)
                    kf = kernel_flops(kname, wl.shape, m)
                    if kb:
                        ent["hbm_frac"] = kb / avg / bw
                    if kf and kname.startswith("gemm"):
                        ent["tensor_frac"] = kf / avg / tc_peak
                    kern[kname] = ent
                res.append({"workload": name, "m": m, "arm": {1: "gemv", 2: "gemm"}.get(arm, arm),
                            "tokens_per_s": m / per, "ms_per_step": per * 1e3, "alg_bytes": byt,
                            "alg_flops": flops, "active_groups": U, "bound": "hbm" if byt / bw >= flops / tc_peak else "tensor",
                            "layer_roofline_frac": t_roof / per, "kernels": kern})
            except Exception as e:  # keep the headline line even if one size fails
                res.append({"workload": name, "m": m, "error": str(e)[:200]})
            finally:
                reps = None
                torch.cuda.synchronize(device)
                torch.cuda.empty_cache()
            emit(_compact_row(res[-1]))
    return res


def _compact_row(row):
    """A sweep row with its figures rounded (one short line per size)."""
    out = {}
    for k, v in row.items():
        if isinstance(v, float):
            out[k] = _r(v)
        elif isinstance(v, dict):
            out[k] = {kk: ({a: _r(b) for a, b in vv.items()} if isinstance(vv, dict) else _r(vv))
                      for kk, vv in v.items()}
        else:
            out[k] = v
    return out


def tail_timing(reps, n, device, eps=1e-6):
    """The layer tail (residual add + the next layer's RMSNorm) folded into the
    combine (moe_forward_residual_rmsnorm) against moe_forward followed by the
    same add and norm as separate torch ops; us per step, same replicas."""
    H = reps[0]["layer"].shape.hidden
    m = reps[0]["x"].shape[0]
    g = torch.Generator(device=device).manual_seed(5)
    norm_w = (torch.randn(H, generator=g, device=device) * 0.2 + 1.0).contiguous()
    residual = torch.randn(m, H, generator=g, device=device).to(torch.bfloat16)
    normed = torch.empty(m, H, dtype=torch.bfloat16, device=device)

    def fused(i):
        r = reps[i % len(reps)]
        t = r["tensors"]
        r["layer"].moe_forward_residual_rmsnorm(r["x"], t["router_w"], residual, norm_w, eps, t["router_bias"],
                                                norm_out=normed)

    def unfused(i):
        r = reps[i % len(reps)]
        t = r["tensors"]
        out = r["layer"].moe_forward(r["x"], t["router_w"], t["router_bias"], out=r["out"])
        residual.copy_((residual.float() + out.float()).to(torch.bfloat16))
        rf = residual.float()
        normed.copy_((rf * torch.rsqrt(rf.pow(2).mean(1, keepdim=True) + eps) * norm_w).to(torch.bfloat16))

    res = {}
    for name, fn in (("fused_us", fused), ("unfused_us", unfused)):
        for i in range(3):
            fn(i)
        torch.cuda.synchronize(device)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(n):
            fn(i)
        b.record()
        torch.cuda.synchronize(device)
        res[name] = a.elapsed_time(b) * 1e3 / n
    return res


def _r(v, sig=4):
    """Round a float to `sig` significant digits (keeps the headline short)."""
    if v is None or not isinstance(v, float) or v == 0.0 or not math.isfinite(v):
        return v
    return round(v, sig - 1 - int(math.floor(math.log10(abs(v)))))


class SideOutput:
    """Where the long results go: stderr, one compact JSON object per line,
    and optionally a JSON-lines file."""

    def __init__(self, path):
        self.f = open(path, "w") if path else None

    def emit(self, kind, obj):
        row = dict(kind=kind, **obj)
        s = json.dumps(row, separators=(",", ":"))
        print(s, file=sys.stderr, flush=True)
        if self.f:
            self.f.write(s + "\n")
            self.f.flush()

    def close(self):
        if self.f:
            self.f.close()


def run_ours(args):
    ws, rank, local = dist_env()
    dist = init_dist(ws)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    wl = I.WORKLOADS[args.workload]
    if args.experts > 0:
        import dataclasses
        wl = dataclasses.replace(wl, shape=dataclasses.replace(wl.shape, num_experts=args.experts))
    m = args.m
    shape = wl.shape
    reps, R, rep_bytes = build_replicas(wl, m, device, seed_base=1000 * rank, replicas=args.replicas)
    run_steps(reps, args.warmup)
    torch.cuda.synchronize(device)
    with ClockSampler(device.index) as clk:
        ms, launches = time_steps(reps, args.steps, device, dist)
    ms_max = max_over_ranks(dist, ms, device)
    value = ws * m * args.steps / (ms_max / 1e3)

    # per-kernel device times (second pass, event-bracketed launches)
    totals, U = kernel_profile(reps, args.steps, wl, m)
    Umean = float(np.mean(U))
    pk, pk_kind = peaks()
    # the dominant kernel among those with a stated algorithmic byte count
    dom = max(((k, v) for k, v in totals.items() if kernel_alg_bytes(k, shape, m, 1.0) is not None),
              key=lambda kv: kv[1][0])
    dname, (dms, dcnt) = dom
    avg_s = dms / dcnt / 1e3
    flops = kernel_flops(dname, shape, m)
    alg = kernel_alg_bytes(dname, shape, m, Umean, gemm_arm=any(k.startswith("gemm") for k in totals))
    bw = pk["hbm_gbs"]
    # a kernel timed inside a step that lasts over a second is held to the
    # sustained tensor peak, a shorter one to the burst peak
    tc_key = "bf16_tflops_sustained" if ms_max > 1000 else "bf16_tflops"
    tc = pk.get(tc_key, FALLBACK_PEAKS["bf16_tflops"]) * tensor_ratio(shape)
    if flops and alg and flops / (tc * 1e12) > alg / (bw * 1e9):
        roof = {"bound": "tensor", "achieved": flops / avg_s / 1e12, "peak": tc, "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": alg / avg_s / 1e9, "peak": bw, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = recorded_traffic(dname, args.workload, m)
    roof.update({"kernel": dname, "launch_us": avg_s * 1e6, "alg_bytes": alg,
                 "peak_src": "measured" if pk_kind == "measured" else "fallback"})
    lay_b, lay_f = layer_alg(shape, m, Umean)
    t_step = ms_max / args.steps / 1e3
    layer_roof = max(lay_b / (bw * 1e9), lay_f / (tc * 1e12)) / t_step

    e2e_ms, bi, bo = e2e_steps(reps, args.steps, device, dist, m, shape)
    e2e_max = max_over_ranks(dist, e2e_ms, device)
    ktot = sum(t[0] for t in totals.values())
    top = sorted(totals.items(), key=lambda kv: -kv[1][0])

    line = {
        "metric": METRIC, "value": _r(value), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": _r(ms_max / args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": _dtype(shape), "data": "synthetic",
        "config": {"workload": args.workload + (f"(E={args.experts})" if args.experts else ""), "m": m,
                   "hidden": shape.hidden, "experts": shape.num_experts, "top_k": shape.top_k,
                   "inter": shape.inter, "shared_inter": shape.shared_inter, "global_batch": ws * m,
                   "parallelism": f"token-parallel x{ws}",
                   "l2": f"inputs > L2: {R} rotating replicas, {rep_bytes / 1e9:.1f} GB"},
        "gpu_launches": launches,
        "roofline": {k: _r(v) if isinstance(v, float) else v for k, v in roof.items()},
        "layer_roofline": {"frac": _r(layer_roof), "alg_bytes": _r(float(lay_b)), "alg_flops": _r(float(lay_f))},
        "kernel_share": {k: _r(v[0] / ktot, 3) for k, v in top[:5]},
        "e2e": {"value": _r(ws * m * args.steps / (e2e_max / 1e3)), "unit": "tokens/s",
                "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo},
        "clocks": {k: v for k, v in clk.summary().items() if k in ("sm_mhz", "sm_max_mhz", "reasons")},
    }
    side = SideOutput(args.sweep_out if rank == 0 else None)
    if rank == 0:
        side.emit("kernels", {"workload": args.workload, "m": m, "us_per_launch": {
            k: _r(v[0] / v[1] * 1e3) for k, v in top}, "launches_per_step": {k: v[1] / args.steps for k, v in top}})
    if rank == 0 and ws == 1:
        cb = cpu_baseline(wl, m, (host_copy(reps[0]["tensors"]), reps[0]["x"].cpu()))
        line["cpu_baseline"] = {k: _r(v) if isinstance(v, float) else v for k, v in cb.items()}
        if not args.no_sweep:
            side.emit("layer_tail", dict(tail_timing(reps, args.steps, device), workload=args.workload, m=m))
            reps = None
            torch.cuda.empty_cache()
            sweep(device, args.steps, args.warmup, lambda row: side.emit("sweep", row))
    side.close()
    if rank == 0:
        sys.stderr.flush()
        print(json.dumps(line, separators=(",", ":")), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ----------------------------------------------------------------- reference arm (the oracle)


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import oracle
    wl = I.WORKLOADS[args.workload]
    if args.experts > 0:
        import dataclasses
        wl = dataclasses.replace(wl, shape=dataclasses.replace(wl.shape, num_experts=args.experts))
    m = args.m
    tensors = I.make_layer(wl, seed=0, device="cpu")
    x = I.make_x(wl.shape, m, seed=0, device="cpu")
    # every step: one oracle forward of the batch's first ns tokens (tokens are
    # independent, so these rows equal the full batch's first ns rows)
    ns = oracle_sample_tokens(wl.shape, m)
    xs = x[:ns].contiguous()
    cores = oracle.set_threads(os.cpu_count() or 1)
    for _ in range(max(0, min(args.warmup, 1))):
        oracle.reference(wl.shape, tensors, xs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.reference(wl.shape, tensors, xs)
    dt = time.perf_counter() - t0
    value = ns * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": _r(value), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": _r(dt / args.steps * 1e3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": _dtype(wl.shape), "data": "synthetic",
        "config": {"workload": args.workload + (f"(E={args.experts})" if args.experts else ""), "m": m,
                   "hidden": wl.shape.hidden, "experts": wl.shape.num_experts, "top_k": wl.shape.top_k,
                   "inter": wl.shape.inter, "shared_inter": wl.shape.shared_inter, "global_batch": m},
        "cpu_baseline": {"value": _r(value), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: oracle forward of the first {ns} of the {m} tokens"},
        "e2e": {"value": _r(value), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line, separators=(",", ":")), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3_prefill", choices=sorted(I.WORKLOADS))
    ap.add_argument("--tokens", dest="m", type=int, default=4096, help="tokens per step (m)")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--sweep-out", default=None, help="also write the stderr result rows to this JSON-lines file")
    ap.add_argument("--experts", type=int, default=0,
                    help="override the workload's expert count (small cases for profiling captures)")
    ap.add_argument("--replicas", type=int, default=0, help="override the number of rotating layer replicas")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
