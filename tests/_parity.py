"""Comparison helpers shared by the GPU parity tests (no arithmetic of the
layer lives here: expected values come from the oracle)."""
from __future__ import annotations

import numpy as np
import torch

INDEX_MARGIN = 1e-4          # ids may differ only where oracle logits are this close
TOL = {False: 1e-2, True: 2e-2}  # rel L2 bound: bf16 weights / fp8 block-scaled weights


def tol(shape) -> float:
    """rel L2 bound of a layer shape: 1e-2 for bf16 weights, 2e-2 for the
    block-scaled formats (fp8, NVFP4)."""
    return TOL[bool(shape.fp8 or getattr(shape, "nvfp4", False))]


def rel_l2(got, ref) -> float:
    g = np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    return float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))


def to_np(t):
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu()
        if t.dtype == torch.bfloat16:
            t = t.float()
        return t.numpy()
    return np.asarray(t)


def check_ids(gpu_ids, ref_ids, ref_logits, margin=INDEX_MARGIN):
    """Expert indices must equal the oracle's, except that position j may hold
    another expert whose oracle logit is within `margin` of the oracle's pick
    at j (a near tie: an order swap, or a swap across the k-th/(k+1)-th
    boundary when that gap is below the margin).

    Returns (rows whose id *sets* differ, list of violations)."""
    g = np.asarray(gpu_ids)
    r = np.asarray(ref_ids)
    L = np.asarray(ref_logits)
    diff_rows = np.nonzero((g != r).any(axis=1))[0]
    bad = []
    swapped = []
    for t in diff_rows:
        lg = L[t, g[t]]
        lr = L[t, r[t]]
        if np.any(np.abs(lg.astype(np.float64) - lr.astype(np.float64)) >= margin) or len(set(g[t])) != len(g[t]):
            bad.append((int(t), g[t].tolist(), r[t].tolist()))
        if set(g[t].tolist()) != set(r[t].tolist()):
            swapped.append(int(t))
    return swapped, bad


def selection_keys(shape, logits, bias):
    """What the top-k ranks, as the oracle forms it: the logits (softmax
    scoring, bias already inside) or fp32 sigmoid(L) + bias (sigmoid scoring),
    for check_ids' margin rule."""
    L = np.asarray(logits, np.float32)
    if getattr(shape, "scoring", "softmax") != "sigmoid":
        return L
    s = (np.float32(1.0) / (np.float32(1.0) + np.exp(-L))).astype(np.float32)
    if bias is not None:
        s = s + np.asarray(bias.cpu() if isinstance(bias, torch.Tensor) else bias, np.float32)
    return s


def compact_experts(shape, layer, expert_ids):
    """CPU copies of only the listed experts (stacked in the listed order)."""
    idx = torch.as_tensor(sorted(set(int(e) for e in expert_ids)), dtype=torch.long)
    dev = layer["w1"].device
    sub = {}
    for n in ("w1", "w3", "w2", "s1", "s3", "s2", "sb1", "sb3", "sb2"):
        if n in layer and layer[n] is not None:
            sub[n] = layer[n].index_select(0, idx.to(dev)).cpu()
    for n in ("ws1", "ws3", "ws2", "ss1", "ss3", "ss2", "ssb1", "ssb3", "ssb2", "shared_gate"):
        if n in layer and layer[n] is not None:
            sub[n] = layer[n].cpu()
    remap = {int(e): i for i, e in enumerate(idx.tolist())}
    return sub, remap, len(idx)


def oracle_rows(oracle, shape, layer, x, ids, w, rows):
    """Oracle output for the token rows `rows` given the routing (ids, w),
    carrying only the experts those rows select over to the host."""
    rows = np.asarray(rows, np.int64)
    ids_r = np.asarray(ids)[rows]
    w_r = np.asarray(w, np.float32)[rows]
    sub, remap, U = compact_experts(shape, layer, ids_r.reshape(-1))
    ids_c = np.vectorize(remap.__getitem__)(ids_r).astype(np.int32)
    import dataclasses
    sub_shape = dataclasses.replace(shape, num_experts=U)
    x_r = x.index_select(0, torch.as_tensor(rows, device=x.device)).cpu()
    return oracle.moe_forward(sub_shape, sub, x_r, ids_c, w_r)


def max_swapped(m: int) -> int:
    """How many tokens may hold a near-tie id set other than the oracle's."""
    return max(2, m // 200)


def forced_routing(oracle, shape, logits, ref_ids, ref_w, gpu_ids, swapped):
    """The routing each token is compared under: the oracle's own ids and
    weights, except for the near-tie tokens in `swapped`, which take the GPU's
    ids with the oracle's weights for those ids (the forced-ids mode)."""
    ids = np.array(ref_ids, np.int32, copy=True)
    w = np.array(ref_w, np.float32, copy=True)
    if len(swapped):
        sw = np.asarray(swapped, np.int64)
        g = np.asarray(gpu_ids, np.int32)[sw]
        ids[sw] = g
        w[sw] = oracle.route_weights(shape, np.asarray(logits, np.float32)[sw], g)
    return ids, w
