"""Expert parallelism, host orchestration on CPU (gloo, world size 2).

Each rank holds half of the experts.  Its shard's partial forward and the
shared-expert add are stood in for by the oracle (the routed sum over the
pairs whose expert the rank holds; the shared expert alone), so these tests
check what expert_parallel_forward itself does: one fp32 all-reduce of the
partial outputs and the shared expert added once, after it -- the EP block of
spark_model/layers/moe/forward_prefill.rs.  The same result must come out on
every rank and equal the oracle's whole layer.
"""
import dataclasses
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SHAPE = dict(hidden=256, num_experts=8, top_k=2, inter=128, shared_inter=128)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleShard:
    """A CPU stand-in for one shard's layer handle, built on the oracle."""

    def __init__(self, oracle, shape, tensors, begin, end):
        self.oracle, self.shape, self.t, self.begin, self.end = oracle, shape, tensors, begin, end

    def moe_forward(self, x, router_w, router_bias=None, arm="auto"):
        host = dict(self.t, router_w=router_w, router_bias=router_bias)
        _, ids, w, _ = self.oracle.route(self.shape, host, x)
        mine = (ids >= self.begin) & (ids < self.end)
        routed_only = dataclasses.replace(self.shape, shared_inter=0)
        part = self.oracle.moe_forward(routed_only, host, x, ids, np.where(mine, w, 0).astype(np.float32))
        return torch.from_numpy(part).to(torch.bfloat16)

    def moe_shared_expert_add(self, x, out, arm="auto"):
        m, k = x.shape[0], self.shape.top_k
        s = self.oracle.moe_forward(self.shape, self.t, x, np.zeros((m, k), np.int32), np.zeros((m, k), np.float32))
        out.copy_((out.float() + torch.from_numpy(s)).to(torch.bfloat16))
        return out


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    from mixture_experts_ffn_gemv_gb300 import expert_parallel as ep
    from mixture_experts_ffn_gemv_gb300 import inputs as I
    dist.init_process_group("gloo", rank=rank, world_size=world)
    shape = I.LayerShape(**SHAPE)
    layer = I.make_layer(I.Workload("ep", shape, (12,)), seed=3)
    x = I.make_x(shape, 12, seed=3)
    begin, end = ep.shard_range(shape.num_experts, world, rank)
    shard = OracleShard(oracle, shape, layer, begin, end)
    out = ep.expert_parallel_forward(shard, x, layer["router_w"], None, has_shared=True)
    q.put((rank, begin, end, out.float().numpy()))
    dist.destroy_process_group()


def test_expert_parallel_forward_gloo(oracle_mod):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=120) for _ in range(world)), key=lambda r: r[0])
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert [(r[1], r[2]) for r in got] == [(0, 4), (4, 8)]
    assert np.array_equal(got[0][3], got[1][3])  # every rank ends with the same output
    from mixture_experts_ffn_gemv_gb300 import inputs as I
    shape = I.LayerShape(**SHAPE)
    layer = I.make_layer(I.Workload("ep", shape, (12,)), seed=3)
    x = I.make_x(shape, 12, seed=3)
    ref = oracle_mod.reference(shape, layer, x)["out"]
    rel = np.linalg.norm(got[0][3] - ref) / np.linalg.norm(ref)
    assert rel < 1e-2, rel


def test_shard_range_and_tensors():
    from mixture_experts_ffn_gemv_gb300 import expert_parallel as ep
    assert [ep.shard_range(10, 4, r) for r in range(4)] == [(0, 3), (3, 6), (6, 8), (8, 10)]
    assert [ep.shard_range(8, 2, r) for r in range(2)] == [(0, 4), (4, 8)]
    with pytest.raises(ValueError):
        ep.shard_range(2, 3, 0)
    t = {"w1": torch.arange(24.0).reshape(6, 2, 2), "ws1": torch.ones(2, 2), "router_w": torch.zeros(6, 2)}
    s = ep.shard_tensors(t, 2, 5)
    assert torch.equal(s["w1"], t["w1"][2:5]) and s["w1"].is_contiguous()
    assert s["ws1"] is t["ws1"] and s["router_w"] is t["router_w"]
