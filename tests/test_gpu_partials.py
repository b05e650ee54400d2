"""The layer split at its expert partials (moe_fp8_forward_partials + moe_fp8_combine_pairs) and
the expert-parallel layer built on them, on the GPU.

* partials then the route reducer equal moe_fp8_forward bit for bit, few-row and sorted-tile
  paths, skipped pairs included (their partial rows are zero);
* the expert-parallel layer with one rank (NCCL, world size 1) and the library's callables
  equals moe_fp8_forward bit for bit (the exchange with several ranks is tested on CPU with
  gloo ranks in tests/test_expert_parallel.py).
"""
import os
import socket

import numpy as np
import pytest
import torch

from fp8_block_scaled_router_gb300 import inputs

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import oracle
    from fp8_block_scaled_router_gb300 import _lib as L
    from gpu_harness import GpuMoE, to_dev


@pytest.fixture(scope="module", autouse=True)
def _build():
    from fp8_block_scaled_router_gb300 import build
    build.build()
    oracle.build()


CASES = [("decode", 1), ("verify", 12), ("wide", 16), ("decode", 300), ("prefill", 4096)]


@pytest.mark.parametrize("name,M", CASES, ids=[f"{n}-M{m}" for n, m in CASES])
def test_partials_then_reducer_equal_forward(name, M):
    x = inputs.make(name, tokens=M) if name == "decode" else inputs.make(name)
    g = GpuMoE(x, M)
    hid = to_dev(x.hidden[:M])
    ids, w = g.route(hid, M)
    ids[0, 0] = -1  # a skipped pair
    torch.cuda.synchronize()
    out = g.forward(hid, ids, w, M)
    y = torch.full((M * g.K, g.H), 7.0, dtype=torch.float32, device="cuda")
    L.moe_fp8_forward_partials(hid, ids, M, g.w13, g.s13, g.w2, g.s2, y, g.ws, g.shape)
    out2 = torch.empty_like(out)
    L.moe_fp8_combine_pairs(y, ids, w, M, out2, g.shape)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
    assert torch.all(y[0] == 0)  # the skipped pair's row
    assert g.status() & L.STATUS_BAD_EXPERT_ID


def test_expert_parallel_one_rank_equals_forward():
    import torch.distributed as dist
    from fp8_block_scaled_router_gb300 import expert_parallel as ep
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    try:
        x = inputs.make("verify_skewed")
        M = 12
        g = GpuMoE(x, M)
        hid = to_dev(x.hidden[:M])
        ids, w = g.route(hid, M)
        run, comb = ep.library_callables(g.w13, g.s13, g.w2, g.s2, g.H, g.I, g.E, g.K, max_rows=M * g.K, max_tokens=M)
        layer = ep.ExpertParallelLayer(dist.group.WORLD, g.E, g.K, g.H, run, comb, device=torch.device("cuda"))
        out = layer.forward(hid, ids, w)
        ref = g.forward(hid, ids, w, M)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    finally:
        dist.destroy_process_group()
