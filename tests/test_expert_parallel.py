"""Expert parallelism (experts split over ranks) on CPU: the dispatch plan, and the whole
exchange with gloo ranks against the one-process oracle, bit for bit.

The layer's two compute steps (each rank's experts on the rows it received; the slot-order
reducer) are the library's kernels in the product; here they are CPU stand-ins written from
the oracle (the per-pair FP32 down projection of oracle.moe_forward's debug output, and the
contract's combine in FP32), so what is tested is the dispatch, the exchange and the return of
the partials: the result must equal the oracle's one-process forward exactly, including
skipped pairs, uneven expert loads and a rank with no tokens.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from fp8_block_scaled_router_gb300 import expert_parallel as ep
from fp8_block_scaled_router_gb300 import inputs


def test_plan_orders_pairs_by_owner_then_pair_index():
    ids = np.array([[5, 0], [1, 7], [4, 2], [-1, 6]], np.int32)  # E = 8 over 2 ranks: 0..3 | 4..7
    plan = ep.dispatch_plan(ids, 8, 2)
    assert plan.order.tolist() == [1, 2, 5, 0, 3, 4, 7]
    assert plan.send_counts.tolist() == [3, 4]
    assert plan.local_ids.tolist() == [0, 1, 2, 1, 3, 0, 2]


def test_plan_skips_invalid_ids_and_handles_empty():
    plan = ep.dispatch_plan(np.array([[8, -3]], np.int32), 8, 4)
    assert len(plan.order) == 0 and plan.send_counts.tolist() == [0, 0, 0, 0]
    plan = ep.dispatch_plan(np.zeros((0, 2), np.int32), 8, 2)
    assert len(plan.order) == 0 and plan.send_counts.tolist() == [0, 0]
    with pytest.raises(ValueError):
        ep.dispatch_plan(np.zeros((1, 2), np.int32), 6, 4)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _cpu_callables(x, per, rank):
    """CPU stand-ins for one rank's expert shard: the oracle's per-pair FP32 y, and the combine."""
    import oracle
    lo = rank * per
    w13, s13 = x.w13[lo:lo + per], x.s13[lo:lo + per]
    w2, s2 = x.w2[lo:lo + per], x.s2[lo:lo + per]

    def run_experts(rows, local_ids):
        r = rows.numpy().view(np.uint16)
        n = r.shape[0]
        _, dbg = oracle.moe_forward(r, local_ids.numpy().reshape(n, 1), np.ones((n, 1), np.float32), w13, s13, w2, s2,
                                    debug=True)
        return torch.from_numpy(np.ascontiguousarray(dbg["y"][:, 0, :]))

    def combine(y_pairs, ids, weights):
        M, K = ids.shape
        y = y_pairs.numpy().reshape(M, K, x.shape.hidden)
        w = weights.numpy()
        idn = ids.numpy()
        acc = np.zeros((M, y.shape[2]), np.float32)
        for j in range(K):
            valid = ((idn[:, j] >= 0) & (idn[:, j] < x.shape.num_experts))[:, None]
            term = (w[:, j:j + 1] * y[:, j, :]).astype(np.float32)  # FP32 multiply
            acc = np.where(valid, (acc + term).astype(np.float32), acc)  # then add, slot order
        return torch.from_numpy(inputs.to_bf16_bits(acc).view(np.int16))

    return run_experts, combine


def _ep_rank(rank, world, port, name, tokens_per_rank, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        x = inputs.make(name, M=sum(tokens_per_rank))
        K, E = x.shape.top_k, x.shape.num_experts
        t0 = sum(tokens_per_rank[:rank])
        M = tokens_per_rank[rank]
        hid = x.hidden[t0:t0 + M]
        if M == 0:  # a rank with no tokens still serves its experts
            ids, w = np.zeros((0, K), np.int32), np.zeros((0, K), np.float32)
        elif x.ids is not None:
            ids, w = x.ids[t0:t0 + M], x.weights[t0:t0 + M]
        else:
            ids, w = oracle.route(hid, x.router_w, x.bias, K)
        ids = ids.copy()
        if M > 1:
            ids[1, 0] = -1  # a skipped pair
        per = ep.experts_per_rank(E, world)
        run, comb = _cpu_callables(x, per, rank)
        layer = ep.ExpertParallelLayer(dist.group.WORLD, E, K, x.shape.hidden, run, comb)
        out = layer.forward(torch.from_numpy(hid.view(np.int16)), torch.from_numpy(ids), torch.from_numpy(w))
        q.put((rank, out.numpy().view(np.uint16).copy(), ids))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name,world,tokens", [("tiny", 2, (5, 3)), ("tiny", 4, (3, 0, 4, 2)),
                                               ("many_experts", 2, (6, 6))])
def test_ep_ranks_equal_the_one_process_oracle(name, world, tokens):
    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ep_rank, args=(r, world, port, name, tokens, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted((q.get(timeout=10) for _ in range(world)), key=lambda g: g[0])
    x = inputs.make(name, M=sum(tokens))
    hid = x.hidden[:sum(tokens)]
    ids = np.concatenate([g[2] for g in got])
    _, w = oracle.route(hid, x.router_w, x.bias, x.shape.top_k)
    ref = oracle.moe_forward(hid, ids, w, x.w13, x.s13, x.w2, x.s2)
    out = np.concatenate([g[1] for g in got])
    assert out.shape == ref.shape
    assert np.array_equal(out, ref)
