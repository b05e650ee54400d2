"""Expert parallelism across ranks (one GPU per rank) for the routed FP8 MoE layer.

Sources: "Inferact/amd-kernels" README (kernels for several GPUs carry a ranks<n> shape token;
expert partials are summed in a fixed order, by a reduce kernel or inside the next kernel,
never with atomic adds) and the "NetraRuntime/netra-kernel" README (the route reducer is a
separate operation with its own reduction order).

Each rank holds its own tokens and a contiguous block of E / world experts (rank r owns
experts r*E/world .. (r+1)*E/world - 1). One step:

1. the caller routes its tokens (the router is replicated: ``moe_route`` on each rank);
2. dispatch: every routed pair (t, j) with a valid expert goes to the expert's owner. The
   plan orders the pairs by owner rank, then by t*K + j (stable), and the hidden rows travel
   in that order with their owner-local expert ids (``all_to_all_single``);
3. each rank runs its experts on the rows it received, one pair per row (K = 1), and keeps
   each pair's down projection in FP32 (``moe_fp8_forward_partials``);
4. the FP32 partials travel back in the same order (``all_to_all_single``) and land at their
   pair's row t*K + j;
5. the route reducer sums them in slot order (``moe_fp8_combine_pairs``): out[t] =
   bf16(sum over j ascending of w[t][j] * y[t*K + j]).

The partials stay FP32 until the reducer, and each pair's arithmetic does not depend on which
rank computes it, so the result equals the one-GPU layer bit for bit. A token routed to two
experts of one rank sends its row twice (no de-duplication). The dispatch plan is host logic
(numpy over the step's ids); the expert FFN and the reducer are the library's kernels. The
exchange and the plan are exercised with gloo ranks on CPU (tests/test_expert_parallel.py),
where the two compute callables are CPU stand-ins.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Optional

import numpy as np
import torch
import torch.distributed as dist


@dataclasses.dataclass(frozen=True)
class Plan:
    """Where each valid routed pair of this rank goes."""
    order: np.ndarray        # int64 [n_send]: pair indices t*K + j, grouped by owner, ascending within
    local_ids: np.ndarray    # int32 [n_send]: the owner-local expert id of each sent pair
    send_counts: np.ndarray  # int64 [world]: pairs sent to each rank


def experts_per_rank(num_experts: int, world: int) -> int:
    if num_experts % world:
        raise ValueError(f"{num_experts} experts do not split evenly over {world} ranks")
    return num_experts // world


def dispatch_plan(ids: np.ndarray, num_experts: int, world: int) -> Plan:
    """ids int [M][K] (pairs with ids outside [0, E) are skipped: they send nothing)."""
    per = experts_per_rank(num_experts, world)
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    valid = (flat >= 0) & (flat < num_experts)
    pairs = np.flatnonzero(valid)
    owner = flat[pairs] // per
    order = pairs[np.argsort(owner, kind="stable")]
    send_counts = np.bincount(owner, minlength=world).astype(np.int64)
    local_ids = (flat[order] % per).astype(np.int32)
    return Plan(order, local_ids, send_counts)


def _exchange_counts(send_counts: np.ndarray, group) -> np.ndarray:
    world = dist.get_world_size(group)
    s = torch.from_numpy(send_counts.astype(np.int64))
    r = torch.empty(world, dtype=torch.int64)
    if dist.get_backend(group) == "nccl":
        s, r = s.cuda(), r.cuda()
    dist.all_to_all_single(r, s, group=group)
    return r.cpu().numpy()


class ExpertParallelLayer:
    """The routed layer with its experts split over the ranks of ``group``.

    run_experts(rows [n][H] BF16 bits as int16, local_ids [n] int32) -> y [n][H] float32
    combine(y_pairs [M*K][H] float32, ids [M][K] int32, weights [M][K] float32) -> out [M][H]
    Both default to the library (see ``library_callables``); tests pass CPU stand-ins.
    """

    def __init__(self, group, num_experts: int, top_k: int, hidden: int,
                 run_experts: Callable, combine: Callable, device: Optional[torch.device] = None):
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.E, self.K, self.H = num_experts, top_k, hidden
        self.per = experts_per_rank(num_experts, self.world)
        self.run_experts = run_experts
        self.combine = combine
        self.device = device if device is not None else torch.device("cpu")

    def forward(self, hidden: torch.Tensor, ids: torch.Tensor, weights: torch.Tensor) -> torch.Tensor:
        M = hidden.shape[0]
        plan = dispatch_plan(ids.cpu().numpy(), self.E, self.world)
        recv_counts = _exchange_counts(plan.send_counts, self.group)
        order = torch.from_numpy(plan.order).to(self.device)
        # the BF16 rows travel as 2-byte float16 words (the collectives have no int16 type; the
        # bits are copied, never converted)
        rows16 = hidden.reshape(M, self.H).view(torch.float16)
        send_rows = rows16.index_select(0, torch.div(order, self.K, rounding_mode="floor"))
        send_ids = torch.from_numpy(plan.local_ids).to(self.device)
        n_recv = int(recv_counts.sum())
        recv_rows = torch.empty((n_recv, self.H), dtype=torch.float16, device=self.device)
        recv_ids = torch.empty(n_recv, dtype=torch.int32, device=self.device)
        sc, rc = plan.send_counts.tolist(), recv_counts.tolist()
        dist.all_to_all_single(recv_rows, send_rows.contiguous(), rc, sc, group=self.group)
        dist.all_to_all_single(recv_ids, send_ids, rc, sc, group=self.group)
        if n_recv:
            y_recv = self.run_experts(recv_rows.view(hidden.dtype), recv_ids)
        else:
            y_recv = torch.empty((0, self.H), dtype=torch.float32, device=self.device)
        y_back = torch.empty((len(plan.order), self.H), dtype=torch.float32, device=self.device)
        dist.all_to_all_single(y_back, y_recv.contiguous(), sc, rc, group=self.group)
        y_pairs = torch.zeros((M * self.K, self.H), dtype=torch.float32, device=self.device)
        if len(plan.order):
            y_pairs.index_copy_(0, order, y_back)
        return self.combine(y_pairs, ids, weights)


def library_callables(w13_local, s13_local, w2_local, s2_local, hidden: int, inter: int, num_experts: int,
                      top_k: int, max_rows: int, max_tokens: int):
    """The library's kernels as the layer's two callables, for one rank's expert shard.

    w13_local / w2_local and their scales are this rank's E/world experts (the layouts of
    moe_fp8_forward); max_rows bounds the rows a rank can receive in one step, max_tokens the
    rank's own tokens. Workspaces are allocated here, once."""
    from . import _lib as L

    E_local = w13_local.shape[0]
    local_shape = L.make_shape(hidden, inter, E_local, 1, max_rows)
    ws = torch.empty(L.moe_fp8_workspace_bytes(local_shape), dtype=torch.uint8, device="cuda")
    L.moe_fp8_workspace_init(ws, local_shape)
    full_shape = L.make_shape(hidden, inter, num_experts, top_k, max_tokens)

    def run_experts(rows, local_ids):
        n = rows.shape[0]
        y = torch.empty((n, hidden), dtype=torch.float32, device="cuda")
        L.moe_fp8_forward_partials(rows, local_ids.reshape(n, 1).contiguous(), n, w13_local, s13_local, w2_local,
                                   s2_local, y, ws, local_shape)
        return y

    def combine(y_pairs, ids, weights):
        M = ids.shape[0]
        out = torch.empty((M, hidden), dtype=torch.int16, device="cuda")
        L.moe_fp8_combine_pairs(y_pairs, ids, weights, M, out, full_shape)
        return out

    return run_experts, combine
