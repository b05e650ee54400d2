"""moe_fp8_route_forward_host: the layer for tokens held in host memory, one call per batch.

It must equal moe_route followed by moe_fp8_forward on the same inputs (bitwise: the same
kernels run on a device copy of the hidden rows), leave the routing in the workspace view,
and copy only the M rows it was given."""
import numpy as np
import pytest
import torch

from fp8_block_scaled_router_gb300 import inputs

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_harness import GpuMoE, to_dev


CASES = [("decode", 1, True), ("verify_skewed", 12, True), ("decode", 300, True), ("decode", 1, False),
         ("verify_skewed", 12, False)]


@pytest.mark.parametrize("name,M,pinned", CASES, ids=[f"{n}-M{m}-{'pinned' if p else 'pageable'}" for n, m, p in CASES])
def test_host_call_equals_device_calls(name, M, pinned):
    # pinned buffers are read and written by the kernels in place; pageable ones are copied
    from fp8_block_scaled_router_gb300 import _lib as L

    x = inputs.make(name, tokens=M) if name == "decode" else inputs.make(name, M=M)
    g = GpuMoE(x, M)
    hid_np = np.ascontiguousarray(x.hidden[:M]).view(np.int16)
    host_in = torch.from_numpy(hid_np.copy())
    host_out = torch.full((M + 2, g.H), 0x1234, dtype=torch.int16)
    if pinned:
        host_in, host_out = host_in.pin_memory(), host_out.pin_memory()
    L.moe_fp8_route_forward_host(host_in, host_out, M, g.router, g.bias, True, g.w13, g.s13, g.w2, g.s2, g.ws,
                                 g.shape)
    torch.cuda.synchronize()
    v = L.moe_fp8_workspace_view(g.ws, g.shape)
    base = g.ws.data_ptr()
    ids_h = g.ws[v.topk_ids - base: v.topk_ids - base + M * g.K * 4].view(torch.int32).reshape(M, g.K).clone()
    w_h = g.ws[v.topk_w - base: v.topk_w - base + M * g.K * 4].view(torch.float32).reshape(M, g.K).clone()

    hid = to_dev(x.hidden[:M])
    ids, w = g.route(hid, M)
    ref = g.forward(hid, ids, w, M)
    torch.cuda.synchronize()
    assert torch.equal(ids_h, ids) and torch.equal(w_h, w)
    assert torch.equal(host_out[:M], ref.cpu())
    assert torch.all(host_out[M:] == 0x1234)  # rows past M untouched
    assert g.status() == 0
