"""moe_fp8_forward_noalloc: the layer for callers that cannot allocate device memory.

Such callers (code running while a memory pool is locked or resized, allocator-free
callbacks, integrations without a device allocator) get the few-row forward with its
scratch compiled into the library. Checked through the C ABI against moe_fp8_forward,
which uses a caller workspace, on two calls in a row (the scratch keeps the previous
call's contents, so the second call must not depend on them). Collected last on purpose.
"""
import numpy as np
import pytest
import torch

from fp8_block_scaled_router_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build_lib():
    from fp8_block_scaled_router_gb300 import build
    build.build()


@pytest.mark.parametrize("name,M", [("decode", 1), ("verify_skewed", 12)])
def test_noalloc_matches_workspace_forward_twice(name, M):
    from fp8_block_scaled_router_gb300 import _lib as L
    from gpu_harness import GpuMoE, to_dev

    x = inputs.make(name, tokens=2 * M) if name == "decode" else inputs.make(name, M=2 * M)
    g = GpuMoE(x, M)
    for call in range(2):
        hid = to_dev(x.hidden[call * M:(call + 1) * M])
        ids, w = g.route(hid, M)
        # the workspace form of the same two kernels (moe_fp8_forward itself when M*K <= 64)
        ref = torch.empty((M, g.H), dtype=torch.int16, device="cuda")
        L.moe_fp8_gate_up_direct(hid, ids, M, g.w13, g.s13, g.ws, g.shape)
        L.moe_fp8_down_combine(ids, w, M, g.w2, g.s2, ref, g.ws, g.shape)
        if M * g.K <= 64:
            assert torch.equal(ref, g.forward(hid, ids, w, M))
        out = torch.full_like(ref, 0x7ABC)
        L.moe_fp8_forward_noalloc(hid, ids, w, M, g.w13, g.s13, g.w2, g.s2, out, g.shape)
        torch.cuda.synchronize()
        # same kernels and arithmetic: bitwise equal (the parity tests' tolerance is looser)
        assert torch.equal(out, ref), f"call {call}"


@pytest.mark.parametrize("name,M", [("verify_skewed", 12), ("decode", 32)], ids=["R96", "R256"])
def test_noalloc_against_oracle(name, M):
    """The no-workspace call above the 64 routed rows where moe_fp8_forward sorts rows into
    expert tiles (the range only the pair kernels serve), against the oracle's output."""
    import oracle
    from fp8_block_scaled_router_gb300 import _lib as L
    from gpu_harness import GpuMoE, check_out, oracle_forward, to_dev, u16

    oracle.build()
    x = inputs.make(name, tokens=M) if name == "decode" else inputs.make(name, M=M)
    g = GpuMoE(x, M)
    ids_o, w_o = oracle.route(x.hidden[:M], x.router_w, x.bias, g.K)
    out = torch.full((M, g.H), 0x7ABC, dtype=torch.int16, device="cuda")
    L.moe_fp8_forward_noalloc(to_dev(x.hidden[:M]), to_dev(ids_o), to_dev(w_o), M, g.w13, g.s13, g.w2, g.s2,
                              out, g.shape)
    torch.cuda.synchronize()
    check_out(u16(out), oracle_forward(x, x.hidden[:M], ids_o, w_o), f"noalloc {name} R={M * g.K}")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from fp8_block_scaled_router_gb300 import _lib as L
    fake = 0x10000
    big = L.make_shape(2048, 4096, 128, 8, 64)      # 64 * 8 rows > the few-row limit
    assert L.moe_fp8_forward_noalloc(fake, fake, fake, 64, fake, fake, fake, fake, fake, big,
                                     stream=0, check=False) == 2
    wide = L.make_shape(2048, 4096, 128, 8, 32)     # 256 rows x 4096 columns > 1 MiB
    assert L.moe_fp8_forward_noalloc(fake, fake, fake, 32, fake, fake, fake, fake, fake, wide,
                                     stream=0, check=False) == 2
