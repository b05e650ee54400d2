"""The C ABI from C (no GPU): tests/abi_client.c is compiled as C11 against include/moe_fp8.h with
warnings as errors, linked to libmoe_fp8.so and run. Its answers must match the header's status
codes and the Python binding's."""
import os
import shutil
import subprocess

import pytest

from fp8_block_scaled_router_gb300 import _lib as L
from fp8_block_scaled_router_gb300 import build as B

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

OK, INVALID_ARG, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3


@pytest.fixture(scope="module")
def client_output(tmp_path_factory):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    lib = B.build()
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(B.nvcc()))), "include")
    exe = str(tmp_path_factory.mktemp("abi") / "abi_client")
    libdir = os.path.dirname(lib)
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", cuda_inc, os.path.join(HERE, "abi_client.c"), "-o", exe, "-L", libdir, "-lmoe_fp8",
                    f"-Wl,-rpath,{libdir}"], check=True, capture_output=True, text=True)
    run = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=60)
    out = {}
    for line in run.stdout.splitlines():
        k, v = line.split(" ", 1)
        out[k] = v
    return out


def test_c_client_sees_the_bindings_answers(client_output):
    o = client_output
    assert o["version"] == L.moe_fp8_version()
    s = L.make_shape(2048, 768, 128, 8, 16)
    assert int(o["ws_bytes"]) == L.moe_fp8_workspace_bytes(s) > 0


def test_c_client_validation_codes(client_output):
    o = {k: int(v) for k, v in client_output.items() if k != "version"}
    assert o["ws_bytes_bad_e"] == 0 and o["ws_bytes_bad_h"] == 0
    assert o["forward_ok_m0"] == OK
    assert o["forward_null_hidden"] == INVALID_ARG
    assert o["forward_m_above_max"] == INVALID_ARG
    assert o["forward_small_ws"] == WORKSPACE
    assert o["forward_bad_shape"] == UNSUPPORTED
    assert o["route_ok_m0"] == OK
    assert o["route_misaligned_bias"] == INVALID_ARG
    assert o["route_bad_shape"] == UNSUPPORTED
    assert o["read_status_null"] == INVALID_ARG
