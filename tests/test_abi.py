"""The C-ABI library builds, loads and exports every symbol of include/w4moe.h;
host-side argument validation answers with status codes (no GPU needed:
nothing here launches a kernel)."""
import ctypes
import os
import subprocess

import pytest

import w4a16_moe_expert_sync_gb300 as w4
from w4a16_moe_expert_sync_gb300 import build as w4build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def clib():
    w4build.build()
    return w4.load_library()


def test_library_exports_every_header_function(clib):
    names = w4.header_functions()
    assert len(names) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", w4build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in names:
        assert n in exported, n
        assert hasattr(clib, n)


def test_header_compiles_as_plain_c():
    src = '#include "w4moe.h"\nint main(void){return W4_OK + W4MOE_ABI_VERSION - 1;}\n'
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-x", "c",
                        "-I", os.path.join(ROOT, "include"), "-"], input=src, text=True,
                       capture_output=True)
    assert r.returncode == 0, r.stderr


def test_status_strings_and_version(clib):
    assert clib.w4_abi_version() == 6
    assert clib.w4_status_string(0) == b"W4_OK"
    assert clib.w4_status_string(2) == b"W4_ERR_UNSUPPORTED_SHAPE"
    assert clib.w4_status_string(99) == b"W4_ERR_UNKNOWN"


def test_align_capacity(clib):
    assert clib.w4_moe_align_capacity(256, 8, 128, 16) == ((2048 + 128 * 15 + 15) // 16) * 16
    assert clib.w4_moe_align_capacity(16, 2, 8, 32) == ((32 + 8 * 31 + 31) // 32) * 32
    assert clib.w4_moe_align_capacity(1, 1, 1, 17) == -1          # bad block_m
    assert clib.w4_moe_layer_workspace_size(256, 2816, 704, 128, 8, 16) > 2048 * 2816 * 4


def test_argument_validation_without_launching(clib):
    P = ctypes.c_void_p
    fake = P(0x10000)          # never dereferenced: validation fails first
    odd = P(0x10004)
    # NULL pointers
    assert clib.w4_quantize(None, 1, 1, 128, 128, fake, fake, fake, None) == 1
    assert clib.w4_moe_route(None, 1, 8, 2, fake, fake, None) == 1
    # bad group / shapes
    assert clib.w4_quantize(fake, 1, 1, 100, 100, fake, fake, fake, None) == 2
    assert clib.w4_moe_route(fake, 4, 8, 40, fake, fake, None) == 2
    # block_m must be a supported power of two
    assert clib.w4_moe_align(fake, 4, 2, 8, 24, fake, fake, fake, fake, None, None) == 1
    # gate_up needs d % 128 == 0, m % 64 == 0, group == 128
    args = [fake, 16, 200, 128, 8, 2, 16, fake, fake, fake, 128, fake, fake, fake, None, None]
    assert clib.w4_grouped_gemm_gate_up(*args) == 2
    args[2] = 256
    args[10] = 64
    assert clib.w4_grouped_gemm_gate_up(*args) == 2
    # misaligned activation pointer
    args[10] = 128
    args[0] = odd
    assert clib.w4_grouped_gemm_gate_up(*args) == 3
    assert b"aligned" in clib.w4_last_error_detail()
    # down group must be 64
    dargs = [fake, 16, 256, 128, 8, 2, 16, fake, fake, fake, 128, fake, fake, fake, None, None]
    assert clib.w4_grouped_gemm_down(*dargs) == 2
    # gather: d must be a multiple of 8
    assert clib.w4_gather_activations(fake, 4, 252, 2, 8, 16, fake, fake, fake, None) == 2
    # workspace too small
    assert clib.w4_moe_layer(fake, fake, fake, 16, 256, 128, 8, 2, 16, fake, fake, fake, 128,
                             fake, fake, fake, 64, fake, 16, fake, None, None) == 6


def test_binding_raises_on_cpu_tensors():
    import torch
    with pytest.raises(ValueError):
        w4.w4_moe_route(torch.zeros(4, 8), 2)
