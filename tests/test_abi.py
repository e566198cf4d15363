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
    assert clib.w4_abi_version() == 9
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
    # down with the folded combine: NULL counters, misaligned out, then the
    # down checks; the counter preparation needs d % 128 == 0
    cargs = [fake, 16, 256, 128, 8, 2, 16, fake, fake, fake, 64, fake, fake, fake, fake, None,
             fake, fake, None, None]
    assert clib.w4_grouped_gemm_down_combine(*cargs) == 1
    cargs[15] = fake
    cargs[17] = P(0x10004)
    assert clib.w4_grouped_gemm_down_combine(*cargs) == 3
    cargs[17] = fake
    cargs[10] = 128
    assert clib.w4_grouped_gemm_down_combine(*cargs) == 2
    assert clib.w4_moe_combine_prepare(fake, 4, 2, 8, 200, fake, fake, None) == 2
    assert clib.w4_moe_combine_prepare(None, 4, 2, 8, 256, fake, fake, None) == 1
    assert clib.w4_moe_combine_prepare(fake, 4, 2, 8, 256, fake, P(0x10002), None) == 3
    # gather: d must be a multiple of 8
    assert clib.w4_gather_activations(fake, 4, 252, 2, 8, 16, fake, fake, fake, None, None) == 2
    # workspace too small
    assert clib.w4_moe_layer(fake, fake, fake, 16, 256, 128, 8, 2, 16, fake, fake, fake, 128,
                             fake, fake, fake, 64, fake, 16, fake, None, None) == 6
    # the host-buffer layer: NULL host buffer, workspace too small, misaligned
    # workspace (all before any copy or launch); the staging follows the layer
    hargs = [fake, fake, fake, 16, 256, 128, 8, 2, 16, fake, fake, fake, 128, fake, fake, fake,
             64, fake, 1 << 30, None, None, None]
    assert clib.w4_moe_layer_host(*hargs) == 1
    need = clib.w4_moe_layer_host_workspace_size(16, 256, 128, 8, 2, 16)
    assert need > clib.w4_moe_layer_workspace_size(16, 256, 128, 8, 2, 16) + 2 * 2 * 16 * 256
    hargs[19] = fake
    hargs[18] = need - 1
    assert clib.w4_moe_layer_host(*hargs) == 6
    hargs[18] = need
    hargs[17] = P(0x10040)
    assert clib.w4_moe_layer_host(*hargs) == 3


def test_binding_raises_on_cpu_tensors():
    import torch
    with pytest.raises(ValueError):
        w4.w4_moe_route(torch.zeros(4, 8), 2)


def test_beside_the_layer_validates_without_launching(clib):
    """RMSNorm, the sampler and the dense linear reject bad arguments on the
    host, before any device call; empty batches are accepted."""
    P = ctypes.c_void_p
    fake = P(0x10000)          # never dereferenced: validation fails first
    odd = P(0x10004)           # 4-byte but not 16-byte aligned
    odd2 = P(0x10002)          # not 4-byte aligned
    # RMSNorm
    assert clib.w4_rmsnorm(fake, fake, 4, 100, 1e-6, fake, None) == 2      # d % 8
    assert clib.w4_rmsnorm(fake, fake, 4, 64, -1.0, fake, None) == 1       # eps < 0
    assert clib.w4_rmsnorm(odd, fake, 4, 64, 1e-6, fake, None) == 3        # misaligned x
    assert clib.w4_rmsnorm(None, fake, 0, 64, 1e-6, None, None) == 0       # empty batch
    # sampler
    big = 1 << 24
    assert clib.w4_sample_logits(fake, 4, 0, 1, 0, fake, None, None, fake, big, None) == 1
    assert clib.w4_sample_logits(fake, 4, 1000, 1, 0, None, None, None, fake, big, None) == 1
    assert clib.w4_sample_logits(odd2, 4, 1000, 1, 0, fake, None, None, fake, big, None) == 3
    assert clib.w4_sample_logits(fake, 4, 1000, 1, 0, fake, None, None, fake, 16, None) == 6
    assert clib.w4_sample_logits(None, 0, 1000, 1, 0, None, None, None, None, 0, None) == 0
    assert clib.w4_sample_logits_workspace_size(256, 262144) == (2048 + 256) * 32
    assert clib.w4_fused_entropy(fake, 4, 1000, None, fake, big, None) == 1
    assert clib.w4_gumbel_argmax_sample(fake, 4, 1000, 1, 0, None, None, fake, big, None) == 1
    # dense linear: shapes, groups, alignment, workspace
    lin = [fake, 4, 512, 256, fake, fake, fake, 128, fake, big, fake, None, None]
    assert clib.w4_w4a16_linear(*lin[:3], 200, *lin[4:]) == 2              # N % 128
    assert clib.w4_w4a16_linear(*lin[:7], 96, *lin[8:]) == 2               # group
    assert clib.w4_w4a16_linear(fake, 4, 128, 256, *lin[4:]) == 2          # K < 256
    assert clib.w4_w4a16_linear(fake, 4, 8192, 256, *lin[4:]) == 2         # 64 groups
    assert clib.w4_w4a16_linear(odd, *lin[1:]) == 3
    assert clib.w4_w4a16_linear(*lin[:9], 16, *lin[10:]) == 6
    assert clib.w4_w4a16_linear(None, 0, 512, 256, None, None, None, 128, None, 0, None, None,
                                None) == 0


def test_linear_split_rule_depends_on_the_shape_only(clib):
    """The contraction split (visible in the workspace's partial sums): about
    128 units of 128 weight rows x 256 tokens, at most 8 splits of at least
    4 steps of 64 codes; no partial buffer when there is no split."""
    ws = clib.w4_w4a16_linear_workspace_size
    base = ws(256, 2816, 16384, 128)              # 128 panels: no split
    assert ws(256, 2816, 4096, 128) - base == 4 * 256 * 4096 * 4     # 32 panels: 4 splits
    one = ws(33, 2816, 128, 128)                  # one panel: 8 splits
    assert one >= 8 * 33 * 128 * 4 and one - 8 * 33 * 128 * 4 < 2 * 48 * 2816 + 4096
    assert ws(16, 256, 128, 128) < 16 * 256 * 2 + 4096                # 4 steps: no split
