"""The grouped GEMMs' bounded pipeline waits, made to run out on purpose
through the library's test hook: each CTA withholds the copy of its first
unit's scales and zeros, its dequantisation warps' wait for them gives up
after 2 ms, and the kernel sets W4_DEV_PIPELINE_TIMEOUT, drains what it
started and exits.  Nothing faults or hangs: every wait in the kernels is
bounded, and the test then checks that the context still computes the
normal result bit for bit."""
import time

import pytest

from helpers import gpu_inputs, gpu_weights

pytestmark = pytest.mark.gpu


@pytest.fixture
def hooks(lib):
    clib = lib.load_library()
    yield clib
    clib.w4_test_pipeline_hooks(0, 0)


@pytest.mark.parametrize("name", ["tiny", "layer256"])
def test_withheld_scales_time_out_and_the_context_stays_usable(lib, hooks, name):
    import torch
    cfg, x, lg, _, _ = gpu_inputs(name)
    gu, dn = gpu_weights(name)
    ids, w = lib.w4_moe_route(lg, cfg.k)
    al, xg = lib.w4_moe_align_gather(ids, x, cfg.E, 16)
    h_ref = lib.w4_grouped_gemm_gate_up(xg, *gu, al)
    y_ref = lib.w4_grouped_gemm_down(h_ref, *dn, al)
    torch.cuda.synchronize()

    hooks.w4_test_pipeline_hooks(2_000_000, 1)
    st_gu = torch.zeros(1, dtype=torch.int32, device="cuda")
    st_dn = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    lib.w4_grouped_gemm_gate_up(xg, *gu, al, dev_status=st_gu)
    lib.w4_grouped_gemm_down(h_ref, *dn, al, dev_status=st_dn)
    counters, out = lib.w4_moe_combine_prepare(ids, cfg.E, cfg.d)
    st_dc = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.w4_grouped_gemm_down_combine(h_ref, *dn, al, ids, w, counters, out, dev_status=st_dc)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    for st in (st_gu, st_dn, st_dc):
        assert int(st.item()) & lib.W4_DEV_PIPELINE_TIMEOUT
    assert elapsed < 5.0          # three launches that each gave up after ~2 ms

    hooks.w4_test_pipeline_hooks(0, 0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    h = lib.w4_grouped_gemm_gate_up(xg, *gu, al, dev_status=st)
    y = lib.w4_grouped_gemm_down(h, *dn, al, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # the columns gate_up writes: m values and the quarter sums of the groups
    # of 64 (padded to a multiple of 16), in the rows below num_padded
    npad = int(al["num_padded"].item())
    cols = cfg.m + 16 * ((4 * (cfg.m // 64) + 15) // 16)
    assert torch.equal(h[:npad, :cols].view(torch.int16), h_ref[:npad, :cols].view(torch.int16))
    flat = ids.reshape(-1).cpu().numpy()
    valid = torch.from_numpy((flat >= 0) & (flat < cfg.E)).cuda()
    assert torch.equal(y[valid].view(torch.int32), y_ref[valid].view(torch.int32))


def test_short_limit_alone_changes_nothing(lib, hooks):
    """A short limit with nothing withheld: a normal pipeline never waits
    that long, so the result is the normal one and no bit is set."""
    import torch
    name = "ragged"
    cfg, x, lg, _, _ = gpu_inputs(name)
    gu, dn = gpu_weights(name)
    ids, w = lib.w4_moe_route(lg, cfg.k)
    al, xg = lib.w4_moe_align_gather(ids, x, cfg.E, 16)
    h_ref = lib.w4_grouped_gemm_gate_up(xg, *gu, al)
    torch.cuda.synchronize()
    hooks.w4_test_pipeline_hooks(50_000_000, 0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    h = lib.w4_grouped_gemm_gate_up(xg, *gu, al, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    npad = int(al["num_padded"].item())
    cols = cfg.m + 16 * ((4 * (cfg.m // 64) + 15) // 16)
    assert torch.equal(h[:npad, :cols].view(torch.int16), h_ref[:npad, :cols].view(torch.int16))
