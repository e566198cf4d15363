"""The whole routed-expert layer on the GPU (router, align, gate_up +
activation, down, fixed-order combine) against the float64 oracle:
max|gpu - oracle| / rms(oracle) <= 2e-2 on the bf16 output, expert ids
bit-exact, and reruns bit-identical ("Inference: Making every denoising pass
fast" -- Quantisation alone leaves a sparse execution problem, The final best
W4 MoE kernel: zero bit mismatches between two runs)."""
import numpy as np
import pytest

import oracle
from helpers import (bf16_round, gpu_inputs, gpu_weights, oracle_weights, rel_max_err,
                     torch_bf16_to_f64)
from w4a16_moe_expert_sync_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
LAYER_TOL = 2e-2


def _layer(lib, name, block_m=16, status=None):
    cfg, x, lg, x_bits, logits = gpu_inputs(name)
    gu, dn = gpu_weights(name)
    ids, w = lib.w4_moe_route(lg, cfg.k)
    out = lib.w4_moe_layer(x, ids, w, gu, dn, block_m=block_m, dev_status=status)
    return cfg, x_bits, logits, ids, w, out


@pytest.mark.parametrize("block_m", [16, 32])
@pytest.mark.parametrize("name", ["tiny", "ragged", "bigjobs"])
def test_layer_matches_oracle(lib, name, block_m):
    import torch
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cfg, x_bits, logits, ids, w, out = _layer(lib, name, block_m, status)
    oids, ow = oracle.route(logits, cfg.k)
    assert np.array_equal(ids.cpu().numpy(), oids)
    ogu, odn = oracle_weights(cfg, range(cfg.E))
    ref = oracle.moe_layer(x_bits, ogu, odn, oids, ow)
    err = rel_max_err(torch_bf16_to_f64(out), ref)
    floor = rel_max_err(bf16_round(ref), ref)
    print(f"{name} block_m={block_m}: max|gpu-oracle|/rms = {err:.3e} "
          f"(bf16 rounding of the exact result alone: {floor:.3e})")
    assert err <= LAYER_TOL
    assert int(status.item()) == 0


# Elementwise bar beside the max/rms one: each output element may differ
# from the oracle by its own bf16 rounding (<= 2^-8 |out|) plus TAU_OUT of the
# output's rms.  TAU_OUT bounds the compute error before that rounding: fp16
# rounding of every dequantised weight, of each group's constant -z*s and of
# h leave ~1e-3 rms relative error in y (see test_gpu_gemm.py), which the
# weighted sum of a token's k rows keeps at that level; ~10x that rms.
TAU_OUT = 1e-2


@pytest.mark.parametrize("name", ["layer256", "zipf256", "canvas2048", "sweep_M1", "sweep_M8",
                                  "sweep_M64"])
def test_layer_full_size(lib, name):
    """Pages' layer shape, every M of the sweep, skewed routing and the
    multi-canvas batch.  Every token is compared with the oracle, except on
    the 2048-token canvas, where the tokens compared reach every 32-slot job
    of every expert (each expert there spans several jobs)."""
    import torch
    from helpers import elementwise_excess, oracle_layer
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cfg, x_bits, logits, ids, w, out = _layer(lib, name, 16, status)
    toks, oids, ow, ref, _, _ = oracle_layer(name, "cover" if name == "canvas2048" else "all")
    assert np.array_equal(ids.cpu().numpy(), oids)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), ow.view(np.uint32))
    got = torch_bf16_to_f64(out)[toks]
    err = rel_max_err(got, ref)
    floor = rel_max_err(bf16_round(ref), ref)
    excess = elementwise_excess(got, ref, 2.0 ** -8)
    print(f"{name}: {len(toks)} tokens, max|gpu-oracle|/rms = {err:.3e} (bf16 rounding alone: "
          f"{floor:.3e}); elementwise excess over 2^-8|ref| = {excess:.3e} rms")
    assert err <= LAYER_TOL
    assert excess <= TAU_OUT
    assert int(status.item()) == 0


@pytest.mark.parametrize("name", ["ragged", "layer256"])
def test_layer_reruns_are_bit_identical(lib, name):
    import torch
    cfg, x, lg, _, _ = gpu_inputs(name)
    gu, dn = gpu_weights(name)
    ids, w = lib.w4_moe_route(lg, cfg.k)
    a = lib.w4_moe_layer(x, ids, w, gu, dn)
    b = lib.w4_moe_layer(x, ids, w, gu, dn)
    ws = torch.full((lib.w4_moe_layer_workspace_size(cfg.M, cfg.d, cfg.m, cfg.E, cfg.k),),
                    255, dtype=torch.uint8, device="cuda")     # dirty workspace
    c = lib.w4_moe_layer(x, ids, w, gu, dn, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_layer_skips_invalid_ids_and_flags_them(lib):
    import torch
    name = "tiny"
    cfg, x, lg, x_bits, logits = gpu_inputs(name)
    gu, dn = gpu_weights(name)
    oids, ow = oracle.route(logits, cfg.k)
    bad = oids.copy()
    bad[3, 1] = cfg.E + 2
    bad[9, 0] = -1
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = lib.w4_moe_layer(x, torch.from_numpy(bad).cuda(), torch.from_numpy(ow).cuda(), gu, dn,
                           dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & lib.W4_DEV_BAD_EXPERT_ID
    ogu, odn = oracle_weights(cfg, range(cfg.E))
    ref = oracle.moe_layer(x_bits, ogu, odn, bad, ow)
    assert rel_max_err(torch_bf16_to_f64(out), ref) <= LAYER_TOL


def test_layer_with_no_tokens(lib):
    import torch
    cfg = wl.CONFIGS["tiny"]
    gu, dn = gpu_weights("tiny")
    x = torch.zeros((0, cfg.d), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((0, cfg.k), dtype=torch.int32, device="cuda")
    w = torch.zeros((0, cfg.k), dtype=torch.float32, device="cuda")
    out = lib.w4_moe_layer(x, ids, w, gu, dn)
    torch.cuda.synchronize()
    assert out.shape == (0, cfg.d)


@pytest.mark.parametrize("name", ["tiny", "ragged", "layer256", "zipf256"])
def test_layer_equals_the_separate_calls(lib, name):
    """w4_moe_layer's out is bit-identical to align+gather, gate_up, down and
    w4_moe_combine_fixed_order called one by one (its launches overlap at their
    boundaries; the arithmetic and its order are the same), also from a dirty
    workspace."""
    import torch
    cfg, x, lg, _, _ = gpu_inputs(name)
    gu, dn = gpu_weights(name)
    ids, w = lib.w4_moe_route(lg, cfg.k)
    al, xg = lib.w4_moe_align_gather(ids, x, cfg.E, 16)
    h = lib.w4_grouped_gemm_gate_up(xg, *gu, al)
    y = lib.w4_grouped_gemm_down(h, *dn, al)
    ref = lib.w4_moe_combine_fixed_order(y, ids, w, cfg.E)
    ws = torch.full((lib.w4_moe_layer_workspace_size(cfg.M, cfg.d, cfg.m, cfg.E, cfg.k),),
                    255, dtype=torch.uint8, device="cuda")
    out = lib.w4_moe_layer(x, ids, w, gu, dn, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_layer_token_with_no_valid_expert_is_zero(lib):
    """A token whose k ids are all invalid contributes to no expert: its output
    row is exactly zero, the status flags the ids, other rows as separately."""
    import torch
    name = "tiny"
    cfg, x, lg, _, logits = gpu_inputs(name)
    gu, dn = gpu_weights(name)
    oids, ow = oracle.route(logits, cfg.k)
    bad = oids.copy()
    bad[5, :] = -1
    ids_d, w_d = torch.from_numpy(bad).cuda(), torch.from_numpy(ow).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = lib.w4_moe_layer(x, ids_d, w_d, gu, dn, dev_status=status)
    al, xg = lib.w4_moe_align_gather(ids_d, x, cfg.E, 16)
    h = lib.w4_grouped_gemm_gate_up(xg, *gu, al)
    y = lib.w4_grouped_gemm_down(h, *dn, al)
    ref = lib.w4_moe_combine_fixed_order(y, ids_d, w_d, cfg.E)
    torch.cuda.synchronize()
    assert int(status.item()) & lib.W4_DEV_BAD_EXPERT_ID
    assert torch.count_nonzero(out[5].view(torch.int16)) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_layer_activation_range_is_flagged(lib):
    """The GEMMs' operands are fp16 (a reading of this build; the pages'
    kernels use bf16).  A token whose activations exceed fp16's range
    (|x| up to ~4e5 here) is saturated and W4_DEV_FP16_RANGE is raised;
    tokens whose activations lie mostly below 2^-14 (fp16 subnormals, absolute
    step 2^-24) keep the layer's bound; every other token is unaffected."""
    import torch
    from helpers import bf16_bits_to_f64
    name = "tiny"
    cfg = wl.CONFIGS[name]
    x_bits = wl.activations(cfg).copy()
    xf = bf16_bits_to_f64(x_bits)
    big, small = 3, [5, 6]
    xf[big] *= 1e5
    xf[small] *= 1e-4
    x_bits = wl.f32_to_bf16_bits(xf.astype(np.float32))
    assert np.abs(bf16_bits_to_f64(x_bits[big])).max() > 65504
    assert np.mean(np.abs(bf16_bits_to_f64(x_bits[small])) < 2.0 ** -14) > 0.3
    logits = wl.router_logits(cfg)
    gu, dn = gpu_weights(name)
    oids, ow = oracle.route(logits, cfg.k)
    ids_d, w_d = torch.from_numpy(oids).cuda(), torch.from_numpy(ow).cuda()
    x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = lib.w4_moe_layer(x, ids_d, w_d, gu, dn, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & lib.W4_DEV_FP16_RANGE
    ogu, odn = oracle_weights(cfg, range(cfg.E))
    ref = oracle.moe_layer(x_bits, ogu, odn, oids, ow)
    keep = np.array([t for t in range(cfg.M) if t != big])
    err = rel_max_err(torch_bf16_to_f64(out)[keep], ref[keep])
    print(f"activation range: other tokens max|gpu-oracle|/rms = {err:.3e}")
    assert err <= LAYER_TOL
    # the same batch without the out-of-range row raises nothing
    x_ok = x.clone()
    x_ok[big] = x[0]
    status.zero_()
    lib.w4_moe_layer(x_ok, ids_d, w_d, gu, dn, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_layer_rejects_shapes_beyond_shared_memory_before_launching(lib):
    """gate_up with d = 5120 (40 groups of 128) needs more shared memory for a
    unit's scales and zeros than an SM has: the layer is rejected with
    W4_ERR_UNSUPPORTED_SHAPE before its first launch, so out keeps its
    contents."""
    import torch
    M, d, m, E, k = 4, 5120, 128, 8, 2
    x = torch.zeros((M, d), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((M, k), dtype=torch.int32, device="cuda")
    ids[:, 1] = 1
    w = torch.full((M, k), 0.5, dtype=torch.float32, device="cuda")
    gu = (torch.zeros((E, 2 * m, d // 2), dtype=torch.uint8, device="cuda"),
          torch.zeros((E, 2 * m, d // 128), dtype=torch.float16, device="cuda"),
          torch.zeros((E, 2 * m, d // 128), dtype=torch.float16, device="cuda"))
    dn = (torch.zeros((E, d, m // 2), dtype=torch.uint8, device="cuda"),
          torch.zeros((E, d, m // 64), dtype=torch.float16, device="cuda"),
          torch.zeros((E, d, m // 64), dtype=torch.float16, device="cuda"))
    out = torch.full((M, d), 3.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.W4Error) as e:
        lib.w4_moe_layer(x, ids, w, gu, dn, out=out)
    assert e.value.status == 2 and "shared memory" in str(e.value)
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())


@pytest.mark.parametrize("name", ["tiny", "ragged", "layer256", "canvas2048"])
def test_layer_from_host_buffers_equals_the_device_call(lib, name):
    """w4_moe_layer_host (x, ids, weights and out in page-locked host memory,
    copied on the stream) gives out bit-identical to w4_moe_layer on the same
    inputs, also with two calls in flight on two streams with their own
    workspaces; M = 0 does nothing."""
    import torch
    cfg, x, lg, _, _ = gpu_inputs(name)
    gu, dn = gpu_weights(name)
    ids, w = lib.w4_moe_route(lg, cfg.k)
    ref = lib.w4_moe_layer(x, ids, w, gu, dn)
    x_h, ids_h, w_h = (t.cpu().pin_memory() for t in (x, ids, w))
    need = lib.w4_moe_layer_host_workspace_size(cfg.M, cfg.d, cfg.m, cfg.E, cfg.k)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.empty((cfg.M, cfg.d), dtype=torch.bfloat16).pin_memory() for _ in streams]
    wss = [torch.full((need,), 255, dtype=torch.uint8, device="cuda") for _ in streams]
    torch.cuda.synchronize()
    for _ in range(2):
        for s, o, ws in zip(streams, outs, wss):
            lib.w4_moe_layer_host(x_h, ids_h, w_h, gu, dn, o, ws, stream=s)
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o.view(torch.int16), ref.cpu().view(torch.int16))
    empty = torch.zeros((0, cfg.d), dtype=torch.bfloat16).pin_memory()
    lib.w4_moe_layer_host(empty, torch.zeros((0, cfg.k), dtype=torch.int32).pin_memory(),
                          torch.zeros((0, cfg.k), dtype=torch.float32).pin_memory(), gu, dn,
                          empty, wss[0])
    torch.cuda.synchronize()
