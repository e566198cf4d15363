"""The fixed-order combine folded into the down GEMM
(w4_grouped_gemm_down_combine after w4_moe_combine_prepare, and the layer's
own folded path) against the standalone down GEMM followed by
w4_moe_combine_fixed_order: bit-identical outputs, invalid ids included
("Inference: Making every denoising pass fast" -- Quantisation alone leaves a
sparse execution problem: a token's expert outputs are reduced in a fixed
order, so that reruns agree to the bit)."""
import numpy as np
import pytest

import oracle
from helpers import gpu_inputs, gpu_weights

pytestmark = pytest.mark.gpu

GARBAGE = 0x7F7F   # a finite bf16 bit pattern that no result here produces


def _ids_with_invalid(name):
    """The config's routing with token 5 fully invalid and one invalid id in
    token 7 (when the batch has them)."""
    cfg, x, lg, _, logits = gpu_inputs(name)
    ids, w = oracle.route(logits, cfg.k)
    ids = ids.copy()
    if cfg.M > 7:
        ids[5, :] = -1
        ids[7, cfg.k // 2] = cfg.E       # out of range
    return cfg, x, ids, w


def _reference(lib, cfg, x, ids_d, w_d, gu, dn):
    al, xg = lib.w4_moe_align_gather(ids_d, x, cfg.E, 16)
    h = lib.w4_grouped_gemm_gate_up(xg, *gu, al)
    y = lib.w4_grouped_gemm_down(h, *dn, al)
    return al, h, y, lib.w4_moe_combine_fixed_order(y, ids_d, w_d, cfg.E)


@pytest.mark.parametrize("name", ["tiny", "ragged", "bigjobs", "layer256", "zipf256", "canvas2048"])
def test_down_combine_equals_down_then_combine(lib, name):
    import torch
    cfg, x, ids, w = _ids_with_invalid(name)
    gu, dn = gpu_weights(name)
    ids_d, w_d = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    al, h, y_ref, ref = _reference(lib, cfg, x, ids_d, w_d, gu, dn)
    counters = torch.full((cfg.M, cfg.d // 128), -12345, dtype=torch.int32, device="cuda")
    out = torch.full((cfg.M, cfg.d), GARBAGE, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    lib.w4_moe_combine_prepare(ids_d, cfg.E, cfg.d, counters=counters, out=out)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y, out = lib.w4_grouped_gemm_down_combine(h, *dn, al, ids_d, w_d, counters, out,
                                              dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    # every valid assignment's y row as the standalone down GEMM's
    flat = ids.reshape(-1)
    valid = torch.from_numpy((flat >= 0) & (flat < cfg.E)).cuda()
    assert torch.equal(y[valid].view(torch.int32), y_ref[valid].view(torch.int32))
    # every counter ran to k: each valid assignment arrived once per panel
    assert bool((counters == cfg.k).all())
    if cfg.M > 7:
        assert torch.count_nonzero(out[5].view(torch.int16)) == 0


def test_down_combine_reruns_are_bit_identical(lib):
    import torch
    name = "layer256"
    cfg, x, ids, w = _ids_with_invalid(name)
    gu, dn = gpu_weights(name)
    ids_d, w_d = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    al, h, _, _ = _reference(lib, cfg, x, ids_d, w_d, gu, dn)
    outs = []
    for _ in range(3):
        counters, out = lib.w4_moe_combine_prepare(ids_d, cfg.E, cfg.d)
        _, out = lib.w4_grouped_gemm_down_combine(h, *dn, al, ids_d, w_d, counters, out)
        outs.append(out.clone())
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "layer256"])
def test_layer_fold_from_a_dirty_output(lib, name):
    """The layer writes every element of out, the zero rows of tokens with
    no valid expert included, whatever out held before; the result is the
    separate calls' bit for bit."""
    import torch
    cfg, x, ids, w = _ids_with_invalid(name)
    gu, dn = gpu_weights(name)
    ids_d, w_d = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    _, _, _, ref = _reference(lib, cfg, x, ids_d, w_d, gu, dn)
    ws = torch.full((lib.w4_moe_layer_workspace_size(cfg.M, cfg.d, cfg.m, cfg.E, cfg.k),),
                    255, dtype=torch.uint8, device="cuda")
    for _ in range(2):      # the second call finds the first one's counters
        out = torch.full((cfg.M, cfg.d), GARBAGE, dtype=torch.int16,
                         device="cuda").view(torch.bfloat16)
        lib.w4_moe_layer(x, ids_d, w_d, gu, dn, workspace=ws, out=out)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
