"""Router and alignment on the GPU against the oracle: expert ids, sorted
slots, offsets, block owners and the router weights are bit-exact
("Inference: Making every denoising pass fast" -- Quantisation alone
leaves a sparse execution problem; "dg-w4-kernels" -- Grouped MoE)."""
import numpy as np
import pytest

import oracle
from w4a16_moe_expert_sync_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _cuda(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("name", ["tiny", "ragged", "layer256", "zipf256", "canvas2048",
                                  "sweep_M1"])
def test_route_matches_oracle(lib, name):
    cfg = wl.CONFIGS[name]
    logits = wl.router_logits(cfg)
    ids, w = lib.w4_moe_route(_cuda(logits), cfg.k)
    oids, ow = oracle.route(logits, cfg.k)
    assert np.array_equal(ids.cpu().numpy(), oids)
    # float64 on both sides, one rounding to fp32: the same bits
    assert np.array_equal(w.cpu().numpy().view(np.uint32), ow.view(np.uint32))


def test_route_ties_go_to_lower_index(lib):
    logits = np.zeros((3, 64), np.float32)
    logits[0, [40, 3, 17]] = 2.0
    logits[1, :] = 1.0
    logits[2, 63] = 5.0
    ids, w = lib.w4_moe_route(_cuda(logits), 3)
    oids, ow = oracle.route(logits, 3)
    assert np.array_equal(ids.cpu().numpy(), oids)
    assert ids.cpu().numpy()[0].tolist() == [3, 17, 40]


def _check_align(lib, ids, E, bm):
    import torch
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = lib.w4_moe_align(_cuda(ids.astype(np.int32)), E, bm, dev_status=status)
    ref = oracle.moe_align(ids.astype(np.int32), E, bm)
    torch.cuda.synchronize()
    assert np.array_equal(r["sorted_ids"].cpu().numpy(), ref["sorted_ids"])
    assert np.array_equal(r["block_expert"].cpu().numpy(), ref["block_expert"])
    assert np.array_equal(r["expert_offsets"].cpu().numpy(), ref["expert_offsets"])
    assert int(r["num_padded"].item()) == ref["num_padded"]
    bad_bit = int(status.item()) & lib.W4_DEV_BAD_EXPERT_ID
    assert bool(bad_bit) == (ref["bad"] > 0)


@pytest.mark.parametrize("bm", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("name", ["tiny", "layer256", "zipf256", "canvas2048"])
def test_align_matches_oracle(lib, name, bm):
    cfg = wl.CONFIGS[name]
    ids, _ = oracle.route(wl.router_logits(cfg), cfg.k)
    _check_align(lib, ids, cfg.E, bm)


@pytest.mark.parametrize("case", ["m1", "one_expert", "empty_experts", "bad_ids", "k1_big",
                                  "e1024", "m0"])
def test_align_edge_cases(lib, case):
    rng = np.random.default_rng(31)
    E = 128
    if case == "m1":
        ids = rng.permutation(E)[:8][None]
    elif case == "one_expert":
        ids = np.full((300, 1), 5)
    elif case == "empty_experts":
        ids = (rng.integers(0, 4, (500, 2)) * 31)
    elif case == "bad_ids":
        ids = rng.integers(-3, E + 3, (100, 8))
    elif case == "k1_big":
        ids = rng.integers(0, E, (20000, 1))
    elif case == "e1024":
        E = 1024
        ids = np.stack([rng.permutation(E)[:8] for _ in range(700)])
    else:
        ids = np.zeros((0, 8))
    _check_align(lib, ids, E, 16)
    _check_align(lib, ids, E, 64)


@pytest.mark.parametrize("name", ["tiny", "ragged", "sweep_M1", "sweep_M8", "sweep_M64",
                                  "layer256", "zipf256", "canvas2048"])
@pytest.mark.parametrize("bm", [16, 64])
def test_route_align_gather_matches_the_separate_calls(lib, name, bm):
    """Router + alignment + gather from the logits (one launch up to 16
    tokens: tiny, sweep_M1; the router launch then the alignment launch
    above that): ids and weights
    bit-identical to w4_moe_route (and ids to the oracle), alignment outputs
    and gathered rows bit-identical to w4_moe_align_gather."""
    import torch
    cfg = wl.CONFIGS[name]
    logits = wl.router_logits(cfg)
    x = _cuda(wl.activations(cfg).view(np.int16)).view(torch.bfloat16)
    lg = _cuda(logits)
    ids, w, al, xg = lib.w4_moe_route_align_gather(lg, x, cfg.k, bm)
    rids, rw = lib.w4_moe_route(lg, cfg.k)
    ral, rxg = lib.w4_moe_align_gather(rids, x, cfg.E, bm)
    torch.cuda.synchronize()
    assert torch.equal(ids, rids)
    assert torch.equal(w.view(torch.int32), rw.view(torch.int32))
    oids, _ = oracle.route(logits, cfg.k)
    assert np.array_equal(ids.cpu().numpy(), oids)
    for key in ("sorted_ids", "block_expert", "expert_offsets", "num_padded"):
        assert torch.equal(al[key], ral[key])
    npad = int(ral["num_padded"].item())
    # rows of padding slots are not written by either fused launch
    real = ral["sorted_ids"][:npad] < cfg.A
    used = cfg.d + 16 * ((cfg.d // 128 + 15) // 16)     # the rest of the sum block is not written
    assert torch.equal(xg[:npad, :used][real].view(torch.int16),
                       rxg[:npad, :used][real].view(torch.int16))


@pytest.mark.parametrize("name", ["ragged", "layer256"])
def test_layer_from_logits_equals_route_then_layer(lib, name):
    import torch
    from helpers import gpu_inputs, gpu_weights
    cfg, x, lg, _, _ = gpu_inputs(name)
    gu, dn = gpu_weights(name)
    out, ids, w = lib.w4_moe_layer_from_logits(x, lg, cfg.k, gu, dn)
    rids, rw = lib.w4_moe_route(lg, cfg.k)
    ref = lib.w4_moe_layer(x, rids, rw, gu, dn)
    torch.cuda.synchronize()
    assert torch.equal(ids, rids)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
