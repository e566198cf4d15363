"""quantize_w4 on the GPU is bit-exact against the oracle
("diffusiongemma-26B-A4B-w4a16" -- Checkpoint format)."""
import numpy as np
import pytest

import oracle
from w4a16_moe_expert_sync_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _gpu_quant(lib, W, group):
    import torch
    q, s, z = lib.w4_quantize(torch.from_numpy(np.ascontiguousarray(W)).cuda(), group)
    torch.cuda.synchronize()
    return (q.cpu().numpy(), s.cpu().view(torch.int16).numpy().view(np.uint16),
            z.cpu().view(torch.int16).numpy().view(np.uint16))


def _assert_same(got, ref):
    for a, b in zip(got, ref):
        assert a.shape == b.reshape(a.shape).shape
        assert np.array_equal(a, b.reshape(a.shape))


@pytest.mark.parametrize("group", [64, 128, 256])
@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_quantize_bit_exact_workload_weights(lib, name, group):
    cfg = wl.CONFIGS[name]
    W = wl.all_gate_up_weights(cfg)
    if cfg.d % group:
        pytest.skip("group does not divide the contraction dim")
    _assert_same(_gpu_quant(lib, W, group), oracle.quantize_w4(W, group))
    Wd = wl.all_down_weights(cfg)
    if cfg.m % group == 0:
        _assert_same(_gpu_quant(lib, Wd, group), oracle.quantize_w4(Wd, group))


def test_quantize_bit_exact_full_size_experts(lib):
    cfg = wl.CONFIGS["layer256"]
    for e in (0, 77):
        Wg = wl.gate_up_weight(cfg, e)[None]
        _assert_same(_gpu_quant(lib, Wg, 128), oracle.quantize_w4(Wg, 128))
        Wd = wl.down_weight(cfg, e)[None]
        _assert_same(_gpu_quant(lib, Wd, 64), oracle.quantize_w4(Wd, 64))


def test_quantize_edge_groups(lib):
    rng = np.random.default_rng(9)
    rows = []
    rows.append(np.zeros(128))                          # all zero
    rows.append(np.full(128, 0.375))                     # constant
    rows.append(np.full(128, -3.1e-3))                   # constant, not fp16-exact
    rows.append(rng.standard_normal(128) * 1e-6)         # subnormal fp16 scale
    rows.append(rng.standard_normal(128) * 1e3)          # large values
    rows.append(np.abs(rng.standard_normal(128)) + 5.0)  # all positive: z < 0
    rows.append(-np.abs(rng.standard_normal(128)) - 5.0)  # all negative: z > 15
    r = rng.standard_normal(128)
    r[::2] = 0.0
    r[1::4] = -0.0
    rows.append(r)                                       # signed zeros
    # exact halfway points between codes
    rows.append(np.concatenate([np.arange(16, dtype=np.float64), np.arange(112) % 16 + 0.5]))
    W = np.stack(rows).astype(np.float32)[None]
    _assert_same(_gpu_quant(lib, W, 128), oracle.quantize_w4(W, 128))
    _assert_same(_gpu_quant(lib, W, 64), oracle.quantize_w4(W, 64))
