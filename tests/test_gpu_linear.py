"""The dense W4A16 linear on the GPU against the oracle ("dg-w4-kernels" --
W4A16: w4a16_linear equals F.linear(x, dequant(W))).

The weights are quantised by the oracle on the CPU (the inputs of both sides);
the GPU result is compared element by element with the float64 oracle:

* |y - oracle| <= 2^-8 |oracle| + 1e-2 rms(oracle): the bf16 rounding of the
  output (at most 2^-8 relative) plus the fp16 roundings of the inputs (x to
  fp16, each dequantised weight as q s + fp16(-z s), about 1e-3 of rms(y) on
  average over K terms) with a margin for the largest of ~1M outputs;
* max |y - oracle| / rms(oracle) <= 2e-2, the bar of the layer's outputs;
* two runs bit-identical.
The 256-row shapes are checked on 24 sampled rows (rows are independent).
"""
import numpy as np
import pytest

import oracle
from w4a16_moe_expert_sync_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _cuda(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run(lib, cfg, x, q, s, z):
    import torch
    xt = _cuda(x.view(np.int16)).view(torch.bfloat16)
    qt, st, zt = _cuda(q), _cuda(s.view(np.int16)).view(torch.float16), _cuda(z.view(np.int16)).view(torch.float16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = lib.w4_w4a16_linear(xt, qt, st, zt, cfg.group, dev_status=status)
    y2 = lib.w4_w4a16_linear(xt, qt, st, zt, cfg.group, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    return (y.float().cpu().numpy()).astype(np.float64)


def _check(got, ref):
    rms = np.sqrt(np.mean(ref * ref))
    err = np.abs(got - ref)
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-2 * rms), (err.max() / rms)
    assert err.max() / rms <= 2e-2


@pytest.mark.parametrize("name", list(wl.LINEAR_CONFIGS))
def test_linear_matches_oracle(lib, name):
    cfg = wl.LINEAR_CONFIGS[name]
    x, W = wl.linear_inputs(cfg)
    q, s, z = oracle.quantize_w4(W, cfg.group)
    got = _run(lib, cfg, x, q, s, z)
    rows = np.arange(cfg.M) if cfg.M <= 40 else np.linspace(0, cfg.M - 1, 24).round().astype(int)
    ref = oracle.w4a16_linear(x[rows], q, s, z, cfg.group)
    _check(got[rows], ref)


@pytest.mark.parametrize("M", [1, 32, 33, 64])
def test_linear_row_counts_around_a_job(lib, M):
    """32 tokens per job: one job, exactly full, one past, two jobs."""
    cfg = wl.LinearShape("m", M, 512, 256, seed=60 + M)
    x, W = wl.linear_inputs(cfg)
    q, s, z = oracle.quantize_w4(W, 128)
    _check(_run(lib, cfg, x, q, s, z), oracle.w4a16_linear(x, q, s, z, 128))


def test_linear_group64_and_empty(lib):
    import torch
    cfg = wl.LinearShape("g64", 9, 704, 256, seed=70, group=64)
    x, W = wl.linear_inputs(cfg)
    q, s, z = oracle.quantize_w4(W, 64)
    _check(_run(lib, cfg, x, q, s, z), oracle.w4a16_linear(x, q, s, z, 64))
    empty = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    qt = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    st = torch.zeros((128, 2), dtype=torch.float16, device="cuda")
    y = lib.w4_w4a16_linear(empty, qt, st, st, 128)
    assert y.shape == (0, 128)


def test_linear_rejects_unsupported_shapes(lib):
    import torch
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((100, 128), dtype=torch.uint8, device="cuda")     # N % 128 != 0
    s = torch.zeros((100, 2), dtype=torch.float16, device="cuda")
    with pytest.raises(lib.W4Error):
        lib.w4_w4a16_linear(x, q, s, s, 128)


def test_linear_rejects_more_than_32_groups(lib):
    """The per-row scales and zeros of a panel are staged whole: at most 32
    groups along the contraction dim."""
    import torch
    x = torch.zeros((4, 4352), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((128, 2176), dtype=torch.uint8, device="cuda")
    s = torch.zeros((128, 34), dtype=torch.float16, device="cuda")
    with pytest.raises(lib.W4Error):
        lib.w4_w4a16_linear(x, q, s, s, 128)


@pytest.mark.parametrize("M", [300, 600])
def test_linear_several_token_tiles(lib, M):
    """More than 256 rows: token tiles of 256, the last one partial (its
    token-tile loads read zero rows past the padded end), every row checked."""
    cfg = wl.LinearShape("tiles", M, 512, 256, seed=80 + M)
    x, W = wl.linear_inputs(cfg)
    q, s, z = oracle.quantize_w4(W, 128)
    _check(_run(lib, cfg, x, q, s, z), oracle.w4a16_linear(x, q, s, z, 128))
