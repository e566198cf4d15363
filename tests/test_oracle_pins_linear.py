"""Pins for the oracle's dense W4A16 linear, y = x . deq(W)^T ("dg-w4-kernels" --
W4A16: w4a16_linear equals F.linear(x, dequant(W))), each against something
other than the oracle's own code path."""
import numpy as np
import pytest

import oracle
from w4a16_moe_expert_sync_gb300 import workloads as wl


def _weights(N, K, seed, group=128):
    W = (np.random.default_rng(seed).standard_normal((N, K)) * 0.02).astype(np.float32)
    q, s, z = oracle.quantize_w4(W, group)
    return W, q, s, z


def test_linear_brute_force_with_an_independent_decoder():
    """Tiny case by plain Python loops: nibbles unpacked with Python ints,
    fp16 scale/zero and bf16 activations decoded by numpy's own types."""
    N, K, M, g = 3, 256, 2, 128
    _, q, s, z = _weights(N, K, 1, g)
    x = wl.f32_to_bf16_bits(np.random.default_rng(2).standard_normal((M, K)))
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    sf = s.view(np.float16).astype(np.float64)
    zf = z.view(np.float16).astype(np.float64)
    want = np.zeros((M, N))
    for t in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                byte = int(q[n, k // 2])
                code = (byte >> 4) if k % 2 else (byte & 15)
                acc += sf[n, k // g] * (code - zf[n, k // g]) * xf[t, k]
            want[t, n] = acc
    got = oracle.w4a16_linear(x, q, s, z, g, nthreads=1)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-15)


def test_linear_one_hot_rows_recover_the_dequantised_columns():
    N, K = 48, 384
    _, q, s, z = _weights(N, K, 3)
    cols = [0, 1, 127, 128, 255, 383]
    x = np.zeros((len(cols), K), np.uint16)
    for i, c in enumerate(cols):
        x[i, c] = 0x3F80                        # bf16 1.0
    y = oracle.w4a16_linear(x, q, s, z, 128)
    deq = oracle.dequant_w4(q, s, z, 128)
    for i, c in enumerate(cols):
        assert np.array_equal(y[i], deq[:, c])


def test_linear_is_within_the_quantiser_bound_of_the_unquantised_product():
    """|x . deq(W)^T - x . W^T| <= sum_k |x_k| s_k / 2 (1 + 2^-10): each
    weight is reconstructed to half a step (fp16 slack on s and z)."""
    torch = pytest.importorskip("torch")
    N, K, M = 64, 512, 7
    W, q, s, z = _weights(N, K, 4)
    x = wl.f32_to_bf16_bits(np.random.default_rng(5).standard_normal((M, K)))
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    y = oracle.w4a16_linear(x, q, s, z, 128)
    ref = torch.nn.functional.linear(torch.from_numpy(xf), torch.from_numpy(W.astype(np.float64)))
    step = np.repeat(s.view(np.float16).astype(np.float64), 128, axis=1)   # [N, K]
    bound = (np.abs(xf) @ step.T) / 2 * (1 + 2.0 ** -10) + 1e-12
    assert np.all(np.abs(y - ref.numpy()) <= bound)


def test_linear_thread_count_invariant():
    _, q, s, z = _weights(40, 256, 6)
    x = wl.f32_to_bf16_bits(np.random.default_rng(7).standard_normal((9, 256)))
    assert np.array_equal(oracle.w4a16_linear(x, q, s, z, 128, nthreads=1),
                          oracle.w4a16_linear(x, q, s, z, 128, nthreads=4))
