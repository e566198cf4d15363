"""Pins for the oracle's RMSNorm, entropy and Gumbel-max sampler, each against
something other than the oracle itself: a library routine, a closed form, a
distributional law or an invariant ("dg-w4-kernels" -- RMSNorm, Sampler;
Philox4x32-10 as published by Salmon et al., SC 2011)."""
import math
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import oracle


def _bf16_bits(a):
    """Round-to-nearest-even fp32 -> bf16 bit patterns (numpy)."""
    u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _bf16_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------- Philox
_TRITON_PHILOX = textwrap.dedent("""
    import os, sys, json
    os.environ["TRITON_INTERPRET"] = "1"
    import numpy as np, torch, triton, triton.language as tl

    @triton.jit
    def k(c_ptr, out, seed, N: tl.constexpr):
        i = tl.arange(0, N)
        c0 = tl.load(c_ptr + 4 * i).to(tl.uint32)
        c1 = tl.load(c_ptr + 4 * i + 1).to(tl.uint32)
        c2 = tl.load(c_ptr + 4 * i + 2).to(tl.uint32)
        c3 = tl.load(c_ptr + 4 * i + 3).to(tl.uint32)
        a, b, c, d = tl.philox(seed, c0, c1, c2, c3, 10)
        tl.store(out + 4 * i, a)
        tl.store(out + 4 * i + 1, b)
        tl.store(out + 4 * i + 2, c)
        tl.store(out + 4 * i + 3, d)

    spec = json.loads(sys.argv[1])
    ctr = torch.tensor(np.array(spec["ctr"], np.uint32).view(np.int32).reshape(-1))
    out = torch.zeros_like(ctr)
    k[(1,)](ctr, out, spec["seed"], N=len(spec["ctr"]))
    print(json.dumps((out.numpy().view(np.uint32)).tolist()))
""")


def test_philox_matches_triton_interpreter():
    """Triton's own Philox4x32-10 (its language library, run by the CPU
    interpreter) on random counters under several keys."""
    pytest.importorskip("triton")
    import json
    rng = np.random.default_rng(5)
    for seed in (0, 1, 0xDEADBEEF, 0x0123456789ABCDEF, 2**64 - 1):
        ctr = rng.integers(0, 2**32, (16, 4), dtype=np.uint64)
        ctr[0] = 0
        ctr[1] = 0xFFFFFFFF
        spec = json.dumps({"ctr": ctr.tolist(), "seed": int(seed) - (2**64 if seed >= 2**63 else 0)})
        env = dict(os.environ, TRITON_INTERPRET="1")
        r = subprocess.run([sys.executable, "-c", _TRITON_PHILOX, spec], capture_output=True,
                           text=True, env=env, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        got = np.array(json.loads(r.stdout.strip().splitlines()[-1]), np.uint64).reshape(-1, 4)
        key = [seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF]
        for row, want in zip(ctr, got):
            assert oracle.philox4x32_10(row, key).tolist() == want.tolist(), (seed, row)


def test_noise_word_counter_layout():
    """Row t, column i reads word i % 4 of counter (i // 4, t, offset lo, hi)."""
    seed, off = 0x1234_5678_9ABC_DEF0, 0x0000_0003_0000_0007
    for t, i in [(0, 0), (0, 3), (5, 4), (255, 262143), (7, 1001)]:
        words = oracle.philox4x32_10([i // 4, t, off & 0xFFFFFFFF, off >> 32],
                                     [seed & 0xFFFFFFFF, seed >> 32])
        assert oracle.noise_word(seed, off, t, i) == int(words[i % 4])


# --------------------------------------------------------------------- Gumbel
def test_gumbel_of_word_follows_the_gumbel_law():
    """Over 200k words the variates pass a KS test against the standard
    Gumbel CDF exp(-exp(-x)), with mean Euler's gamma and variance pi^2/6;
    the map is strictly decreasing in the word and bounded."""
    stats = pytest.importorskip("scipy.stats")
    rng = np.random.default_rng(11)
    words = rng.integers(0, 2**32, 200_000, dtype=np.uint64)
    g = np.array([oracle.gumbel_of_word(int(w)) for w in words])
    assert stats.kstest(g, "gumbel_r").pvalue > 1e-3
    assert abs(g.mean() - 0.5772156649) < 0.01
    assert abs(g.var() - math.pi ** 2 / 6) < 0.03
    lo, hi = oracle.gumbel_of_word(2**32 - 1), oracle.gumbel_of_word(0)
    assert -3.2 < lo < hi < 22.9
    assert oracle.gumbel_of_word(1000) > oracle.gumbel_of_word(1001)


def test_sampler_frequencies_follow_softmax():
    """20000 rows of the same five logits: the sample frequencies agree with
    softmax(logits) by a chi-square test (the Gumbel-max identity)."""
    stats = pytest.importorskip("scipy.stats")
    logits = np.array([0.0, 1.0, -0.5, 2.0, 0.3], np.float32)
    M = 20000
    r = oracle.gumbel_argmax(np.tile(logits, (M, 1)), seed=2024, offset=1)
    counts = np.bincount(r["sample"], minlength=5)
    p = np.exp(logits.astype(np.float64) - logits.max())
    p /= p.sum()
    assert stats.chisquare(counts, p * M).pvalue > 1e-4
    assert np.all(r["argmax"] == 3)


def test_sampler_offsets_give_independent_draws():
    """Different offsets (steps) give different noise; the same seed and
    offset give the same draw."""
    logits = np.zeros((64, 1000), np.float32)
    a = oracle.gumbel_argmax(logits, 3, 0)["sample"]
    b = oracle.gumbel_argmax(logits, 3, 1)["sample"]
    c = oracle.gumbel_argmax(logits, 3, 0)["sample"]
    assert np.array_equal(a, c)
    assert np.mean(a == b) < 0.05


def test_sampler_dominant_logit_always_wins():
    """g lies in (-3.2, 22.9): a logit ahead of all others by more than 26.1
    is the sample whatever the noise."""
    rng = np.random.default_rng(3)
    l = rng.standard_normal((50, 3000)).astype(np.float32)
    pos = rng.integers(0, 3000, 50)
    l[np.arange(50), pos] = l.max(axis=1) + 26.2
    r = oracle.gumbel_argmax(l, 99, 5)
    assert np.array_equal(r["sample"], pos)
    assert np.array_equal(r["argmax"], pos)


def test_argmax_matches_numpy_with_ties():
    rng = np.random.default_rng(8)
    l = rng.integers(-3, 4, (40, 257)).astype(np.float32)   # many ties
    l[0, :] = -np.inf
    l[0, 100] = 1.0
    r = oracle.gumbel_argmax(l, 1, 0)
    assert np.array_equal(r["argmax"], np.argmax(l, axis=1))


def test_sampler_best_scores_are_the_perturbed_maxima():
    """best and second are the two largest logit + g of the row."""
    rng = np.random.default_rng(4)
    l = rng.standard_normal((3, 50)).astype(np.float32)
    seed, off = 77, 9
    r = oracle.gumbel_argmax(l, seed, off)
    for t in range(3):
        s = np.array([float(l[t, i]) + oracle.gumbel_of_word(oracle.noise_word(seed, off, t, i))
                      for i in range(50)])
        order = np.argsort(-s, kind="stable")
        assert r["sample"][t] == order[0]
        assert r["best"][t] == s[order[0]] and r["second"][t] == s[order[1]]


# -------------------------------------------------------------------- entropy
def test_entropy_matches_torch_categorical():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(2)
    l = (rng.standard_normal((6, 5000)) * np.array([[0.1], [1], [3], [10], [30], [100]]))
    l = l.astype(np.float32)
    ref = torch.distributions.Categorical(logits=torch.from_numpy(l).double()).entropy().numpy()
    assert np.allclose(oracle.entropy(l), ref, rtol=1e-12, atol=1e-12)


def test_entropy_closed_forms():
    V = 262144
    l = np.zeros((1, V), np.float32)
    assert abs(oracle.entropy(l)[0] - math.log(V)) < 1e-9
    l = np.full((1, 1000), -np.inf, np.float32)
    l[0, 17] = 3.0
    assert oracle.entropy(l)[0] == 0.0
    l = np.full((1, 7), -np.inf, np.float32)
    l[0, 2], l[0, 5] = 0.0, np.float32(math.log(3.0))
    q = np.exp(np.float64(np.float32(math.log(3.0))))
    p = np.array([1.0, q]) / (1.0 + q)
    assert abs(oracle.entropy(l)[0] + np.sum(p * np.log(p))) < 1e-12
    rng = np.random.default_rng(6)
    l = rng.standard_normal((3, 999)).astype(np.float32)
    assert np.allclose(oracle.entropy(l), oracle.entropy(l + np.float32(64.0)), atol=1e-5)


def test_entropy_and_sampler_thread_invariant():
    rng = np.random.default_rng(9)
    l = rng.standard_normal((13, 777)).astype(np.float32)
    assert np.array_equal(oracle.entropy(l, nthreads=1), oracle.entropy(l, nthreads=5))
    a = oracle.gumbel_argmax(l, 5, 6, nthreads=1)
    b = oracle.gumbel_argmax(l, 5, 6, nthreads=4)
    for key in a:
        assert np.array_equal(a[key], b[key])


# -------------------------------------------------------------------- RMSNorm
def test_rmsnorm_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(12)
    x = _bf16_bits(rng.standard_normal((9, 2816)) * 3)
    w = _bf16_bits(1.0 + 0.1 * rng.standard_normal(2816))
    xt = torch.from_numpy(_bf16_to_f64(x))
    wt = torch.from_numpy(_bf16_to_f64(w))
    ref = torch.nn.functional.rms_norm(xt, (2816,), wt, 1e-6).numpy()
    assert np.allclose(oracle.rmsnorm(x, w, 1e-6), ref, rtol=1e-13, atol=1e-14)


def test_rmsnorm_closed_forms():
    d = 64
    w = _bf16_bits(np.linspace(0.5, 2.0, d))
    wv = _bf16_to_f64(w)
    x = np.full((1, d), _bf16_bits(np.float32(1.5)), np.uint16)
    y = oracle.rmsnorm(x, w, 0.25)[0]
    assert np.allclose(y, 1.5 / math.sqrt(1.5 ** 2 + 0.25) * wv, rtol=1e-15)
    z = np.zeros((1, d), np.uint16)
    assert np.all(oracle.rmsnorm(z, w, 1e-6) == 0.0)
    rng = np.random.default_rng(13)
    x = _bf16_bits(rng.standard_normal((4, d)))
    ones = np.full(d, 0x3F80, np.uint16)
    y = oracle.rmsnorm(x, ones, 0.0)
    assert np.allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-14)
    x2 = _bf16_bits(_bf16_to_f64(x) * 8.0)       # exact in bf16
    assert np.allclose(oracle.rmsnorm(x2, ones, 0.0), y, rtol=1e-14)
