"""Pins for the float64 CPU oracle (no GPU).

The oracle is checked against things other than itself: IEEE-754 conversions
from numpy, the packing rule worked by hand, the storage sizes printed on the
pages, closed-form bounds of round-to-nearest quantisation, brute-force
nearest-code search, brute-force stable sorting, scipy's softmax, torch's
tanh-GELU and F.linear, and an independent dense numpy evaluation of the
whole layer.  Each test names the passage it pins (page title -- section).
"""
import os

import numpy as np
import pytest

import oracle
from w4a16_moe_expert_sync_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# number formats (IEEE-754 binary16 / bfloat16)
# ---------------------------------------------------------------------------
def test_f16_decode_matches_numpy_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.f16_bits_to_f64_array(bits)
    finite = ~np.isnan(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.all(np.isnan(got[~finite]))


def test_f32_to_f16_round_to_nearest_even_matches_numpy():
    rng = np.random.default_rng(123)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-5).astype(np.float32),      # subnormal range
        (rng.standard_normal(2000) * 3e4).astype(np.float32),       # near overflow
        np.float32([0.0, -0.0, 65504.0, 65519.0, 65520.0, -65520.0, 1e-8, 6e-8, 2.0**-25,
                    3 * 2.0**-26, 1 + 2.0**-11, 1 + 3 * 2.0**-11, 2048 + 1, 2048 + 3]),
    ])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    for v, r in zip(vals, ref):
        assert oracle.f32_to_f16(v) == int(r), v


def test_bf16_decode_is_top_half_of_binary32():
    for v in [1.0, -2.5, 3.140625, 1e-3, -7.0e20]:
        bits = int(np.float32(v).view(np.uint32) >> 16)
        assert oracle.bf16_to_f64(bits) == float(np.uint32(bits << 16).view(np.float32))


# ---------------------------------------------------------------------------
# "diffusiongemma-26B-A4B-w4a16" -- Checkpoint format: packing
# ---------------------------------------------------------------------------
def _golden_pack_cases():
    cases = []
    with open(os.path.join(GOLDEN, "pack_nibbles.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            codes, packed = line.split(";")
            cases.append((np.array([int(c) for c in codes.split()], np.uint8),
                          np.array([int(b, 16) for b in packed.split()], np.uint8)))
    return cases


@pytest.mark.parametrize("codes,packed", _golden_pack_cases())
def test_pack_matches_hand_worked_examples(codes, packed):
    assert np.array_equal(oracle.pack_codes(codes), packed)
    assert np.array_equal(oracle.unpack_codes(packed), codes)


def test_pack_round_trip_exact():
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 16, size=(33, 64), dtype=np.uint8)
    assert np.array_equal(oracle.unpack_codes(oracle.pack_codes(codes)), codes)


# ---------------------------------------------------------------------------
# quantize_w4: asymmetric uint4, fp16 scale and zero per group, min/max RTN
# ("diffusiongemma-26B-A4B-w4a16" -- Checkpoint format, Benchmarks;
#  "Inference: Making every denoising pass fast" -- The first constraint was
#  capacity)
# ---------------------------------------------------------------------------
def _np_dequant(q, s, z, group):
    """Independent numpy restatement used only to check the oracle's bound."""
    codes = np.stack([q & 0xF, q >> 4], axis=-1).reshape(q.shape[:-1] + (q.shape[-1] * 2,))
    sf = s.view(np.float16).astype(np.float64).repeat(group, axis=-1)
    zf = z.view(np.float16).astype(np.float64).repeat(group, axis=-1)
    return codes.astype(np.float64), sf, zf


@pytest.mark.parametrize("group", [64, 128])
def test_quantizer_error_at_most_half_a_step(group):
    rng = np.random.default_rng(group)
    W = (rng.standard_normal((24, 512)) * 0.02).astype(np.float32)
    q, s, z = oracle.quantize_w4(W, group)
    codes, sf, zf = _np_dequant(q, s, z, group)
    w_hat = oracle.dequant_w4(q, s, z, group)
    err = np.abs(w_hat - W.astype(np.float64))
    # round to nearest: |w - s(q - z)| <= s/2, up to the fp32 evaluation of
    # w/s + z (a few ulps of a value below 16)
    assert np.all(err <= sf * (0.5 + 2.0**-18)), err.max()
    assert np.allclose(w_hat, sf * (codes - zf), rtol=0, atol=0)


@pytest.mark.parametrize("group", [64, 128])
def test_quantizer_picks_the_nearest_code_by_brute_force(group):
    rng = np.random.default_rng(100 + group)
    W = (rng.standard_normal((8, 256)) * 0.02).astype(np.float32)
    q, s, z = oracle.quantize_w4(W, group)
    codes, sf, zf = _np_dequant(q, s, z, group)
    grid = sf[..., None] * (np.arange(16)[None, None, :] - zf[..., None])   # every code
    best = np.abs(grid - W.astype(np.float64)[..., None]).min(-1)
    mine = np.abs(sf * (codes - zf) - W)
    assert np.all(mine <= best + sf * 2.0**-18)


def test_quantizer_hits_both_ends_of_the_code_range():
    rng = np.random.default_rng(5)
    W = (rng.standard_normal((16, 1024)) * 0.02).astype(np.float32)
    q, s, z = oracle.quantize_w4(W, 128)
    codes = oracle.unpack_codes(q).reshape(16, 8, 128)
    assert np.all(codes.min(-1) == 0) and np.all(codes.max(-1) == 15)
    # the min maps to 0 and the max to 15
    Wg = W.reshape(16, 8, 128)
    assert np.all(codes[np.arange(16)[:, None], np.arange(8)[None], Wg.argmin(-1)] == 0)
    assert np.all(codes[np.arange(16)[:, None], np.arange(8)[None], Wg.argmax(-1)] == 15)


def test_quantizer_constant_and_zero_groups_reconstruct_exactly():
    W = np.zeros((3, 128), np.float32)
    W[1, :] = 0.375          # representable in fp16
    W[2, :] = -1.5
    q, s, z = oracle.quantize_w4(W, 64)
    assert np.array_equal(oracle.dequant_w4(q, s, z, 64), W.astype(np.float64))
    # a constant group has zero range: the scale falls back to 1
    assert np.all(s.view(np.float16) == 1.0)


def test_quantizer_rejects_bad_group():
    with pytest.raises(ValueError):
        oracle.quantize_w4(np.zeros((2, 100), np.float32), 64)


def test_storage_sizes_match_the_pages():
    """Byte counts of the packed format reproduce the printed expert sizes."""
    d, m, E = 2816, 704, 128
    rng = np.random.default_rng(0)
    gu = oracle.quantize_w4((rng.standard_normal((2 * m, d)) * 0.02).astype(np.float32), 128)
    dn = oracle.quantize_w4((rng.standard_normal((d, m)) * 0.02).astype(np.float32), 64)
    per_expert = sum(a.nbytes for a in gu) + sum(a.nbytes for a in dn)
    assert per_expert == 3_221_504
    GiB = 2.0**30
    printed = {}
    with open(os.path.join(GOLDEN, "storage_sizes.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, val, unit, _ = [p.strip() for p in line.split(";")]
                printed[key] = float(val)
    params_per_layer = E * (2 * m * d + d * m)
    bf16_60 = 60 * params_per_layer * 2 / GiB
    w4_30_shared = 30 * E * per_expert / GiB
    w4_quarter = 60 * params_per_layer * 0.5 / GiB
    assert round(bf16_60, 1) == printed["bf16_experts_60_layers"]
    assert round(w4_30_shared, 1) == printed["w4a16_experts_30_shared_shards"]
    assert round(w4_quarter, 1) == printed["w4a16_experts_quarter_of_bf16"]


# ---------------------------------------------------------------------------
# router: softmax -> top-k -> renormalise
# ("Inference: Making every denoising pass fast" -- Quantisation alone leaves
#  a sparse execution problem)
# ---------------------------------------------------------------------------
def test_router_against_brute_force_and_scipy_softmax():
    from scipy.special import softmax
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((64, 128)).astype(np.float32)
    ids, w = oracle.route(logits, 8)
    order = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :8]
    assert np.array_equal(ids, order)
    for t in range(64):
        p = softmax(logits[t].astype(np.float64))
        ref = p[ids[t]] / p[ids[t]].sum()
        assert np.allclose(w[t], ref, rtol=1e-6, atol=0)
        assert abs(float(w[t].astype(np.float64).sum()) - 1.0) <= 8 * 2.0**-24
        assert len(set(ids[t].tolist())) == 8
        assert np.all(np.diff(w[t]) <= 0)


def test_router_ties_go_to_the_lower_index():
    logits = np.zeros((2, 8), np.float32)
    logits[0, [6, 2, 5]] = 1.0
    logits[1, :] = 0.5
    ids, w = oracle.route(logits, 3)
    assert ids[0].tolist() == [2, 5, 6]
    assert ids[1].tolist() == [0, 1, 2]
    assert np.allclose(w, 1 / 3, rtol=1e-7)


# ---------------------------------------------------------------------------
# alignment: count, padded prefix scan, stable placement
# ("Inference: Making every denoising pass fast" -- Quantisation alone leaves a
#  sparse execution problem; "dg-w4-kernels" -- Grouped MoE)
# ---------------------------------------------------------------------------
def _brute_align(ids, E, bm):
    A = ids.size
    flat = ids.ravel()
    valid = [(int(e), a) for a, e in enumerate(flat) if 0 <= e < E]
    valid.sort(key=lambda p: p[0])              # Python's sort is stable
    by_e = {e: [a for (ee, a) in valid if ee == e] for e in range(E)}
    sorted_ids, offs, owners = [], [0], []
    for e in range(E):
        seg = by_e[e]
        padded = -(-len(seg) // bm) * bm
        sorted_ids += seg + [A] * (padded - len(seg))
        owners += [e] * (padded // bm)
        offs.append(offs[-1] + padded)
    return sorted_ids, offs, owners


@pytest.mark.parametrize("bm", [16, 32, 64, 128])
@pytest.mark.parametrize("case", ["random", "one_expert", "m1", "k1", "empty_experts", "bad_ids"])
def test_align_matches_brute_force_stable_sort(bm, case):
    rng = np.random.default_rng(hash((bm, case)) % 2**32)
    E = 16
    if case == "random":
        ids = np.stack([rng.permutation(E)[:4] for _ in range(37)]).astype(np.int32)
    elif case == "one_expert":
        ids = np.full((20, 1), 3, np.int32)
    elif case == "m1":
        ids = rng.permutation(E)[:8][None].astype(np.int32)
    elif case == "k1":
        ids = rng.integers(0, E, (50, 1)).astype(np.int32)
    elif case == "empty_experts":
        ids = rng.integers(0, 3, (40, 2)).astype(np.int32) * 5      # experts 0, 5, 10 only
    else:
        ids = rng.integers(-2, E + 2, (30, 3)).astype(np.int32)
    r = oracle.moe_align(ids, E, bm)
    ref_sorted, ref_offs, ref_owner = _brute_align(ids, E, bm)
    A = ids.size
    cap = oracle.align_capacity(ids.shape[0], ids.shape[1], E, bm)
    assert cap % bm == 0 and cap >= A + E * (bm - 1)
    n = r["num_padded"]
    assert n == ref_offs[-1]
    assert r["sorted_ids"][:n].tolist() == ref_sorted
    assert np.all(r["sorted_ids"][n:] == A)
    assert r["expert_offsets"].tolist() == ref_offs
    assert np.all(r["expert_offsets"] % bm == 0)
    nb = n // bm
    assert r["block_expert"][:nb].tolist() == ref_owner
    assert np.all(r["block_expert"][nb:] == -1)
    # every valid assignment appears exactly once
    real = r["sorted_ids"][r["sorted_ids"] < A]
    valid = np.flatnonzero((ids.ravel() >= 0) & (ids.ravel() < E))
    assert sorted(real.tolist()) == valid.tolist()
    assert r["bad"] == A - valid.size


# ---------------------------------------------------------------------------
# expert MLP and fixed-order combine
# ---------------------------------------------------------------------------
def test_gelu_tanh_matches_torch_and_special_values():
    import torch
    v = np.linspace(-8, 8, 161)
    ref = torch.nn.functional.gelu(torch.tensor(v, dtype=torch.float64), approximate="tanh").numpy()
    got = np.array([oracle.gelu_tanh(t) for t in v])
    assert np.allclose(got, ref, rtol=1e-14, atol=1e-15)
    assert oracle.gelu_tanh(0.0) == 0.0
    assert abs(oracle.gelu_tanh(30.0) - 30.0) < 1e-12 and abs(oracle.gelu_tanh(-30.0)) < 1e-12


def _quantized_layer(cfg):
    x = wl.activations(cfg)
    gu = oracle.quantize_w4(wl.all_gate_up_weights(cfg), cfg.gu_group)
    dn = oracle.quantize_w4(wl.all_down_weights(cfg), cfg.dn_group)
    ids, w = oracle.route(wl.router_logits(cfg), cfg.k)
    return x, gu, dn, ids, w


def _dense_numpy_layer(cfg, x_bits, gu, dn, ids, w):
    """Every expert on every token, gated by a zero-filled routing vector."""
    x = x_bits.astype(np.uint32) << 16
    x = x.view(np.float32).astype(np.float64)

    def deq(qsz, group):
        codes, sf, zf = _np_dequant(*qsz, group)
        return sf * (codes - zf)

    Wgu = deq(gu, cfg.gu_group)            # [E, 2m, d]
    Wdn = deq(dn, cfg.dn_group)            # [E, d, m]
    gate = np.zeros((cfg.M, cfg.E))
    for t in range(cfg.M):
        for j in range(cfg.k):
            gate[t, ids[t, j]] += float(w[t, j])
    out = np.zeros((cfg.M, cfg.d))
    c = np.sqrt(2.0 / np.pi)
    for e in range(cfg.E):
        g = x @ Wgu[e, :cfg.m].T
        u = x @ Wgu[e, cfg.m:].T
        h = 0.5 * g * (1.0 + np.tanh(c * (g + 0.044715 * g ** 3))) * u
        out += gate[:, e:e + 1] * (h @ Wdn[e].T)
    return out


@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_layer_matches_dense_brute_force(name):
    cfg = wl.CONFIGS[name]
    x, gu, dn, ids, w = _quantized_layer(cfg)
    out = oracle.moe_layer(x, gu, dn, ids, w, cfg.gu_group, cfg.dn_group, nthreads=4)
    ref = _dense_numpy_layer(cfg, x, gu, dn, ids, w)
    scale = np.sqrt(np.mean(ref ** 2))
    assert np.max(np.abs(out - ref)) <= 1e-12 * scale


def test_dense_check_has_teeth():
    """Plausible mistakes in the layer (gate/up swapped, transposed down,
    weights applied to the wrong slot) move the result far outside 1e-12."""
    cfg = wl.CONFIGS["tiny"]
    x, gu, dn, ids, w = _quantized_layer(cfg)
    out = oracle.moe_layer(x, gu, dn, ids, w, cfg.gu_group, cfg.dn_group, nthreads=2)
    scale = np.sqrt(np.mean(out ** 2))
    m = cfg.m
    swapped = tuple(np.concatenate([a[:, m:], a[:, :m]], axis=1) for a in gu)
    assert np.max(np.abs(oracle.moe_layer(x, swapped, dn, ids, w, nthreads=2) - out)) > 1e-3 * scale
    assert np.max(np.abs(oracle.moe_layer(x, gu, dn, ids, w[:, ::-1].copy(), nthreads=2) - out)) > 1e-3 * scale


def test_layer_with_one_expert_reduces_to_linear_layers():
    """E=1, k=1: the layer is F.linear on the dequantised weights
    ("dg-w4-kernels" -- W4A16: w4a16_linear(x, ...) == F.linear(x, dequant(W)))."""
    import torch
    cfg = wl.LayerShape("one", 5, 256, 128, 1, 1, seed=3)
    x = wl.activations(cfg)
    gu = oracle.quantize_w4(wl.all_gate_up_weights(cfg), 128)
    dn = oracle.quantize_w4(wl.all_down_weights(cfg), 64)
    ids = np.zeros((5, 1), np.int32)
    w = np.ones((5, 1), np.float32)
    out = oracle.moe_layer(x, gu, dn, ids, w, nthreads=1)
    xt = torch.tensor((x.astype(np.uint32) << 16).view(np.float32), dtype=torch.float64)
    Wgu = torch.tensor(oracle.dequant_w4(*gu, 128)[0])
    Wdn = torch.tensor(oracle.dequant_w4(*dn, 64)[0])
    gu_out = torch.nn.functional.linear(xt, Wgu)
    h = torch.nn.functional.gelu(gu_out[:, :128], approximate="tanh") * gu_out[:, 128:]
    ref = torch.nn.functional.linear(h, Wdn).numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-14)


def test_combine_is_a_plain_weighted_sum_and_thread_count_free():
    cfg = wl.CONFIGS["tiny"]
    x, gu, dn, ids, w = _quantized_layer(cfg)
    out1, h, y = oracle.moe_layer(x, gu, dn, ids, w, nthreads=1, want_intermediates=True)
    out7 = oracle.moe_layer(x, gu, dn, ids, w, nthreads=7)
    assert np.array_equal(out1, out7)      # same bits for any thread count
    yk = y.reshape(cfg.M, cfg.k, cfg.d)
    ref = np.einsum("tj,tjd->td", w.astype(np.float64), yk)
    assert np.allclose(out1, ref, rtol=1e-13, atol=1e-15)
    # reversing the slot order changes float64 results only by rounding
    rev = np.einsum("tj,tjd->td", w[:, ::-1].astype(np.float64), yk[:, ::-1])
    assert np.max(np.abs(rev - out1)) <= 1e-13 * np.max(np.abs(out1))


def test_invalid_ids_are_skipped():
    cfg = wl.CONFIGS["tiny"]
    x, gu, dn, ids, w = _quantized_layer(cfg)
    bad = ids.copy()
    bad[3, 1] = cfg.E + 5
    bad[7, 0] = -1
    out = oracle.moe_layer(x, gu, dn, bad, w, nthreads=2)
    ref = oracle.moe_layer(x, gu, dn, ids, w, nthreads=2, want_intermediates=True)
    yk = ref[2].reshape(cfg.M, cfg.k, cfg.d)
    assert np.allclose(out[3], w[3, 0] * yk[3, 0], rtol=1e-13)
    assert np.allclose(out[7], w[7, 1] * yk[7, 1], rtol=1e-13)
