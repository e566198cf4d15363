"""Float64 CPU oracle for the W4A16 routed mixture-of-experts layer.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
package.  It shares nothing with the CUDA library: the arithmetic lives in
``w4moe_oracle.c`` (the MoE layer) and ``sampler_norm_oracle.c`` (RMSNorm,
entropy, Gumbel-max sampler), plain C in float64, and this module only
compiles them with gcc, loads them with ctypes and marshals numpy arrays.

Each wrapper names the passage of the pages it follows (page title and
section); the readings taken where the pages are silent are listed at the top
of ``w4moe_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "w4moe_oracle.c"), os.path.join(_HERE, "sampler_norm_oracle.c")]
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no FMA contraction, IEEE semantics)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(f) for f in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off",
           "-fno-fast-math", "-fPIC", "-shared", "-pthread", "-o", tmp, *_SRCS, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_f32_to_f16.argtypes = [f32]
        lib.oracle_f32_to_f16.restype = ctypes.c_uint16
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_pack_codes.argtypes = [P, i64, P]
        lib.oracle_unpack_codes.argtypes = [P, i64, P]
        lib.oracle_quantize_w4.argtypes = [P, i64, i64, i32, P, P, P]
        lib.oracle_quantize_w4.restype = i32
        lib.oracle_dequant_w4.argtypes = [P, P, P, i64, i64, i32, P]
        lib.oracle_route.argtypes = [P, i32, i32, i32, P, P]
        lib.oracle_route.restype = i32
        lib.oracle_align_capacity.argtypes = [i32, i32, i32, i32]
        lib.oracle_align_capacity.restype = i64
        lib.oracle_moe_align.argtypes = [P, i32, i32, i32, i32, P, P, P, P]
        lib.oracle_moe_align.restype = i64
        lib.oracle_gelu_tanh.argtypes = [ctypes.c_double]
        lib.oracle_gelu_tanh.restype = ctypes.c_double
        lib.oracle_moe_layer.argtypes = [P, i32, i32, i32, i32, i32,
                                         P, P, P, i32, P, P, P, i32,
                                         P, P, i32, P, P, P]
        lib.oracle_moe_layer.restype = i32
        lib.oracle_w4a16_linear.argtypes = [P, i32, i32, i32, P, P, P, i32, i32, P]
        lib.oracle_w4a16_linear.restype = i32
        u32, u64 = ctypes.c_uint32, ctypes.c_uint64
        lib.oracle_rmsnorm.argtypes = [P, P, i32, i32, ctypes.c_double, P]
        lib.oracle_philox4x32_10.argtypes = [P, P, P]
        lib.oracle_noise_word.argtypes = [u64, u64, i64, i64]
        lib.oracle_noise_word.restype = u32
        lib.oracle_gumbel_of_word.argtypes = [u32]
        lib.oracle_gumbel_of_word.restype = ctypes.c_double
        lib.oracle_entropy.argtypes = [P, i32, i64, P, i32]
        lib.oracle_gumbel_argmax.argtypes = [P, i32, i64, u64, u64, P, P, P, P, i32]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------
def f16_to_f64(bits: int) -> float:
    """binary16 bits -> value (IEEE-754 definition)."""
    return _load().oracle_f16_to_f64(int(bits) & 0xFFFF)


def f32_to_f16(v: float) -> int:
    """binary32 value -> binary16 bits, round to nearest even."""
    return int(_load().oracle_f32_to_f16(float(np.float32(v))))


def f16_bits_to_f64_array(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_f16_to_f64(int(b)) for b in flat],
                    dtype=np.float64).reshape(np.shape(bits))


def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(int(bits) & 0xFFFF)


# --------------------------------------------------------------------------
# "diffusiongemma-26B-A4B-w4a16" -- Checkpoint format: packing
# --------------------------------------------------------------------------
def pack_codes(codes: np.ndarray) -> np.ndarray:
    """byte j = q[2j] | q[2j+1] << 4 along the last axis."""
    c = _c(codes, np.uint8)
    assert c.shape[-1] % 2 == 0
    out = np.empty(c.shape[:-1] + (c.shape[-1] // 2,), np.uint8)
    _load().oracle_pack_codes(_ptr(c), c.size, _ptr(out))
    return out


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    p = _c(packed, np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), np.uint8)
    _load().oracle_unpack_codes(_ptr(p), out.size, _ptr(out))
    return out


def quantize_w4(W: np.ndarray, group: int):
    """Asymmetric uint4 min/max round-to-nearest quantisation.

    "diffusiongemma-26B-A4B-w4a16" -- Checkpoint format and Benchmarks;
    "Inference: Making every denoising pass fast" -- The first constraint
    was capacity.  ``W`` is [..., K] fp32; returns (q [..., K/2] uint8,
    s [..., K/group] uint16 fp16 bits, z [..., K/group] uint16 fp16 bits).
    """
    w = _c(W, np.float32)
    K = w.shape[-1]
    rows = w.size // K
    lead = w.shape[:-1]
    q = np.empty(lead + (K // 2,), np.uint8)
    s = np.empty(lead + (K // group,), np.uint16)
    z = np.empty(lead + (K // group,), np.uint16)
    rc = _load().oracle_quantize_w4(_ptr(w), rows, K, group, _ptr(q), _ptr(s), _ptr(z))
    if rc != 0:
        raise ValueError(f"oracle_quantize_w4: unsupported shape K={K} group={group}")
    return q, s, z


def dequant_w4(q: np.ndarray, s: np.ndarray, z: np.ndarray, group: int) -> np.ndarray:
    """w_hat = s_g * (q - z_g) in float64, shape [..., K]."""
    q = _c(q, np.uint8)
    s = _c(s, np.uint16)
    z = _c(z, np.uint16)
    K = q.shape[-1] * 2
    rows = q.size // q.shape[-1]
    out = np.empty(q.shape[:-1] + (K,), np.float64)
    _load().oracle_dequant_w4(_ptr(q), _ptr(s), _ptr(z), rows, K, group, _ptr(out))
    return out


# --------------------------------------------------------------------------
# "Inference: Making every denoising pass fast" -- Quantisation alone leaves a
# sparse execution problem: router, alignment, expert MLP, combine
# --------------------------------------------------------------------------
def route(logits: np.ndarray, k: int):
    """softmax (float64) -> top-k (ties to the lower index) -> renormalise."""
    l = _c(logits, np.float32)
    M, E = l.shape
    ids = np.empty((M, k), np.int32)
    w = np.empty((M, k), np.float32)
    if _load().oracle_route(_ptr(l), M, E, k, _ptr(ids), _ptr(w)) != 0:
        raise ValueError("oracle_route: bad arguments")
    return ids, w


def align_capacity(M: int, k: int, E: int, block_m: int) -> int:
    return int(_load().oracle_align_capacity(M, k, E, block_m))


def moe_align(ids: np.ndarray, E: int, block_m: int):
    """Counting sort of flat assignments by expert, stable, padded to block_m.

    Returns dict(sorted_ids, block_expert, expert_offsets, num_padded, bad).
    """
    i = _c(ids, np.int32)
    M, k = i.shape
    cap = align_capacity(M, k, E, block_m)
    sorted_ids = np.empty(cap, np.int32)
    block_expert = np.empty(cap // block_m, np.int32)
    offs = np.empty(E + 1, np.int32)
    npad = np.empty(1, np.int32)
    bad = _load().oracle_moe_align(_ptr(i), M, k, E, block_m, _ptr(sorted_ids),
                                   _ptr(block_expert), _ptr(offs), _ptr(npad))
    if bad < 0:
        raise ValueError("oracle_moe_align: bad arguments")
    return dict(sorted_ids=sorted_ids, block_expert=block_expert,
                expert_offsets=offs, num_padded=int(npad[0]), bad=int(bad))


def gelu_tanh(v: float) -> float:
    return _load().oracle_gelu_tanh(float(v))


def moe_layer(x_bf16_bits: np.ndarray, gu, dn, ids: np.ndarray, weights: np.ndarray,
              gu_group: int = 128, dn_group: int = 64, nthreads: int | None = None,
              want_intermediates: bool = False):
    """The whole layer in float64: per token, per selected expert, dequantised
    gate_up, gelu_tanh(gate) * up, dequantised down, then the fixed-order
    weighted combine.

    x_bf16_bits [M, d] uint16; gu = (q [E,2m,d/2], s, z); dn = (q [E,d,m/2], s, z);
    ids [M, k] int32; weights [M, k] fp32.  Returns out [M, d] float64, or
    (out, h [M*k, m], y [M*k, d]) when want_intermediates.
    """
    x = _c(x_bf16_bits, np.uint16)
    M, d = x.shape
    gq, gs, gz = (_c(gu[0], np.uint8), _c(gu[1], np.uint16), _c(gu[2], np.uint16))
    dq, ds, dz = (_c(dn[0], np.uint8), _c(dn[1], np.uint16), _c(dn[2], np.uint16))
    E = gq.shape[0]
    m = gq.shape[1] // 2
    assert gq.shape == (E, 2 * m, d // 2) and dq.shape == (E, d, m // 2)
    i = _c(ids, np.int32)
    w = _c(weights, np.float32)
    k = i.shape[1]
    assert i.shape == (M, k) and w.shape == (M, k)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    out = np.empty((M, d), np.float64)
    h = np.empty((M * k, m), np.float64) if want_intermediates else None
    y = np.empty((M * k, d), np.float64) if want_intermediates else None
    rc = _load().oracle_moe_layer(
        _ptr(x), M, d, m, E, k, _ptr(gq), _ptr(gs), _ptr(gz), gu_group,
        _ptr(dq), _ptr(ds), _ptr(dz), dn_group, _ptr(i), _ptr(w), int(nthreads),
        _ptr(h) if h is not None else None, _ptr(y) if y is not None else None, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_moe_layer: bad arguments")
    return (out, h, y) if want_intermediates else out


# --------------------------------------------------------------------------
# "dg-w4-kernels" -- W4A16: the dense linear
# --------------------------------------------------------------------------
def w4a16_linear(x_bf16_bits: np.ndarray, q: np.ndarray, s: np.ndarray, z: np.ndarray,
                 group: int = 128, nthreads: int | None = None) -> np.ndarray:
    """y = x . deq(W)^T in float64 (F.linear of the dequantised weight).

    x [M, K] bf16 bits; q [N, K/2] packed codes, s/z [N, K/group] fp16 bits;
    returns y [M, N] float64."""
    x = _c(x_bf16_bits, np.uint16)
    q = _c(q, np.uint8)
    s = _c(s, np.uint16)
    z = _c(z, np.uint16)
    M, K = x.shape
    N = q.shape[0]
    assert q.shape == (N, K // 2) and s.shape == (N, K // group) and z.shape == s.shape
    y = np.empty((M, N), np.float64)
    rc = _load().oracle_w4a16_linear(_ptr(x), M, K, N, _ptr(q), _ptr(s), _ptr(z), group,
                                     int(nthreads or os.cpu_count() or 1), _ptr(y))
    if rc != 0:
        raise ValueError("oracle_w4a16_linear: bad arguments")
    return y


# --------------------------------------------------------------------------
# "dg-w4-kernels" -- RMSNorm
# --------------------------------------------------------------------------
def rmsnorm(x_bf16_bits: np.ndarray, w_bf16_bits: np.ndarray, eps: float) -> np.ndarray:
    """y = x / sqrt(mean(x^2) + eps) * weight per row, float64, unrounded.

    x [M, d] and weight [d] are bf16 bit patterns (uint16)."""
    x = _c(x_bf16_bits, np.uint16)
    w = _c(w_bf16_bits, np.uint16)
    M, d = x.shape
    assert w.shape == (d,)
    y = np.empty((M, d), np.float64)
    _load().oracle_rmsnorm(_ptr(x), _ptr(w), M, d, float(eps), _ptr(y))
    return y


# --------------------------------------------------------------------------
# "dg-w4-kernels" -- Sampler: fused_entropy, gumbel_argmax_sample
# --------------------------------------------------------------------------
def philox4x32_10(counter, key) -> np.ndarray:
    """Philox4x32-10 (Salmon et al., SC 2011) of one counter under one key."""
    c = np.array(counter, np.uint32)
    k = np.array(key, np.uint32)
    out = np.empty(4, np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def noise_word(seed: int, offset: int, t: int, i: int) -> int:
    """The 32-bit Philox word of row t, column i: key (seed lo, seed hi),
    counter (i // 4, t, offset lo, offset hi), word i % 4."""
    return int(_load().oracle_noise_word(seed, offset, t, i))


def gumbel_of_word(r: int) -> float:
    """g = -ln(-ln(1 - v)), v = (r + 1/2) / 2^32."""
    return float(_load().oracle_gumbel_of_word(int(r) & 0xFFFFFFFF))


def entropy(logits: np.ndarray, nthreads: int | None = None) -> np.ndarray:
    """-sum p ln p of softmax over the last axis, float64 nats."""
    l = _c(logits, np.float32)
    M, V = l.shape
    H = np.empty(M, np.float64)
    _load().oracle_entropy(_ptr(l), M, V, _ptr(H), int(nthreads or os.cpu_count() or 1))
    return H


def gumbel_argmax(logits: np.ndarray, seed: int, offset: int = 0,
                  nthreads: int | None = None):
    """Gumbel-max sample and plain argmax per row (ties to the lower index).

    Returns dict(sample, argmax, best, second): best and second are the two
    largest perturbed scores logit + g in float64."""
    l = _c(logits, np.float32)
    M, V = l.shape
    sample = np.empty(M, np.int64)
    amax = np.empty(M, np.int64)
    best = np.empty(M, np.float64)
    second = np.empty(M, np.float64)
    _load().oracle_gumbel_argmax(_ptr(l), M, V, seed & (2**64 - 1), offset & (2**64 - 1),
                                 _ptr(sample), _ptr(amax), _ptr(best), _ptr(second),
                                 int(nthreads or os.cpu_count() or 1))
    return dict(sample=sample, argmax=amax, best=best, second=second)
