"""Shared helpers for the parity tests: seeded inputs from the workloads
module, uploaded to the GPU for the CUDA path and kept on the host for the
oracle.  Nothing here does any of the layer's arithmetic."""
from __future__ import annotations

import functools

import numpy as np

from w4a16_moe_expert_sync_gb300 import workloads as wl


def rel_max_err(got, ref) -> float:
    """max |got - ref| / rms(ref), the layer's parity metric."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    return float(np.max(np.abs(got - ref)) / rms) if ref.size else 0.0


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (via torch), as float64:
    the error floor any bf16 output carries."""
    import torch
    return torch.from_numpy(np.asarray(a, np.float64)).to(torch.bfloat16).double().numpy()


def torch_bf16_to_f64(t) -> np.ndarray:
    import torch
    return bf16_bits_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))


@functools.lru_cache(maxsize=2)
def gpu_weights(name: str):
    """Quantise every expert of a workload on the GPU with w4_quantize.
    Returns ((gu_q, gu_s, gu_z), (dn_q, dn_s, dn_z)) as CUDA tensors."""
    import torch
    import w4a16_moe_expert_sync_gb300 as w4
    cfg = wl.CONFIGS[name]
    dev = torch.device("cuda")
    gu = (torch.empty((cfg.E, 2 * cfg.m, cfg.d // 2), dtype=torch.uint8, device=dev),
          torch.empty((cfg.E, 2 * cfg.m, cfg.d // cfg.gu_group), dtype=torch.float16, device=dev),
          torch.empty((cfg.E, 2 * cfg.m, cfg.d // cfg.gu_group), dtype=torch.float16, device=dev))
    dn = (torch.empty((cfg.E, cfg.d, cfg.m // 2), dtype=torch.uint8, device=dev),
          torch.empty((cfg.E, cfg.d, cfg.m // cfg.dn_group), dtype=torch.float16, device=dev),
          torch.empty((cfg.E, cfg.d, cfg.m // cfg.dn_group), dtype=torch.float16, device=dev))
    for e in range(cfg.E):
        wg = torch.from_numpy(wl.gate_up_weight(cfg, e)).to(dev)
        w4.w4_quantize(wg, cfg.gu_group, out=tuple(t[e:e + 1] for t in gu))
        wd = torch.from_numpy(wl.down_weight(cfg, e)).to(dev)
        w4.w4_quantize(wd, cfg.dn_group, out=tuple(t[e:e + 1] for t in dn))
    torch.cuda.synchronize()
    return gu, dn


def oracle_weights(cfg, experts):
    """Oracle-quantised weights for the listed experts, scattered into full
    [E, ...] arrays (other experts left zero: the sampled tokens never use them)."""
    import oracle
    gu_q = np.zeros((cfg.E, 2 * cfg.m, cfg.d // 2), np.uint8)
    gu_s = np.zeros((cfg.E, 2 * cfg.m, cfg.d // cfg.gu_group), np.uint16)
    gu_z = np.zeros_like(gu_s)
    dn_q = np.zeros((cfg.E, cfg.d, cfg.m // 2), np.uint8)
    dn_s = np.zeros((cfg.E, cfg.d, cfg.m // cfg.dn_group), np.uint16)
    dn_z = np.zeros_like(dn_s)
    for e in sorted(set(int(v) for v in experts)):
        gu_q[e], gu_s[e], gu_z[e] = oracle.quantize_w4(wl.gate_up_weight(cfg, e), cfg.gu_group)
        dn_q[e], dn_s[e], dn_z[e] = oracle.quantize_w4(wl.down_weight(cfg, e), cfg.dn_group)
    return (gu_q, gu_s, gu_z), (dn_q, dn_s, dn_z)


def gpu_inputs(name: str):
    """x (bf16) and router logits on the GPU, plus their host copies."""
    import torch
    cfg = wl.CONFIGS[name]
    x_bits = wl.activations(cfg)
    logits = wl.router_logits(cfg)
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda()
    lg = torch.from_numpy(logits).cuda()
    return cfg, x, lg, x_bits, logits


def job_covering_tokens(ids: np.ndarray, E: int, block_m: int = 16, job_slots: int = 32):
    """Tokens that together reach every job of every expert: the alignment
    splits an expert's padded slot range into jobs of `job_slots`; walking
    the jobs in order, the first token of each job not yet reached is taken.
    Used where the oracle cannot afford every token (the 2048-token canvas)."""
    import oracle
    M, k = ids.shape
    al = oracle.moe_align(ids, E, block_m)
    offs, sorted_ids = al["expert_offsets"], al["sorted_ids"]
    A = M * k
    covered = set()
    toks = []
    for e in range(E):
        for start in range(int(offs[e]), int(offs[e + 1]), job_slots):
            job = (e, start)
            if job in covered:
                continue
            a = int(sorted_ids[start])
            if a >= A:
                continue
            t = a // k
            toks.append(t)
            # every job this token's assignments fall in
            for j in range(k):
                aa = t * k + j
                slot = int(np.nonzero(sorted_ids == aa)[0][0])
                ee = int(ids[t, j])
                covered.add((ee, int(offs[ee]) + (slot - int(offs[ee])) // job_slots * job_slots))
    return np.array(sorted(set(toks)), dtype=np.int64)


@functools.lru_cache(maxsize=8)
def oracle_layer(name: str, token_set: str = "all"):
    """The oracle's layer on a workload, with its intermediates: returns
    (toks, ids, w, out, h, y) where toks are the tokens evaluated ("all", or
    "cover": job_covering_tokens), ids/w the oracle's routing of every
    token, and out [len(toks), d], h/y [len(toks)*k, ...] the oracle's
    results for those tokens only."""
    import oracle
    cfg = wl.CONFIGS[name]
    x_bits = wl.activations(cfg)
    ids, w = oracle.route(wl.router_logits(cfg), cfg.k)
    toks = (np.arange(cfg.M) if token_set == "all" else job_covering_tokens(ids, cfg.E))
    ogu, odn = oracle_weights(cfg, ids[toks].ravel())
    out, h, y = oracle.moe_layer(x_bits[toks], ogu, odn, ids[toks], w[toks],
                                 want_intermediates=True)
    return toks, ids, w, out, h, y


def elementwise_excess(got, ref, rel: float) -> float:
    """max over elements of (|got - ref| - rel * |ref|) / rms(ref): the part of
    each element's error that its own rounding (rel * |ref|) does not account
    for, in units of the reference's rms.  <= tau means every element is
    within rel * |ref| + tau * rms(ref)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    if not ref.size:
        return 0.0
    return float(np.max(np.abs(got - ref) - rel * np.abs(ref)) / rms)
