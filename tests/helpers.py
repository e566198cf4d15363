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
