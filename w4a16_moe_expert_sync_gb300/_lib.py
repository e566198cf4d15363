"""ctypes binding of libw4moe.so: the C entry points of include/w4moe.h under
the same names, taking torch tensors.  Argument marshalling only: shapes are
read from the tensors, outputs are allocated with torch (device memory), the
pointers and the current CUDA stream are passed through, and a nonzero status
raises W4Error.  Every step of the layer runs in the library's CUDA kernels;
there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from .build import LIB as _LIB_PATH

_lock = threading.Lock()
_lib = None

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "w4moe.h")

# device status bits (include/w4moe.h)
W4_DEV_BAD_EXPERT_ID = 0x1
W4_DEV_PIPELINE_TIMEOUT = 0x2
W4_DEV_TOO_MANY_JOBS = 0x4
W4_DEV_FP16_RANGE = 0x8
W4_DEV_OUT_OF_BOUNDS = 0x10
# xg and h rows end in one block of 64 columns of activation group sums, the
# grouped GEMMs' input for the low parts of their dequantisation constants
SUM_COLS = 64


class W4Error(RuntimeError):
    def __init__(self, status: int, name: str, detail: str):
        super().__init__(f"{name} ({status}): {detail}")
        self.status = status
        self.name = name
        self.detail = detail


def header_functions() -> list[str]:
    """Names of the functions declared in include/w4moe.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(w4_[a-z_0-9]+)\s*\(",
                                 text, flags=re.M)))


def load_library(path: str | None = None):
    """Load libw4moe.so (built by __graft_entry__.build()); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build the CUDA library first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        V, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        U64 = ctypes.c_uint64
        sig = {
            "w4_status_string": ([I], ctypes.c_char_p),
            "w4_last_error_detail": ([], ctypes.c_char_p),
            "w4_abi_version": ([], I),
            "w4_quantize": ([V, I, I, I, I, V, V, V, V], I),
            "w4_moe_route": ([V, I, I, I, V, V, V], I),
            "w4_moe_align_capacity": ([I, I, I, I], I64),
            "w4_moe_align": ([V, I, I, I, I, V, V, V, V, V, V], I),
            "w4_gather_activations": ([V, I, I, I, I, I, V, V, V, V, V], I),
            "w4_moe_align_gather": ([V, V, I, I, I, I, I, V, V, V, V, V, V, V], I),
            "w4_moe_route_align_gather": ([V, V, I, I, I, I, I, V, V, V, V, V, V, V, V, V],
                                          I),
            "w4_grouped_gemm_gate_up": ([V, I, I, I, I, I, I, V, V, V, I, V, V, V, V, V], I),
            "w4_grouped_gemm_down": ([V, I, I, I, I, I, I, V, V, V, I, V, V, V, V, V], I),
            "w4_moe_combine_fixed_order": ([V, V, V, I, I, I, I, V, V], I),
            "w4_grouped_gemm_down_combine": ([V, I, I, I, I, I, I, V, V, V, I, V, V, V, V, V, V,
                                              V, V, V], I),
            "w4_moe_combine_prepare": ([V, I, I, I, I, V, V, V], I),
            "w4_test_pipeline_hooks": ([U64, I], I),
            "w4_moe_layer_workspace_size": ([I, I, I, I, I, I], SZ),
            "w4_moe_layer": ([V, V, V, I, I, I, I, I, I, V, V, V, I, V, V, V, I, V, SZ, V, V,
                              V], I),
            "w4_moe_layer_host_workspace_size": ([I, I, I, I, I, I], SZ),
            "w4_moe_layer_host": ([V, V, V, I, I, I, I, I, I, V, V, V, I, V, V, V, I, V, SZ, V,
                                   V, V], I),
            "w4_moe_layer_static_scratch": ([V, V, V, I, I, I, I, I, I, V, V, V, I, V, V, V, I,
                                             V, V, V], I),
            "w4_moe_layer_from_logits": ([V, V, I, I, I, I, I, I, V, V, V, I, V, V, V, I, V,
                                          SZ, V, V, V, V, V], I),
            "w4_w4a16_linear_workspace_size": ([I, I, I, I], SZ),
            "w4_w4a16_linear": ([V, I, I, I, V, V, V, I, V, SZ, V, V, V], I),
            "w4_rmsnorm": ([V, V, I, I, ctypes.c_float, V, V], I),
            "w4_sample_logits_workspace_size": ([I, I64], SZ),
            "w4_sample_logits": ([V, I, I64, U64, U64, V, V, V, V, SZ, V], I),
            "w4_fused_entropy": ([V, I, I64, V, V, SZ, V], I),
            "w4_gumbel_argmax_sample": ([V, I, I64, U64, U64, V, V, V, SZ, V], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(rc: int, what: str):
    if rc != 0:
        lib = load_library()
        raise W4Error(rc, lib.w4_status_string(rc).decode(),
                      f"{what}: {lib.w4_last_error_detail().decode()}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors passed to the CUDA library must live on the GPU")
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors passed to the CUDA library must be contiguous")


# --------------------------------------------------------------------------
# entry points (same names as the C ABI)
# --------------------------------------------------------------------------
def w4_quantize(W, group: int, out=None, stream=None):
    """quantize_w4: W [E, N, K] fp32 -> (q [E,N,K/2] u8, s, z [E,N,K/group] fp16)."""
    import torch
    _require_cuda(W)
    if W.dim() == 2:
        W = W.unsqueeze(0)
    E, N, K = W.shape
    if out is None:
        out = (torch.empty((E, N, K // 2), dtype=torch.uint8, device=W.device),
               torch.empty((E, N, K // group), dtype=torch.float16, device=W.device),
               torch.empty((E, N, K // group), dtype=torch.float16, device=W.device))
    q, s, z = out
    _check(load_library().w4_quantize(_ptr(W), E, N, K, group, _ptr(q), _ptr(s), _ptr(z),
                                      _stream(stream)), "w4_quantize")
    return q, s, z


def w4_moe_route(logits, k: int, stream=None):
    """Router: logits [M, E] fp32 -> (topk_ids [M,k] int32, topk_weights [M,k] fp32)."""
    import torch
    _require_cuda(logits)
    M, E = logits.shape
    ids = torch.empty((M, k), dtype=torch.int32, device=logits.device)
    w = torch.empty((M, k), dtype=torch.float32, device=logits.device)
    _check(load_library().w4_moe_route(_ptr(logits), M, E, k, _ptr(ids), _ptr(w),
                                       _stream(stream)), "w4_moe_route")
    return ids, w


def w4_moe_align_capacity(M: int, k: int, E: int, block_m: int) -> int:
    cap = load_library().w4_moe_align_capacity(M, k, E, block_m)
    if cap < 0:
        raise W4Error(1, "W4_ERR_INVALID_ARG", "w4_moe_align_capacity: bad arguments")
    return int(cap)


def w4_moe_align(topk_ids, E: int, block_m: int = 16, dev_status=None, out=None,
                 stream=None):
    """Alignment: topk_ids [M, k] int32 -> dict of device tensors (sorted_ids,
    block_expert, expert_offsets, num_padded) plus the shape keys the GEMMs
    need.  Pass a previous result as ``out`` to reuse its buffers."""
    import torch
    _require_cuda(topk_ids, dev_status)
    M, k = topk_ids.shape
    cap = w4_moe_align_capacity(M, k, E, block_m)
    dev = topk_ids.device
    if out is not None:
        if (out["sorted_ids"].numel() != cap or out["expert_offsets"].numel() != E + 1
                or out["block_expert"].numel() != cap // block_m):
            raise ValueError("w4_moe_align: reused buffers have the wrong sizes")
        r = out
        r.update(M=M, k=k, E=E, block_m=block_m)
    else:
        r = dict(sorted_ids=torch.empty(cap, dtype=torch.int32, device=dev),
                 block_expert=torch.empty(cap // block_m, dtype=torch.int32, device=dev),
                 expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                 num_padded=torch.empty(1, dtype=torch.int32, device=dev),
                 M=M, k=k, E=E, block_m=block_m)
    _check(load_library().w4_moe_align(_ptr(topk_ids), M, k, E, block_m, _ptr(r["sorted_ids"]),
                                       _ptr(r["block_expert"]), _ptr(r["expert_offsets"]),
                                       _ptr(r["num_padded"]), _ptr(dev_status),
                                       _stream(stream)), "w4_moe_align")
    return r


def w4_gather_activations(x, align: dict, out=None, dev_status=None, stream=None):
    """x [M, d] bf16 -> xg [cap, d + 64] fp16 in slot order: d values in block
    order, then the sums of the groups of 128 (zero rows for padding slots;
    rows past num_padded are left untouched).  Values beyond fp16's range
    saturate and set W4_DEV_FP16_RANGE in dev_status."""
    import torch
    _require_cuda(x, out, dev_status)
    M, d = x.shape
    cap = align["sorted_ids"].numel()
    if out is None:
        out = torch.empty((cap, d + SUM_COLS), dtype=torch.float16, device=x.device)
    _check(load_library().w4_gather_activations(
        _ptr(x), M, d, align["k"], align["E"], align["block_m"], _ptr(align["sorted_ids"]),
        _ptr(align["num_padded"]), _ptr(out), _ptr(dev_status), _stream(stream)),
        "w4_gather_activations")
    return out


def w4_moe_align_gather(topk_ids, x, E: int, block_m: int = 16, dev_status=None, out=None,
                        xg=None, stream=None):
    """Alignment and activation gather in one launch.  Returns (align dict, xg)."""
    import torch
    _require_cuda(topk_ids, x, dev_status, xg)
    M, k = topk_ids.shape
    d = x.shape[1]
    cap = w4_moe_align_capacity(M, k, E, block_m)
    dev = x.device
    if out is None:
        out = dict(sorted_ids=torch.empty(cap, dtype=torch.int32, device=dev),
                   block_expert=torch.empty(cap // block_m, dtype=torch.int32, device=dev),
                   expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   num_padded=torch.empty(1, dtype=torch.int32, device=dev))
    out.update(M=M, k=k, E=E, block_m=block_m)
    if xg is None:
        xg = torch.empty((cap, d + SUM_COLS), dtype=torch.float16, device=dev)
    _check(load_library().w4_moe_align_gather(
        _ptr(topk_ids), _ptr(x), M, d, k, E, block_m, _ptr(out["sorted_ids"]),
        _ptr(out["block_expert"]), _ptr(out["expert_offsets"]), _ptr(out["num_padded"]),
        _ptr(xg), _ptr(dev_status), _stream(stream)), "w4_moe_align_gather")
    return out, xg


def w4_grouped_gemm_gate_up(xg, gu_q, gu_s, gu_z, align: dict, group: int = 128, h=None,
                            dev_status=None, stream=None):
    """xg [cap, d + 64] fp16 (from w4_gather_activations) -> h [cap, m + 64]
    fp16: m values in block order, gelu_tanh(gate) * up per alignment slot,
    then the sums of every quarter (16 values) of each group of 64."""
    import torch
    _require_cuda(xg, gu_q, gu_s, gu_z, h, dev_status)
    M, d = align["M"], xg.shape[1] - SUM_COLS
    E, two_m, _ = gu_q.shape
    m = two_m // 2
    cap = align["sorted_ids"].numel()
    if h is None:
        h = torch.empty((cap, m + SUM_COLS), dtype=torch.float16, device=xg.device)
    _check(load_library().w4_grouped_gemm_gate_up(
        _ptr(xg), M, d, m, E, align["k"], align["block_m"], _ptr(gu_q), _ptr(gu_s), _ptr(gu_z),
        group, _ptr(align["sorted_ids"]), _ptr(align["expert_offsets"]), _ptr(h),
        _ptr(dev_status), _stream(stream)), "w4_grouped_gemm_gate_up")
    return h


def korder_to_natural(a):
    """Undo the GEMMs' block order along the last axis (for inspection and
    tests): column p of every block of 8 holds element (p >> 1) + 4 * (p & 1)."""
    import numpy as np
    n = a.shape[-1]
    perm = np.array([(p >> 1) + 4 * (p & 1) for p in range(8)])
    src = (np.arange(n) // 8) * 8
    inv = np.empty(8, dtype=np.int64)
    inv[perm] = np.arange(8)
    return a[..., src + inv[np.arange(n) % 8]]


def w4_grouped_gemm_down(h, dn_q, dn_s, dn_z, align: dict, group: int = 64, y=None,
                         dev_status=None, stream=None):
    """h [cap, m + 64] fp16 (from w4_grouped_gemm_gate_up) -> y [M*k, d] fp32
    (row = flat assignment index)."""
    import torch
    _require_cuda(h, dn_q, dn_s, dn_z, y, dev_status)
    E, d, half_m = dn_q.shape
    m = half_m * 2
    M, k = align["M"], align["k"]
    if y is None:
        y = torch.empty((M * k, d), dtype=torch.float32, device=h.device)
    _check(load_library().w4_grouped_gemm_down(
        _ptr(h), M, d, m, E, k, align["block_m"], _ptr(dn_q), _ptr(dn_s), _ptr(dn_z), group,
        _ptr(align["sorted_ids"]), _ptr(align["expert_offsets"]), _ptr(y), _ptr(dev_status),
        _stream(stream)), "w4_grouped_gemm_down")
    return y


def w4_moe_combine_fixed_order(y, topk_ids, topk_weights, E: int, out=None, stream=None):
    """out [M, d] bf16 = fixed-order sum_j w[t,j] * y[t*k+j]."""
    import torch
    _require_cuda(y, topk_ids, topk_weights, out)
    M, k = topk_ids.shape
    d = y.shape[1]
    if out is None:
        out = torch.empty((M, d), dtype=torch.bfloat16, device=y.device)
    _check(load_library().w4_moe_combine_fixed_order(
        _ptr(y), _ptr(topk_ids), _ptr(topk_weights), M, k, d, E, _ptr(out), _stream(stream)),
        "w4_moe_combine_fixed_order")
    return out


def w4_moe_combine_prepare(topk_ids, E: int, d: int, counters=None, out=None, stream=None):
    """The counters [M, d/128] int32 of w4_grouped_gemm_down_combine (and
    the zero out rows of tokens with no valid expert id); returns
    (counters, out)."""
    import torch
    _require_cuda(topk_ids, counters, out)
    M, k = topk_ids.shape
    if counters is None:
        counters = torch.empty((M, d // 128), dtype=torch.int32, device=topk_ids.device)
    if out is None:
        out = torch.empty((M, d), dtype=torch.bfloat16, device=topk_ids.device)
    _check(load_library().w4_moe_combine_prepare(
        _ptr(topk_ids), M, k, E, d, _ptr(counters), _ptr(out), _stream(stream)),
        "w4_moe_combine_prepare")
    return counters, out


def w4_grouped_gemm_down_combine(h, dn_q, dn_s, dn_z, align: dict, topk_ids, topk_weights,
                                 counters, out, group: int = 64, y=None, dev_status=None,
                                 stream=None):
    """w4_grouped_gemm_down with the fixed-order combine folded in: out
    [M, d] bf16 (prepared with w4_moe_combine_prepare, which set counters);
    returns (y, out)."""
    import torch
    _require_cuda(h, dn_q, dn_s, dn_z, topk_ids, topk_weights, counters, out, y, dev_status)
    E, d, half_m = dn_q.shape
    m = half_m * 2
    M, k = align["M"], align["k"]
    if y is None:
        y = torch.empty((M * k, d), dtype=torch.float32, device=h.device)
    _check(load_library().w4_grouped_gemm_down_combine(
        _ptr(h), M, d, m, E, k, align["block_m"], _ptr(dn_q), _ptr(dn_s), _ptr(dn_z), group,
        _ptr(align["sorted_ids"]), _ptr(align["expert_offsets"]), _ptr(topk_ids),
        _ptr(topk_weights), _ptr(counters), _ptr(y), _ptr(out), _ptr(dev_status),
        _stream(stream)), "w4_grouped_gemm_down_combine")
    return y, out


def w4_moe_layer_workspace_size(M, d, m, E, k, block_m=16) -> int:
    return int(load_library().w4_moe_layer_workspace_size(M, d, m, E, k, block_m))


def w4_moe_layer(x, topk_ids, topk_weights, gu, dn, block_m: int = 16, gu_group: int = 128,
                 dn_group: int = 64, workspace=None, out=None, dev_status=None, stream=None):
    """The whole routed-expert layer (align+gather, gate_up + activation,
    down, fixed-order combine) as four launches on the current stream."""
    import torch
    gu_q, gu_s, gu_z = gu
    dn_q, dn_s, dn_z = dn
    _require_cuda(x, topk_ids, topk_weights, gu_q, gu_s, gu_z, dn_q, dn_s, dn_z, workspace,
                  out, dev_status)
    M, d = x.shape
    E, two_m, _ = gu_q.shape
    m = two_m // 2
    k = topk_ids.shape[1]
    need = w4_moe_layer_workspace_size(M, d, m, E, k, block_m)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty((M, d), dtype=torch.bfloat16, device=x.device)
    _check(load_library().w4_moe_layer(
        _ptr(x), _ptr(topk_ids), _ptr(topk_weights), M, d, m, E, k, block_m, _ptr(gu_q),
        _ptr(gu_s), _ptr(gu_z), gu_group, _ptr(dn_q), _ptr(dn_s), _ptr(dn_z), dn_group,
        _ptr(workspace), workspace.numel(), _ptr(out), _ptr(dev_status), _stream(stream)),
        "w4_moe_layer")
    return out


def w4_moe_layer_host_workspace_size(M, d, m, E, k, block_m=16) -> int:
    return int(load_library().w4_moe_layer_host_workspace_size(M, d, m, E, k, block_m))


def w4_moe_layer_host(x_host, topk_ids_host, topk_weights_host, gu, dn, out_host, workspace,
                      block_m: int = 16, gu_group: int = 128, dn_group: int = 64,
                      dev_status=None, stream=None):
    """w4_moe_layer from host memory: x [M, d] bf16, topk_ids [M, k] int32
    and topk_weights [M, k] fp32 (page-locked CPU tensors) are copied in and
    out [M, d] bf16 is copied back to out_host, all enqueued on the stream;
    synchronise before reading out_host.  workspace: a device uint8 tensor of
    w4_moe_layer_host_workspace_size(...) bytes."""
    gu_q, gu_s, gu_z = gu
    dn_q, dn_s, dn_z = dn
    _require_cuda(gu_q, gu_s, gu_z, dn_q, dn_s, dn_z, workspace, dev_status)
    for t in (x_host, topk_ids_host, topk_weights_host, out_host):
        if t.is_cuda:
            raise ValueError("w4_moe_layer_host takes host tensors for x, ids, weights and out")
    M, d = x_host.shape
    E, two_m, _ = gu_q.shape
    m = two_m // 2
    k = topk_ids_host.shape[1]
    _check(load_library().w4_moe_layer_host(
        _ptr(x_host), _ptr(topk_ids_host), _ptr(topk_weights_host), M, d, m, E, k, block_m,
        _ptr(gu_q), _ptr(gu_s), _ptr(gu_z), gu_group, _ptr(dn_q), _ptr(dn_s), _ptr(dn_z),
        dn_group, _ptr(workspace), workspace.numel(), _ptr(out_host), _ptr(dev_status),
        _stream(stream)), "w4_moe_layer_host")
    return out_host


def w4_moe_route_align_gather(logits, x, k: int, block_m: int = 16, dev_status=None, out=None,
                              xg=None, ids=None, weights=None, stream=None):
    """Router, alignment and activation gather in one launch, from the logits
    [M, E] fp32.  Returns (topk_ids, topk_weights, align dict, xg)."""
    import torch
    _require_cuda(logits, x, dev_status, xg, ids, weights)
    M, E = logits.shape
    d = x.shape[1]
    cap = w4_moe_align_capacity(M, k, E, block_m)
    dev = x.device
    if out is None:
        out = dict(sorted_ids=torch.empty(cap, dtype=torch.int32, device=dev),
                   block_expert=torch.empty(cap // block_m, dtype=torch.int32, device=dev),
                   expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   num_padded=torch.empty(1, dtype=torch.int32, device=dev))
    out.update(M=M, k=k, E=E, block_m=block_m)
    if xg is None:
        xg = torch.empty((cap, d + SUM_COLS), dtype=torch.float16, device=dev)
    if ids is None:
        ids = torch.empty((M, k), dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty((M, k), dtype=torch.float32, device=dev)
    _check(load_library().w4_moe_route_align_gather(
        _ptr(logits), _ptr(x), M, d, k, E, block_m, _ptr(ids), _ptr(weights),
        _ptr(out["sorted_ids"]), _ptr(out["block_expert"]), _ptr(out["expert_offsets"]),
        _ptr(out["num_padded"]), _ptr(xg), _ptr(dev_status), _stream(stream)),
        "w4_moe_route_align_gather")
    return ids, weights, out, xg


def w4_moe_layer_from_logits(x, logits, k: int, gu, dn, block_m: int = 16, gu_group: int = 128,
                             dn_group: int = 64, workspace=None, out=None, ids=None,
                             weights=None, dev_status=None, stream=None):
    """w4_moe_layer with the router in its first launch: from the logits
    [M, E] fp32.  Returns (out, topk_ids, topk_weights)."""
    import torch
    gu_q, gu_s, gu_z = gu
    dn_q, dn_s, dn_z = dn
    _require_cuda(x, logits, gu_q, gu_s, gu_z, dn_q, dn_s, dn_z, workspace, out, ids, weights,
                  dev_status)
    M, d = x.shape
    E, two_m, _ = gu_q.shape
    m = two_m // 2
    need = w4_moe_layer_workspace_size(M, d, m, E, k, block_m)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty((M, d), dtype=torch.bfloat16, device=x.device)
    if ids is None:
        ids = torch.empty((M, k), dtype=torch.int32, device=x.device)
    if weights is None:
        weights = torch.empty((M, k), dtype=torch.float32, device=x.device)
    _check(load_library().w4_moe_layer_from_logits(
        _ptr(x), _ptr(logits), M, d, m, E, k, block_m, _ptr(gu_q), _ptr(gu_s), _ptr(gu_z),
        gu_group, _ptr(dn_q), _ptr(dn_s), _ptr(dn_z), dn_group, _ptr(workspace),
        workspace.numel(), _ptr(ids), _ptr(weights), _ptr(out), _ptr(dev_status),
        _stream(stream)), "w4_moe_layer_from_logits")
    return out, ids, weights


def w4_moe_layer_static_scratch(x, topk_ids, topk_weights, gu, dn, out, block_m: int = 16,
                                gu_group: int = 128, dn_group: int = 64, dev_status=None,
                                stream=None):
    """w4_moe_layer with the intermediates in the library's own static device
    array instead of a workspace: for callers that cannot allocate device
    memory when they run the layer.  Nothing is allocated here either, so the
    caller passes `out` ([M, d] bf16).  Calls that overlap on the GPU share
    the array and race: keep them on one stream."""
    gu_q, gu_s, gu_z = gu
    dn_q, dn_s, dn_z = dn
    _require_cuda(x, topk_ids, topk_weights, gu_q, gu_s, gu_z, dn_q, dn_s, dn_z, out,
                  dev_status)
    M, d = x.shape
    E, two_m, _ = gu_q.shape
    m = two_m // 2
    k = topk_ids.shape[1]
    _check(load_library().w4_moe_layer_static_scratch(
        _ptr(x), _ptr(topk_ids), _ptr(topk_weights), M, d, m, E, k, block_m, _ptr(gu_q),
        _ptr(gu_s), _ptr(gu_z), gu_group, _ptr(dn_q), _ptr(dn_s), _ptr(dn_z), dn_group,
        _ptr(out), _ptr(dev_status), _stream(stream)), "w4_moe_layer_static_scratch")
    return out


def w4_w4a16_linear_workspace_size(M: int, K: int, N: int, group: int = 128) -> int:
    return int(load_library().w4_w4a16_linear_workspace_size(M, K, N, group))


def w4_w4a16_linear(x, q, s, z, group: int = 128, workspace=None, out=None, dev_status=None,
                    stream=None):
    """w4a16_linear: y [M, N] bf16 = x [M, K] bf16 . deq(W)^T with W packed as
    w4_quantize writes it (q [N, K/2] uint8, s/z [N, K/group] fp16)."""
    import torch
    _require_cuda(x, q, s, z, workspace, out, dev_status)
    M, K = x.shape
    N = q.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    need = w4_w4a16_linear_workspace_size(M, K, N, group)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    _check(load_library().w4_w4a16_linear(
        _ptr(x), M, K, N, _ptr(q), _ptr(s), _ptr(z), group, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _ptr(dev_status),
        _stream(stream)), "w4_w4a16_linear")
    return out


# --------------------------------------------------------------------------
# Beside the layer: RMSNorm and the sampler ("dg-w4-kernels" -- RMSNorm, Sampler)
# --------------------------------------------------------------------------
def w4_rmsnorm(x, weight, eps: float = 1e-6, out=None, stream=None):
    """fused_rmsnorm: y = x / sqrt(mean(x^2) + eps) * weight over the last
    axis; x [..., d] and weight [d] bf16, y bf16."""
    import torch
    _require_cuda(x, weight, out)
    d = x.shape[-1]
    M = x.numel() // d if d else 0
    if out is None:
        out = torch.empty_like(x)
    _check(load_library().w4_rmsnorm(_ptr(x), _ptr(weight), M, d, float(eps), _ptr(out),
                                     _stream(stream)), "w4_rmsnorm")
    return out


def w4_sample_logits_workspace_size(M: int, V: int) -> int:
    return int(load_library().w4_sample_logits_workspace_size(M, V))


def _sampler_ws(logits, workspace):
    import torch
    M, V = logits.shape
    need = w4_sample_logits_workspace_size(M, V)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=logits.device)
    return workspace, workspace.numel() * workspace.element_size()


def w4_sample_logits(logits, seed: int = 0, offset: int = 0, entropy=True, sample=True,
                     argmax=True, workspace=None, stream=None):
    """One pass over logits [M, V] fp32: (entropy [M] fp32 nats, Gumbel-max
    sample [M] int64, argmax [M] int64); an output passed as False is skipped
    (None in its place), a tensor is written in place."""
    import torch
    _require_cuda(logits, workspace)
    M, V = logits.shape
    dev = logits.device

    def out(spec, dtype):
        if spec is False or spec is None:
            return None
        if spec is True:
            return torch.empty(M, dtype=dtype, device=dev)
        _require_cuda(spec)
        return spec
    ent = out(entropy, torch.float32)
    smp = out(sample, torch.int64)
    amx = out(argmax, torch.int64)
    ws, ws_bytes = _sampler_ws(logits, workspace)
    _check(load_library().w4_sample_logits(
        _ptr(logits), M, V, seed & (2**64 - 1), offset & (2**64 - 1), _ptr(ent), _ptr(smp),
        _ptr(amx), _ptr(ws), ws_bytes, _stream(stream)), "w4_sample_logits")
    return ent, smp, amx


def w4_fused_entropy(logits, workspace=None, stream=None):
    """fused_entropy: [M, V] fp32 -> [M] fp32 nats, one pass."""
    ent, _, _ = w4_sample_logits(logits, entropy=True, sample=False, argmax=False,
                                 workspace=workspace, stream=stream)
    return ent


def w4_gumbel_argmax_sample(logits, seed: int, offset: int = 0, workspace=None, stream=None):
    """gumbel_argmax_sample: (sample, argmax), both [M] int64, one pass."""
    _, smp, amx = w4_sample_logits(logits, seed, offset, entropy=False, sample=True,
                                   argmax=True, workspace=workspace, stream=stream)
    return smp, amx
