"""Runs the layer, the two GEMMs and the folded combine with the library
given on the command line (the W4_CHECK_BOUNDS build) and saves the
outputs and device status words to an .npz: a child process of
test_gpu_check_bounds.py, which loads the normal build in its own process."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def run(lib_path, names, out_path):
    import torch
    import w4a16_moe_expert_sync_gb300 as w4
    w4.load_library(lib_path)
    from helpers import gpu_inputs, gpu_weights
    res = {}
    for name in names:
        cfg, x, lg, _, _ = gpu_inputs(name)
        gu, dn = gpu_weights(name)
        st = torch.zeros(4, dtype=torch.int32, device="cuda")
        ids, w = w4.w4_moe_route(lg, cfg.k)
        out = w4.w4_moe_layer(x, ids, w, gu, dn, dev_status=st[0:1])
        al, xg = w4.w4_moe_align_gather(ids, x, cfg.E, 16, dev_status=st[1:2])
        h = w4.w4_grouped_gemm_gate_up(xg, *gu, al, dev_status=st[1:2])
        y = w4.w4_grouped_gemm_down(h, *dn, al, dev_status=st[2:3])
        counters, out2 = w4.w4_moe_combine_prepare(ids, cfg.E, cfg.d)
        _, out2 = w4.w4_grouped_gemm_down_combine(h, *dn, al, ids, w, counters, out2,
                                                  dev_status=st[3:4])
        torch.cuda.synchronize()
        res[f"{name}_out"] = out.view(torch.int16).cpu().numpy()
        res[f"{name}_out2"] = out2.view(torch.int16).cpu().numpy()
        res[f"{name}_status"] = st.cpu().numpy()
    np.savez(out_path, **res)


if __name__ == "__main__":
    run(sys.argv[1], sys.argv[3:], sys.argv[2])
