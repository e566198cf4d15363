"""w4_moe_layer_static_scratch: the layer with its intermediates in the
library's static device array instead of a caller workspace.  Through the C
ABI it must give the same bytes as w4_moe_layer, on two calls in a row, and
refuse shapes whose scratch does not fit.  (A library convenience with no
counterpart in the pages.)  Collected last so that it runs both after the
other tests and alone in a fresh process."""
import pytest

from helpers import gpu_inputs, gpu_weights
from w4a16_moe_expert_sync_gb300 import workloads as wl

W4_ERR_WORKSPACE = 6
STATIC_SCRATCH_BYTES = 64 << 20


def test_static_scratch_rejects_oversized_shape(lib):
    """A shape whose workspace exceeds the static array is refused before any
    launch, so this needs no GPU."""
    cfg = wl.CONFIGS["canvas2048"]
    need = lib.w4_moe_layer_workspace_size(cfg.M, cfg.d, cfg.m, cfg.E, cfg.k, 16)
    assert need > STATIC_SCRATCH_BYTES
    raw = lib.load_library()
    rc = raw.w4_moe_layer_static_scratch(None, None, None, cfg.M, cfg.d, cfg.m, cfg.E, cfg.k, 16,
                                         None, None, None, 128, None, None, None, 64, None, None,
                                         None)
    assert rc == W4_ERR_WORKSPACE
    detail = raw.w4_last_error_detail().decode()
    assert str(need) in detail and str(STATIC_SCRATCH_BYTES) in detail


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["layer256", "ragged", "tiny"])
def test_static_scratch_matches_workspace_layer(lib, name):
    import torch
    cfg, x, lg, _, _ = gpu_inputs(name)
    assert lib.w4_moe_layer_workspace_size(cfg.M, cfg.d, cfg.m, cfg.E, cfg.k, 16) \
        <= STATIC_SCRATCH_BYTES
    gu, dn = gpu_weights(name)
    ids, w = lib.w4_moe_route(lg, cfg.k)
    want = lib.w4_moe_layer(x, ids, w, gu, dn)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full((cfg.M, cfg.d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lib.w4_moe_layer_static_scratch(x, ids, w, gu, dn, out, dev_status=status)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), want.view(torch.int16)), f"call {call}"
    assert int(status.item()) == 0
