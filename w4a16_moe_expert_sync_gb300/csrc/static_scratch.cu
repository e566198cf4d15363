// static_scratch.cu -- w4_moe_layer_static_scratch: the whole routed-expert
// layer with its intermediates in a fixed device array owned by this library,
// for callers that cannot allocate device memory at call time.
//
// Who needs it: a caller with no device allocator of its own (a plain C host
// that links only this library), or one that must not allocate once it is
// serving (a fixed memory budget reserved at start-up, or code that runs
// inside an allocator's own callback, where re-entering that allocator, or
// calling cudaMalloc/cudaFree, which synchronise the device, is not allowed).
// This entry point takes no workspace argument and allocates nothing: no
// cudaMalloc, no cudaFree, no allocating library routine.
//
// The array is shared by every call in the process on a given device, so
// calls whose GPU work overlaps (two streams, or two host threads with
// different streams) race on it; issue them on one stream, one after another.
#include <cstdio>

#include "../../include/w4moe.h"
#include "launch.h"

namespace {

// The layer's intermediates: alignment outputs, gathered activations, h and y
// (the same layout w4_moe_layer uses for its caller-provided workspace).
// Nothing in it needs to start at zero: each call writes every byte it reads
// before reading it.
__device__ __align__(256) unsigned char g_layer_scratch[W4_STATIC_SCRATCH_BYTES];

// Device address of g_layer_scratch on the current device.  It is looked up
// on every call (a host-side table lookup once the module is loaded), so an
// address never outlives the context it belongs to: after cudaDeviceReset
// the next call finds the array in the new context.  The first lookup on a
// device may load this library's module onto it.
int scratch_address(void **out)
{
    void *p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_layer_scratch);
    if (err != cudaSuccess || !p) {
        (void)cudaGetLastError();   // leave no pending error for later launches to report
        return w4::set_error_detail(W4_ERR_CUDA,
                                    "cudaGetSymbolAddress(static layer scratch) failed");
    }
    *out = p;
    return W4_OK;
}

}  // namespace

extern "C" int w4_moe_layer_static_scratch(
    const uint16_t *x, const int32_t *topk_ids, const float *topk_weights, int M, int d, int m,
    int E, int k, int block_m, const uint8_t *gu_q, const uint16_t *gu_s, const uint16_t *gu_z,
    int gu_group, const uint8_t *dn_q, const uint16_t *dn_s, const uint16_t *dn_z, int dn_group,
    uint16_t *out, int32_t *dev_status, w4_stream_t stream)
{
    const size_t need = w4_moe_layer_workspace_size(M, d, m, E, k, block_m);
    if (need == 0)
        return w4::set_error_detail(W4_ERR_INVALID_ARG, "bad sizes or block_m");
    if (need > static_cast<size_t>(W4_STATIC_SCRATCH_BYTES)) {
        char msg[160];
        snprintf(msg, sizeof(msg),
                 "this shape needs %zu bytes of scratch; the static scratch holds %zu "
                 "(use w4_moe_layer with a workspace instead)",
                 need, static_cast<size_t>(W4_STATIC_SCRATCH_BYTES));
        return w4::set_error_detail(W4_ERR_WORKSPACE, msg);
    }
    if (int rc = w4::check_device_sm103())   // before the lookup: a wrong device is not a CUDA error
        return rc;
    void *scratch = nullptr;
    if (int rc = scratch_address(&scratch))
        return rc;
    return w4_moe_layer(x, topk_ids, topk_weights, M, d, m, E, k, block_m, gu_q, gu_s, gu_z,
                        gu_group, dn_q, dn_s, dn_z, dn_group, scratch,
                        static_cast<size_t>(W4_STATIC_SCRATCH_BYTES), out, dev_status, stream);
}
