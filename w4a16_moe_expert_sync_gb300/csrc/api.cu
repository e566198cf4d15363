// api.cu -- the extern "C" entry points declared in include/w4moe.h: argument
// validation on the host, then kernel launches on the caller's stream.  No
// device allocation, no synchronisation, no device-to-host reads.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "../../include/w4moe.h"
#include "launch.h"

namespace w4 {
PipelineTestHooks &pipeline_test_hooks()
{
    thread_local PipelineTestHooks hooks;
    return hooks;
}
}  // namespace w4

namespace {

thread_local char g_detail[512] = "";

int fail(int status, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
    va_end(ap);
    return status;
}

int cuda_fail(cudaError_t err, const char *what)
{
    return fail(W4_ERR_CUDA, "%s: %s", what, cudaGetErrorString(err));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

cudaStream_t as_stream(w4_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// The cubin targets sm_103a only; refuse anything else up front.
int check_device()
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return cuda_fail(err, "cudaGetDevice");
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
        return fail(W4_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a",
                    dev, major, minor);
    return W4_OK;
}

bool valid_block_m(int bm) { return bm == 16 || bm == 32 || bm == 64 || bm == 128 || bm == 256; }

int64_t align_capacity(int M, int k, int E, int bm)
{
    const int64_t A = static_cast<int64_t>(M) * k;
    const int64_t cap = A + static_cast<int64_t>(E) * (bm - 1);
    return (cap + bm - 1) / bm * bm;
}

// Shared checks for the two grouped GEMMs.
int check_gemm_common(int M, int d, int m, int E, int k, int block_m, const void *act,
                      const void *q, const void *s, const void *z, const void *sorted_ids,
                      const void *offsets, const void *out)
{
    if (!act || !q || !s || !z || !sorted_ids || !offsets || !out)
        return fail(W4_ERR_INVALID_ARG, "NULL pointer argument");
    if (M < 0 || d <= 0 || m <= 0 || E <= 0 || k <= 0)
        return fail(W4_ERR_INVALID_ARG, "sizes must be positive (M >= 0)");
    if (!valid_block_m(block_m))
        return fail(W4_ERR_INVALID_ARG, "block_m must be 16, 32, 64, 128 or 256 (got %d)", block_m);
    if (d % 128 || m % 64)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "need d %% 128 == 0 and m %% 64 == 0 (d=%d, m=%d)", d,
                    m);
    if (d > 8192 || m > 1024)
        return fail(W4_ERR_UNSUPPORTED_SHAPE,
                    "need d <= 8192 and m <= 1024: the group sums of xg and h fill at most one "
                    "64-column block (d=%d, m=%d)", d, m);
    if (E > 1024 || k > E)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "need k <= E <= 1024");
    const int64_t A = static_cast<int64_t>(M) * k;
    if (A > (1ll << 30) || static_cast<int64_t>(E) * 2 * m > (1ll << 30) ||
        static_cast<int64_t>(E) * d > (1ll << 30))
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "problem too large for 32-bit indexing");
    if (!aligned16(act) || !aligned16(q) || !aligned16(s) || !aligned16(z) || !aligned16(out))
        return fail(W4_ERR_MISALIGNED, "activation, weight, scale, zero and output pointers "
                                       "must be 16-byte aligned");
    if (!aligned4(sorted_ids) || !aligned4(offsets))
        return fail(W4_ERR_MISALIGNED, "index arrays must be 4-byte aligned");
    return W4_OK;
}

}  // namespace

int w4::check_device_sm103() { return check_device(); }

int w4::set_error_detail(int status, const char *detail)
{
    return fail(status, "%s", detail);
}

extern "C" {

const char *w4_status_string(int status)
{
    switch (status) {
    case W4_OK: return "W4_OK";
    case W4_ERR_INVALID_ARG: return "W4_ERR_INVALID_ARG";
    case W4_ERR_UNSUPPORTED_SHAPE: return "W4_ERR_UNSUPPORTED_SHAPE";
    case W4_ERR_MISALIGNED: return "W4_ERR_MISALIGNED";
    case W4_ERR_CUDA: return "W4_ERR_CUDA";
    case W4_ERR_NO_DEVICE: return "W4_ERR_NO_DEVICE";
    case W4_ERR_WORKSPACE: return "W4_ERR_WORKSPACE";
    default: return "W4_ERR_UNKNOWN";
    }
}

const char *w4_last_error_detail(void) { return g_detail; }

int w4_abi_version(void) { return W4MOE_ABI_VERSION; }

int w4_quantize(const float *W, int E, int N, int K, int group, uint8_t *q, uint16_t *s,
                uint16_t *z, w4_stream_t stream)
{
    if (!W || !q || !s || !z)
        return fail(W4_ERR_INVALID_ARG, "NULL pointer argument");
    if (E < 0 || N < 0 || K <= 0)
        return fail(W4_ERR_INVALID_ARG, "bad sizes E=%d N=%d K=%d", E, N, K);
    if (group != 64 && group != 128 && group != 256)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "group must be 64, 128 or 256 (got %d)", group);
    if (K % group)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "group %d does not divide K=%d", group, K);
    if (!aligned16(W) || !aligned4(q) || !aligned4(s) || !aligned4(z))
        return fail(W4_ERR_MISALIGNED, "W must be 16-byte aligned, outputs 4-byte aligned");
    if (int rc = check_device())
        return rc;
    const int64_t rows = static_cast<int64_t>(E) * N;
    cudaError_t err = w4::launch_quantize(W, rows, K, group, q, s, z, as_stream(stream));
    return err == cudaSuccess ? W4_OK : cuda_fail(err, "quantize launch");
}

int w4_moe_route(const float *logits, int M, int E, int k, int32_t *topk_ids, float *topk_weights,
                 w4_stream_t stream)
{
    if (!logits || !topk_ids || !topk_weights)
        return fail(W4_ERR_INVALID_ARG, "NULL pointer argument");
    if (M < 0 || E <= 0 || k <= 0)
        return fail(W4_ERR_INVALID_ARG, "bad sizes M=%d E=%d k=%d", M, E, k);
    if (k > 32 || k > E || E > 1024)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "need 1 <= k <= 32, k <= E <= 1024");
    if (!aligned4(logits) || !aligned4(topk_ids) || !aligned4(topk_weights))
        return fail(W4_ERR_MISALIGNED, "pointers must be 4-byte aligned");
    if (int rc = check_device())
        return rc;
    cudaError_t err = w4::launch_route(logits, M, E, k, topk_ids, topk_weights, as_stream(stream));
    return err == cudaSuccess ? W4_OK : cuda_fail(err, "route launch");
}

int64_t w4_moe_align_capacity(int M, int k, int E, int block_m)
{
    if (M < 0 || k <= 0 || E <= 0 || !valid_block_m(block_m))
        return -1;
    return align_capacity(M, k, E, block_m);
}

int w4_moe_align(const int32_t *topk_ids, int M, int k, int E, int block_m, int32_t *sorted_ids,
                 int32_t *block_expert, int32_t *expert_offsets, int32_t *num_padded,
                 int32_t *dev_status, w4_stream_t stream)
{
    if (!sorted_ids || !block_expert || !expert_offsets || !num_padded || (M > 0 && !topk_ids))
        return fail(W4_ERR_INVALID_ARG, "NULL pointer argument");
    if (M < 0 || k <= 0 || E <= 0)
        return fail(W4_ERR_INVALID_ARG, "bad sizes M=%d k=%d E=%d", M, k, E);
    if (!valid_block_m(block_m))
        return fail(W4_ERR_INVALID_ARG, "block_m must be 16, 32, 64, 128 or 256 (got %d)", block_m);
    if (E > 1024)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "E must be <= 1024");
    const int64_t cap = align_capacity(M, k, E, block_m);
    if (cap > (1ll << 30))
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "too many assignments");
    if (int rc = check_device())
        return rc;
    cudaError_t err = w4::launch_align(topk_ids, M, k, E, block_m, cap, sorted_ids, block_expert,
                                       expert_offsets, num_padded, dev_status, as_stream(stream));
    return err == cudaSuccess ? W4_OK : cuda_fail(err, "align launch");
}

int w4_gather_activations(const uint16_t *x, int M, int d, int k, int E, int block_m,
                          const int32_t *sorted_ids, const int32_t *num_padded, uint16_t *xg,
                          int32_t *dev_status, w4_stream_t stream)
{
    if (!xg || !sorted_ids || !num_padded || (M > 0 && !x))
        return fail(W4_ERR_INVALID_ARG, "NULL pointer argument");
    if (M < 0 || d <= 0 || k <= 0 || E <= 0)
        return fail(W4_ERR_INVALID_ARG, "bad sizes M=%d d=%d k=%d E=%d", M, d, k, E);
    if (!valid_block_m(block_m))
        return fail(W4_ERR_INVALID_ARG, "block_m must be 16, 32, 64, 128 or 256 (got %d)", block_m);
    if (d % 128 || d > 8192)
        return fail(W4_ERR_UNSUPPORTED_SHAPE,
                    "d must be a multiple of 128 and at most 8192 (its group sums fill one "
                    "64-column block)");
    if (!aligned16(x) || !aligned16(xg) || !aligned4(sorted_ids) || !aligned4(num_padded))
        return fail(W4_ERR_MISALIGNED, "x and xg must be 16-byte aligned");
    if (int rc = check_device())
        return rc;
    const int64_t cap = align_capacity(M, k, E, block_m);
    cudaError_t err =
        w4::launch_gather(x, M, d, k, cap, sorted_ids, num_padded, xg, dev_status,
                          as_stream(stream));
    return err == cudaSuccess ? W4_OK : cuda_fail(err, "gather launch");
}

int w4_moe_align_gather(const int32_t *topk_ids, const uint16_t *x, int M, int d, int k, int E,
                        int block_m, int32_t *sorted_ids, int32_t *block_expert,
                        int32_t *expert_offsets, int32_t *num_padded, uint16_t *xg,
                        int32_t *dev_status, w4_stream_t stream)
{
    if (!sorted_ids || !block_expert || !expert_offsets || !num_padded || !xg ||
        (M > 0 && (!topk_ids || !x)))
        return fail(W4_ERR_INVALID_ARG, "NULL pointer argument");
    if (M < 0 || d <= 0 || k <= 0 || E <= 0)
        return fail(W4_ERR_INVALID_ARG, "bad sizes M=%d d=%d k=%d E=%d", M, d, k, E);
    if (!valid_block_m(block_m))
        return fail(W4_ERR_INVALID_ARG, "block_m must be 16, 32, 64, 128 or 256 (got %d)", block_m);
    if (E > 1024 || d % 128 || d > 8192)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "need E <= 1024, d %% 128 == 0 and d <= 8192");
    if (!aligned16(x) || !aligned16(xg))
        return fail(W4_ERR_MISALIGNED, "x and xg must be 16-byte aligned");
    const int64_t cap = align_capacity(M, k, E, block_m);
    if (cap > (1ll << 30))
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "too many assignments");
    if (int rc = check_device())
        return rc;
    cudaError_t err;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (w4::align_gather_smem_bytes(M, k, E, sms) <= 200 * 1024) {
        err = w4::launch_align_gather(topk_ids, M, k, E, block_m, cap, sorted_ids, block_expert,
                                      expert_offsets, num_padded, dev_status, x, d, xg, sms,
                                      as_stream(stream));
    } else {   // too many assignments to keep their slots in shared memory
        err = w4::launch_align(topk_ids, M, k, E, block_m, cap, sorted_ids, block_expert,
                               expert_offsets, num_padded, dev_status, as_stream(stream));
        if (err == cudaSuccess)
            err = w4::launch_gather(x, M, d, k, cap, sorted_ids, num_padded, xg, dev_status,
                                    as_stream(stream));
    }
    return err == cudaSuccess ? W4_OK : cuda_fail(err, "align+gather launch");
}

int w4_moe_route_align_gather(const float *logits, const uint16_t *x, int M, int d, int k, int E,
                              int block_m, int32_t *topk_ids, float *topk_weights,
                              int32_t *sorted_ids, int32_t *block_expert,
                              int32_t *expert_offsets, int32_t *num_padded, uint16_t *xg,
                              int32_t *dev_status, w4_stream_t stream)
{
    if (!topk_ids || !topk_weights || (M > 0 && !logits))
        return fail(W4_ERR_INVALID_ARG, "NULL pointer argument");
    if (k > 32 || k > E || E > 1024)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "need 1 <= k <= 32, k <= E <= 1024");
    if (!aligned4(logits) || !aligned4(topk_ids) || !aligned4(topk_weights))
        return fail(W4_ERR_MISALIGNED, "logits, ids and weights must be 4-byte aligned");
    if (!sorted_ids || !block_expert || !expert_offsets || !num_padded || !xg ||
        (M > 0 && !x))
        return fail(W4_ERR_INVALID_ARG, "NULL pointer argument");
    if (M < 0 || d <= 0 || k <= 0 || E <= 0)
        return fail(W4_ERR_INVALID_ARG, "bad sizes M=%d d=%d k=%d E=%d", M, d, k, E);
    if (!valid_block_m(block_m))
        return fail(W4_ERR_INVALID_ARG, "block_m must be 16, 32, 64, 128 or 256 (got %d)", block_m);
    if (d % 128 || d > 8192)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "need d %% 128 == 0 and d <= 8192");
    if (!aligned16(x) || !aligned16(xg))
        return fail(W4_ERR_MISALIGNED, "x and xg must be 16-byte aligned");
    if (int rc = check_device())
        return rc;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (M > 0 && w4::route_align_gather_fits(M, k, E, sms)) {
        const int64_t cap = align_capacity(M, k, E, block_m);
        cudaError_t err = w4::launch_route_align_gather(
            logits, M, k, E, block_m, cap, topk_ids, topk_weights, sorted_ids, block_expert,
            expert_offsets, num_padded, dev_status, x, d, xg, sms, as_stream(stream));
        return err == cudaSuccess ? W4_OK : cuda_fail(err, "route+align+gather launch");
    }
    // larger shapes: the router launch, then the fused alignment and gather
    if (int rc = w4_moe_route(logits, M, E, k, topk_ids, topk_weights, stream))
        return rc;
    return w4_moe_align_gather(topk_ids, x, M, d, k, E, block_m, sorted_ids, block_expert,
                               expert_offsets, num_padded, xg, dev_status, stream);
}

}  // extern "C"

namespace {
// The layer's combine folded into the GEMMs (w4_moe_layer only; comb_cnt
// NULL elsewhere): see GroupedGemmProblem.
struct FoldedCombine {
    const int32_t *topk_ids = nullptr;
    const float *topk_w = nullptr;
    int32_t *cnt = nullptr;
    uint16_t *out = nullptr;
};

int grouped_gemm_gate_up(const uint16_t *xg, int M, int d, int m, int E, int k, int block_m,
                         const uint8_t *gu_q, const uint16_t *gu_s, const uint16_t *gu_z,
                         int group, const int32_t *sorted_ids, const int32_t *expert_offsets,
                         uint16_t *h, int32_t *dev_status, w4_stream_t stream,
                         const FoldedCombine &fc)
{
    if (int rc = check_gemm_common(M, d, m, E, k, block_m, xg, gu_q, gu_s, gu_z, sorted_ids,
                                   expert_offsets, h))
        return rc;
    if (group != 128)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "gate_up group must be 128 (got %d)", group);
    if (int rc = check_device())
        return rc;
    w4::GroupedGemmProblem p{};
    p.gate_up = true;
    p.act = xg;
    p.wq = gu_q;
    p.ws = gu_s;
    p.wz = gu_z;
    p.sorted_ids = sorted_ids;
    p.expert_offsets = expert_offsets;
    p.out = h;
    p.dev_status = dev_status;
    p.M = M;
    p.k = k;
    p.E = E;
    p.K = d;
    p.R = 2 * m;
    p.group = group;
    p.out_cols = m;
    p.cap = align_capacity(M, k, E, block_m);
    p.topk_ids = fc.topk_ids;
    p.comb_cnt = fc.cnt;
    p.comb_out = fc.out;
    p.comb_d = d;
    p.wait_ns = w4::pipeline_test_hooks().wait_ns;
    p.test_withhold_sz = w4::pipeline_test_hooks().withhold_sz;
    if (M == 0)
        return W4_OK;
    const char *why = nullptr;
    cudaError_t err = w4::launch_grouped_gemm(p, as_stream(stream), &why);
    if (why)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "%s", why);
    return err == cudaSuccess ? W4_OK : cuda_fail(err, "gate_up launch");
}

// early_schedule: see GroupedGemmProblem (set only by w4_moe_layer, where the
// alignment is two launches back and gate_up waits for it before triggering)
int grouped_gemm_down(const uint16_t *h, int M, int d, int m, int E, int k, int block_m,
                      const uint8_t *dn_q, const uint16_t *dn_s, const uint16_t *dn_z, int group,
                      const int32_t *sorted_ids, const int32_t *expert_offsets, float *y,
                      int32_t *dev_status, w4_stream_t stream, bool early_schedule,
                      const FoldedCombine &fc)
{
    if (int rc = check_gemm_common(M, d, m, E, k, block_m, h, dn_q, dn_s, dn_z, sorted_ids,
                                   expert_offsets, y))
        return rc;
    if (group != 64)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "down group must be 64 (got %d)", group);
    if (int rc = check_device())
        return rc;
    w4::GroupedGemmProblem p{};
    p.gate_up = false;
    p.act = h;
    p.wq = dn_q;
    p.ws = dn_s;
    p.wz = dn_z;
    p.sorted_ids = sorted_ids;
    p.expert_offsets = expert_offsets;
    p.out = y;
    p.dev_status = dev_status;
    p.M = M;
    p.k = k;
    p.E = E;
    p.K = m;
    p.R = d;
    p.group = group;
    p.out_cols = d;
    p.cap = align_capacity(M, k, E, block_m);
    p.early_schedule = early_schedule;
    p.topk_ids = fc.topk_ids;
    p.topk_w = fc.topk_w;
    p.comb_cnt = fc.cnt;
    p.comb_out = fc.out;
    p.comb_d = d;
    p.wait_ns = w4::pipeline_test_hooks().wait_ns;
    p.test_withhold_sz = w4::pipeline_test_hooks().withhold_sz;
    if (M == 0)
        return W4_OK;
    const char *why = nullptr;
    cudaError_t err = w4::launch_grouped_gemm(p, as_stream(stream), &why);
    if (why)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "%s", why);
    return err == cudaSuccess ? W4_OK : cuda_fail(err, "down launch");
}
}  // namespace

extern "C" {

int w4_grouped_gemm_gate_up(const uint16_t *xg, int M, int d, int m, int E, int k, int block_m,
                            const uint8_t *gu_q, const uint16_t *gu_s, const uint16_t *gu_z,
                            int group, const int32_t *sorted_ids, const int32_t *expert_offsets,
                            uint16_t *h, int32_t *dev_status, w4_stream_t stream)
{
    return grouped_gemm_gate_up(xg, M, d, m, E, k, block_m, gu_q, gu_s, gu_z, group, sorted_ids,
                                expert_offsets, h, dev_status, stream, FoldedCombine{});
}

int w4_grouped_gemm_down(const uint16_t *h, int M, int d, int m, int E, int k, int block_m,
                         const uint8_t *dn_q, const uint16_t *dn_s, const uint16_t *dn_z, int group,
                         const int32_t *sorted_ids, const int32_t *expert_offsets, float *y,
                         int32_t *dev_status, w4_stream_t stream)
{
    return grouped_gemm_down(h, M, d, m, E, k, block_m, dn_q, dn_s, dn_z, group, sorted_ids,
                             expert_offsets, y, dev_status, stream, false, FoldedCombine{});
}

int w4_grouped_gemm_down_combine(const uint16_t *h, int M, int d, int m, int E, int k,
                                 int block_m, const uint8_t *dn_q, const uint16_t *dn_s,
                                 const uint16_t *dn_z, int group, const int32_t *sorted_ids,
                                 const int32_t *expert_offsets, const int32_t *topk_ids,
                                 const float *topk_weights, int32_t *counters, float *y,
                                 uint16_t *out, int32_t *dev_status, w4_stream_t stream)
{
    if (M > 0 && (!topk_ids || !topk_weights || !counters || !out))
        return fail(W4_ERR_INVALID_ARG, "NULL pointer argument");
    if ((reinterpret_cast<uintptr_t>(out) & 7u) || !aligned4(topk_ids) ||
        !aligned4(topk_weights) || !aligned4(counters))
        return fail(W4_ERR_MISALIGNED, "out must be 8-byte and topk_ids, topk_weights and "
                                       "counters 4-byte aligned");
    FoldedCombine fc;
    fc.topk_ids = topk_ids;
    fc.topk_w = topk_weights;
    fc.cnt = counters;
    fc.out = out;
    return grouped_gemm_down(h, M, d, m, E, k, block_m, dn_q, dn_s, dn_z, group, sorted_ids,
                             expert_offsets, y, dev_status, stream, false, fc);
}

int w4_test_pipeline_hooks(uint64_t wait_limit_ns, int withhold_first_scales)
{
    w4::PipelineTestHooks &h = w4::pipeline_test_hooks();
    h.wait_ns = wait_limit_ns ? wait_limit_ns : 1000000000ull;
    h.withhold_sz = withhold_first_scales != 0;
    return W4_OK;
}

int w4_moe_combine_prepare(const int32_t *topk_ids, int M, int k, int E, int d,
                           int32_t *counters, uint16_t *out, w4_stream_t stream)
{
    if (M > 0 && (!topk_ids || !counters || !out))
        return fail(W4_ERR_INVALID_ARG, "NULL pointer argument");
    if (M < 0 || k <= 0 || d <= 0 || E <= 0)
        return fail(W4_ERR_INVALID_ARG, "bad sizes M=%d k=%d d=%d E=%d", M, k, d, E);
    if (d % 128)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "d must be a multiple of 128 (got %d)", d);
    if (static_cast<int64_t>(M) * k >= (1ll << 31) || static_cast<int64_t>(M) * d >= (1ll << 31))
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "M * k and M * d must be below 2^31");
    if ((reinterpret_cast<uintptr_t>(out) & 7u) || !aligned4(topk_ids) || !aligned4(counters))
        return fail(W4_ERR_MISALIGNED, "out must be 8-byte and topk_ids and counters 4-byte "
                                       "aligned");
    if (M == 0)
        return W4_OK;
    if (int rc = check_device())
        return rc;
    cudaError_t err = w4::launch_combine_prepare(topk_ids, M, k, E, d, counters, out,
                                                 as_stream(stream));
    return err == cudaSuccess ? W4_OK : cuda_fail(err, "combine prepare launch");
}

int w4_moe_combine_fixed_order(const float *y, const int32_t *topk_ids, const float *topk_weights,
                               int M, int k, int d, int E, uint16_t *out, w4_stream_t stream)
{
    if (!out || (M > 0 && (!y || !topk_ids || !topk_weights)))
        return fail(W4_ERR_INVALID_ARG, "NULL pointer argument");
    if (M < 0 || k <= 0 || d <= 0 || E <= 0)
        return fail(W4_ERR_INVALID_ARG, "bad sizes M=%d k=%d d=%d E=%d", M, k, d, E);
    if (d % 4)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "d must be a multiple of 4");
    if (!aligned16(y) || (reinterpret_cast<uintptr_t>(out) & 7u))
        return fail(W4_ERR_MISALIGNED, "y must be 16-byte and out 8-byte aligned");
    if (int rc = check_device())
        return rc;
    cudaError_t err =
        w4::launch_combine(y, topk_ids, topk_weights, M, k, d, E, out, as_stream(stream));
    return err == cudaSuccess ? W4_OK : cuda_fail(err, "combine launch");
}

}  // extern "C"

// Workspace layout of w4_moe_layer (each piece 256-byte aligned):
//   sorted_ids [cap] i32 | block_expert [cap/bm] i32 | expert_offsets [E+1] i32 |
//   num_padded [1] i32 | xg [cap, d + 64] fp16 | h [cap, m + 64] fp16 |
//   y [M*k, d] fp32
//   (xg and h rows end in their 64-column group-sum block)
namespace {
struct LayerWs {
    size_t sorted, block, offs, npad, xg, h, y, total;
};
size_t up256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }
LayerWs layer_ws(int M, int d, int m, int E, int k, int bm)
{
    const size_t cap = static_cast<size_t>(align_capacity(M, k, E, bm));
    LayerWs w;
    w.sorted = 0;
    w.block = up256(w.sorted + 4 * cap);
    w.offs = up256(w.block + 4 * (cap / bm));
    w.npad = up256(w.offs + 4 * (static_cast<size_t>(E) + 1));
    w.xg = up256(w.npad + 4);
    w.h = up256(w.xg + 2 * cap * (static_cast<size_t>(d) + 64));
    w.y = up256(w.h + 2 * cap * (static_cast<size_t>(m) + 64));
    w.total = up256(w.y + 4 * static_cast<size_t>(M) * k * d);
    return w;
}

// The checks of the layer's GEMM and combine arguments, made before its
// first launch (the workspace pieces stand in for the intermediates).
int check_layer(int M, int d, int m, int E, int k, int block_m, const uint8_t *gu_q,
                const uint16_t *gu_s, const uint16_t *gu_z, int gu_group, const uint8_t *dn_q,
                const uint16_t *dn_s, const uint16_t *dn_z, int dn_group, const uint8_t *ws,
                const LayerWs &L, const float *topk_weights, const uint16_t *out)
{
    if (int rc = check_gemm_common(M, d, m, E, k, block_m, ws + L.xg, gu_q, gu_s, gu_z,
                                   ws + L.sorted, ws + L.offs, ws + L.h))
        return rc;
    if (int rc = check_gemm_common(M, d, m, E, k, block_m, ws + L.h, dn_q, dn_s, dn_z,
                                   ws + L.sorted, ws + L.offs, ws + L.y))
        return rc;
    if (gu_group != 128 || dn_group != 64)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "need gate_up group 128 and down group 64 (got %d, %d)",
                    gu_group, dn_group);
    if (int rc = check_device())
        return rc;
    if (!w4::grouped_gemm_fits(true, d, gu_group, E) || !w4::grouped_gemm_fits(false, m, dn_group, E))
        return fail(W4_ERR_UNSUPPORTED_SHAPE,
                    "the grouped GEMMs' scale/zero stages do not fit shared memory (d=%d, m=%d, "
                    "E=%d; gate_up takes d up to about 3584 at E = 128)", d, m, E);
    if (M > 0 && (!out || !topk_weights))
        return fail(W4_ERR_INVALID_ARG, "NULL pointer argument");
    if ((reinterpret_cast<uintptr_t>(out) & 7u) || !aligned4(topk_weights))
        return fail(W4_ERR_MISALIGNED, "out must be 8-byte and topk_weights 4-byte aligned");
    return W4_OK;
}

// gate_up (which also sets the combine counters) and down with the combine
// folded into its epilogue: the layer's launches after alignment+gather
int layer_gemms(const int32_t *topk_ids, const float *topk_weights, int M,
                int d, int m, int E, int k, int block_m, const uint8_t *gu_q,
                const uint16_t *gu_s, const uint16_t *gu_z, int gu_group, const uint8_t *dn_q,
                const uint16_t *dn_s, const uint16_t *dn_z, int dn_group, uint8_t *ws,
                const LayerWs &L, uint16_t *out, int32_t *dev_status, w4_stream_t stream)
{
    const int32_t *sorted = reinterpret_cast<const int32_t *>(ws + L.sorted);
    const int32_t *offs = reinterpret_cast<const int32_t *>(ws + L.offs);
    const uint16_t *xg = reinterpret_cast<const uint16_t *>(ws + L.xg);
    uint16_t *h = reinterpret_cast<uint16_t *>(ws + L.h);
    float *y = reinterpret_cast<float *>(ws + L.y);
    // The combine runs as its own launch: folded into the down GEMM
    // (w4_grouped_gemm_down_combine) the completed tokens gather on the CTAs
    // that finish last and their y reads (23 MB at M = 256, d = 2816, top-8)
    // run in those CTAs' tails, which measured ~13 us slower per layer than
    // the standalone fixed-order combine, which reads the same bytes with the
    // whole GPU and overlaps its start with the down GEMM's end.
    int rc = grouped_gemm_gate_up(xg, M, d, m, E, k, block_m, gu_q, gu_s, gu_z, gu_group, sorted,
                                  offs, h, dev_status, stream, FoldedCombine{});
    if (rc)
        return rc;
    rc = grouped_gemm_down(h, M, d, m, E, k, block_m, dn_q, dn_s, dn_z, dn_group, sorted, offs, y,
                           dev_status, stream, true, FoldedCombine{});
    if (rc)
        return rc;
    cudaError_t err = w4::launch_combine(y, topk_ids, topk_weights, M, k, d, E, out,
                                         as_stream(stream));
    return err == cudaSuccess ? W4_OK : cuda_fail(err, "combine launch");
}
}  // namespace

extern "C" {

size_t w4_moe_layer_workspace_size(int M, int d, int m, int E, int k, int block_m)
{
    if (M < 0 || d <= 0 || m <= 0 || E <= 0 || k <= 0 || !valid_block_m(block_m))
        return 0;
    return layer_ws(M, d, m, E, k, block_m).total;
}

int w4_moe_layer(const uint16_t *x, const int32_t *topk_ids, const float *topk_weights, int M,
                 int d, int m, int E, int k, int block_m, const uint8_t *gu_q,
                 const uint16_t *gu_s, const uint16_t *gu_z, int gu_group, const uint8_t *dn_q,
                 const uint16_t *dn_s, const uint16_t *dn_z, int dn_group, void *workspace,
                 size_t workspace_bytes, uint16_t *out, int32_t *dev_status, w4_stream_t stream)
{
    if (!valid_block_m(block_m))
        return fail(W4_ERR_INVALID_ARG, "block_m must be 16, 32, 64, 128 or 256 (got %d)", block_m);
    if (M < 0 || d <= 0 || m <= 0 || E <= 0 || k <= 0)
        return fail(W4_ERR_INVALID_ARG, "bad sizes");
    const LayerWs L = layer_ws(M, d, m, E, k, block_m);
    if (!workspace || workspace_bytes < L.total)
        return fail(W4_ERR_WORKSPACE, "workspace needs %zu bytes", L.total);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(W4_ERR_MISALIGNED, "workspace must be 256-byte aligned");
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if (int rc = check_layer(M, d, m, E, k, block_m, gu_q, gu_s, gu_z, gu_group, dn_q, dn_s, dn_z,
                             dn_group, ws, L, topk_weights, out))
        return rc;
    int32_t *sorted = reinterpret_cast<int32_t *>(ws + L.sorted);
    int32_t *block = reinterpret_cast<int32_t *>(ws + L.block);
    int32_t *offs = reinterpret_cast<int32_t *>(ws + L.offs);
    int32_t *npad = reinterpret_cast<int32_t *>(ws + L.npad);
    uint16_t *xg = reinterpret_cast<uint16_t *>(ws + L.xg);
    // alignment and the activation gather share one launch
    if (int rc0 = w4_moe_align_gather(topk_ids, x, M, d, k, E, block_m, sorted, block, offs, npad,
                                      xg, dev_status, stream))
        return rc0;
    if (M == 0)
        return W4_OK;
    return layer_gemms(topk_ids, topk_weights, M, d, m, E, k, block_m, gu_q, gu_s, gu_z,
                       gu_group, dn_q, dn_s, dn_z, dn_group, ws, L, out, dev_status, stream);
}

// Staging buffers of w4_moe_layer_host after the layer's workspace.
struct HostStaging {
    size_t x, ids, w, out, total;
};

static HostStaging host_staging(size_t base, int M, int d, int k)
{
    auto up = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
    HostStaging h;
    h.x = up(base);
    h.ids = up(h.x + 2 * static_cast<size_t>(M) * d);
    h.w = up(h.ids + 4 * static_cast<size_t>(M) * k);
    h.out = up(h.w + 4 * static_cast<size_t>(M) * k);
    h.total = up(h.out + 2 * static_cast<size_t>(M) * d);
    return h;
}

size_t w4_moe_layer_host_workspace_size(int M, int d, int m, int E, int k, int block_m)
{
    if (M < 0 || d <= 0 || m <= 0 || E <= 0 || k <= 0 || !valid_block_m(block_m))
        return 0;
    return host_staging(layer_ws(M, d, m, E, k, block_m).total, M, d, k).total;
}

int w4_moe_layer_host(const uint16_t *x_host, const int32_t *topk_ids_host,
                      const float *topk_weights_host, int M, int d, int m, int E, int k,
                      int block_m, const uint8_t *gu_q, const uint16_t *gu_s,
                      const uint16_t *gu_z, int gu_group, const uint8_t *dn_q,
                      const uint16_t *dn_s, const uint16_t *dn_z, int dn_group, void *workspace,
                      size_t workspace_bytes, uint16_t *out_host, int32_t *dev_status,
                      w4_stream_t stream)
{
    if (!valid_block_m(block_m))
        return fail(W4_ERR_INVALID_ARG, "block_m must be 16, 32, 64, 128 or 256 (got %d)", block_m);
    if (M < 0 || d <= 0 || m <= 0 || E <= 0 || k <= 0)
        return fail(W4_ERR_INVALID_ARG, "bad sizes");
    if (M > 0 && (!x_host || !topk_ids_host || !topk_weights_host || !out_host))
        return fail(W4_ERR_INVALID_ARG, "NULL host buffer");
    const LayerWs L = layer_ws(M, d, m, E, k, block_m);
    const HostStaging H = host_staging(L.total, M, d, k);
    if (!workspace || workspace_bytes < H.total)
        return fail(W4_ERR_WORKSPACE, "workspace needs %zu bytes", H.total);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(W4_ERR_MISALIGNED, "workspace must be 256-byte aligned");
    if (M == 0)   // no rows to copy or compute
        return W4_OK;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint16_t *x_d = reinterpret_cast<uint16_t *>(ws + H.x);
    int32_t *ids_d = reinterpret_cast<int32_t *>(ws + H.ids);
    float *w_d = reinterpret_cast<float *>(ws + H.w);
    uint16_t *out_d = reinterpret_cast<uint16_t *>(ws + H.out);
    const cudaStream_t s = as_stream(stream);
    const size_t nx = 2 * static_cast<size_t>(M) * d, nk = 4 * static_cast<size_t>(M) * k;
    cudaError_t err = cudaMemcpyAsync(x_d, x_host, nx, cudaMemcpyHostToDevice, s);
    if (err == cudaSuccess)
        err = cudaMemcpyAsync(ids_d, topk_ids_host, nk, cudaMemcpyHostToDevice, s);
    if (err == cudaSuccess)
        err = cudaMemcpyAsync(w_d, topk_weights_host, nk, cudaMemcpyHostToDevice, s);
    if (err != cudaSuccess)
        return fail(W4_ERR_CUDA, "host-to-device copy: %s", cudaGetErrorString(err));
    if (int rc = w4_moe_layer(x_d, ids_d, w_d, M, d, m, E, k, block_m, gu_q, gu_s, gu_z, gu_group,
                              dn_q, dn_s, dn_z, dn_group, workspace, L.total, out_d, dev_status,
                              stream))
        return rc;
    err = cudaMemcpyAsync(out_host, out_d, nx, cudaMemcpyDeviceToHost, s);
    if (err != cudaSuccess)
        return fail(W4_ERR_CUDA, "device-to-host copy: %s", cudaGetErrorString(err));
    return W4_OK;
}

int w4_moe_layer_from_logits(const uint16_t *x, const float *logits, int M, int d, int m, int E,
                             int k, int block_m, const uint8_t *gu_q, const uint16_t *gu_s,
                             const uint16_t *gu_z, int gu_group, const uint8_t *dn_q,
                             const uint16_t *dn_s, const uint16_t *dn_z, int dn_group,
                             void *workspace, size_t workspace_bytes, int32_t *topk_ids,
                             float *topk_weights, uint16_t *out, int32_t *dev_status,
                             w4_stream_t stream)
{
    if (!valid_block_m(block_m))
        return fail(W4_ERR_INVALID_ARG, "block_m must be 16, 32, 64, 128 or 256 (got %d)", block_m);
    if (M < 0 || d <= 0 || m <= 0 || E <= 0 || k <= 0)
        return fail(W4_ERR_INVALID_ARG, "bad sizes");
    const LayerWs L = layer_ws(M, d, m, E, k, block_m);
    if (!workspace || workspace_bytes < L.total)
        return fail(W4_ERR_WORKSPACE, "workspace needs %zu bytes", L.total);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(W4_ERR_MISALIGNED, "workspace must be 256-byte aligned");
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if (int rc = check_layer(M, d, m, E, k, block_m, gu_q, gu_s, gu_z, gu_group, dn_q, dn_s, dn_z,
                             dn_group, ws, L, topk_weights, out))
        return rc;
    int32_t *sorted = reinterpret_cast<int32_t *>(ws + L.sorted);
    int32_t *block = reinterpret_cast<int32_t *>(ws + L.block);
    int32_t *offs = reinterpret_cast<int32_t *>(ws + L.offs);
    int32_t *npad = reinterpret_cast<int32_t *>(ws + L.npad);
    uint16_t *xg = reinterpret_cast<uint16_t *>(ws + L.xg);
    // router, alignment and activation gather share one launch
    if (int rc0 = w4_moe_route_align_gather(logits, x, M, d, k, E, block_m, topk_ids,
                                            topk_weights, sorted, block, offs, npad, xg,
                                            dev_status, stream))
        return rc0;
    if (M == 0)
        return W4_OK;
    return layer_gemms(topk_ids, topk_weights, M, d, m, E, k, block_m, gu_q, gu_s, gu_z,
                       gu_group, dn_q, dn_s, dn_z, dn_group, ws, L, out, dev_status, stream);
}

}  // extern "C"

// ------------------------------------------------------------------ RMSNorm
int w4_rmsnorm(const uint16_t *x, const uint16_t *weight, int M, int d, float eps, uint16_t *y,
               w4_stream_t stream)
{
    if (!weight || (M > 0 && (!x || !y)))
        return fail(W4_ERR_INVALID_ARG, "NULL pointer argument");
    if (M < 0 || d <= 0 || !(eps >= 0.0f))
        return fail(W4_ERR_INVALID_ARG, "bad sizes or eps (M=%d d=%d)", M, d);
    if (d % 8)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "d must be a multiple of 8 (got %d)", d);
    if (static_cast<int64_t>(M) * d >= (1ll << 31))
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "M * d must be below 2^31");
    if (!aligned16(x) || !aligned16(weight) || !aligned16(y))
        return fail(W4_ERR_MISALIGNED, "x, weight and y must be 16-byte aligned");
    if (M == 0)
        return W4_OK;
    if (int rc = check_device())
        return rc;
    cudaError_t err = w4::launch_rmsnorm(x, weight, M, d, eps, y, as_stream(stream));
    return err == cudaSuccess ? W4_OK : cuda_fail(err, "rmsnorm launch");
}

// ------------------------------------------------------------------ sampler
size_t w4_sample_logits_workspace_size(int M, int64_t V)
{
    if (M <= 0 || V <= 0 || V >= (1ll << 31))
        return 0;
    return w4::sampler_workspace_bytes(M, V);
}

int w4_sample_logits(const float *logits, int M, int64_t V, uint64_t seed, uint64_t offset,
                     float *entropy, int64_t *sample, int64_t *argmax, void *workspace,
                     size_t workspace_bytes, w4_stream_t stream)
{
    if (M < 0 || V <= 0 || V >= (1ll << 31))
        return fail(W4_ERR_INVALID_ARG, "need M >= 0 and 0 < V < 2^31 (M=%d V=%lld)", M,
                    static_cast<long long>(V));
    if (M == 0)
        return W4_OK;
    if (!logits)
        return fail(W4_ERR_INVALID_ARG, "NULL logits");
    if (!entropy && !sample && !argmax)
        return fail(W4_ERR_INVALID_ARG, "no output requested");
    if (!aligned4(logits))
        return fail(W4_ERR_MISALIGNED, "logits must be 4-byte aligned");
    if (!workspace || workspace_bytes < w4::sampler_workspace_bytes(M, V) || !aligned16(workspace))
        return fail(W4_ERR_WORKSPACE, "workspace must be 16-byte aligned and hold %zu bytes",
                    w4::sampler_workspace_bytes(M, V));
    if (int rc = check_device())
        return rc;
    cudaError_t err = w4::launch_sampler(logits, M, V, seed, offset, entropy, sample, argmax,
                                         workspace, as_stream(stream));
    return err == cudaSuccess ? W4_OK : cuda_fail(err, "sampler launch");
}

int w4_fused_entropy(const float *logits, int M, int64_t V, float *entropy, void *workspace,
                     size_t workspace_bytes, w4_stream_t stream)
{
    if (!entropy)
        return fail(W4_ERR_INVALID_ARG, "NULL entropy");
    return w4_sample_logits(logits, M, V, 0, 0, entropy, nullptr, nullptr, workspace,
                            workspace_bytes, stream);
}

int w4_gumbel_argmax_sample(const float *logits, int M, int64_t V, uint64_t seed,
                            uint64_t offset, int64_t *sample, int64_t *argmax, void *workspace,
                            size_t workspace_bytes, w4_stream_t stream)
{
    if (!sample)
        return fail(W4_ERR_INVALID_ARG, "NULL sample");
    return w4_sample_logits(logits, M, V, seed, offset, nullptr, sample, argmax, workspace,
                            workspace_bytes, stream);
}

// ----------------------------------------------------------- dense linear
// Workspace of w4_w4a16_linear (each piece 256-byte aligned):
//   sorted_ids [padded] i32 | offsets [2] i32 | xg [padded, K] fp16 |
//   partial sums [splits, M, N] fp32 (dense kernel with a split contraction)
// with padded = M rounded up to 16 (the one expert's slots).
namespace {
constexpr int kLinearBlockM = 16;
struct LinearWs {
    size_t sorted, offs, xg, part, total;
    int padded;
};
LinearWs linear_ws(int M, int K, int N, int group)
{
    LinearWs w;
    w.padded = (M + kLinearBlockM - 1) / kLinearBlockM * kLinearBlockM;
    w.sorted = 0;
    w.offs = up256(4 * static_cast<size_t>(w.padded));
    w.xg = up256(w.offs + 8);
    w.part = up256(w.xg + 2 * static_cast<size_t>(w.padded) * K);
    const bool split = M > 0 && w4::dense_gemm_supported(M, N, K, group);
    w.total = up256(w.part + (split ? w4::dense_gemm_partial_bytes(M, N, K) : 0));
    return w;
}
}  // namespace

size_t w4_w4a16_linear_workspace_size(int M, int K, int N, int group)
{
    if (M < 0 || K <= 0 || N <= 0)
        return 0;
    return linear_ws(M, K, N, group).total;
}

int w4_w4a16_linear(const uint16_t *x, int M, int K, int N, const uint8_t *q, const uint16_t *s,
                    const uint16_t *z, int group, void *workspace, size_t workspace_bytes,
                    uint16_t *y, int32_t *dev_status, w4_stream_t stream)
{
    if (M < 0 || K <= 0 || N <= 0)
        return fail(W4_ERR_INVALID_ARG, "bad sizes M=%d K=%d N=%d", M, K, N);
    if (M == 0)
        return W4_OK;
    if (!x || !q || !s || !z || !y)
        return fail(W4_ERR_INVALID_ARG, "NULL pointer argument");
    if (group != 64 && group != 128)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "group must be 64 or 128 (got %d)", group);
    if (K % group || K % 64 || K < 256 || N % 128 || K / group > 32)
        return fail(W4_ERR_UNSUPPORTED_SHAPE,
                    "need K >= 256, a multiple of the group and of 64, with at most 32 groups, "
                    "N a multiple of 128 (K=%d N=%d group=%d)", K, N, group);
    if (static_cast<int64_t>(M) * K > (1ll << 30) || static_cast<int64_t>(M) * N > (1ll << 30) ||
        static_cast<int64_t>(N) * K > (1ll << 31))
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "problem too large for 32-bit indexing");
    if (!aligned16(x) || !aligned16(q) || !aligned16(s) || !aligned16(z) || !aligned16(y))
        return fail(W4_ERR_MISALIGNED, "x, q, s, z and y must be 16-byte aligned");
    const LinearWs L = linear_ws(M, K, N, group);
    if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(W4_ERR_WORKSPACE, "workspace must be 256-byte aligned and hold %zu bytes",
                    L.total);
    if (int rc = check_device())
        return rc;
    char *ws = static_cast<char *>(workspace);
    int32_t *sorted = reinterpret_cast<int32_t *>(ws + L.sorted);
    int32_t *offs = reinterpret_cast<int32_t *>(ws + L.offs);
    uint16_t *xg = reinterpret_cast<uint16_t *>(ws + L.xg);
    // every token in the one "expert" that is the whole matrix, one slot each
    cudaError_t err = w4::launch_identity_align_gather(x, M, K, L.padded, sorted, offs, xg,
                                                       as_stream(stream));
    if (err != cudaSuccess)
        return cuda_fail(err, "identity alignment launch");
    w4::DenseGemmProblem d{};
    d.xg = xg;
    d.q = q;
    d.s = s;
    d.z = z;
    d.y = y;
    d.partials = reinterpret_cast<float *>(ws + L.part);
    d.dev_status = dev_status;
    d.M = M;
    d.N = N;
    d.K = K;
    d.group = group;
    const char *why = nullptr;
    err = w4::launch_dense_gemm(d, as_stream(stream), &why);
    if (why)
        return fail(W4_ERR_UNSUPPORTED_SHAPE, "%s", why);
    return err == cudaSuccess ? W4_OK : cuda_fail(err, "dense GEMM launch");
}
