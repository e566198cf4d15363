// launch.h -- internal launchers shared between the kernel translation units
// and the C-ABI layer (api.cu).  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace w4 {

// Device status bits (mirrors include/w4moe.h).
constexpr int32_t kDevBadExpertId = 0x1;
constexpr int32_t kDevPipelineTimeout = 0x2;
constexpr int32_t kDevTooManyJobs = 0x4;
constexpr int32_t kDevFp16Range = 0x8;
// kDevOutOfBounds = 0x10 (checks.cuh): a store failed its range check
// (only in the W4_CHECK_BOUNDS build)

cudaError_t launch_quantize(const float *W, int64_t rows, int K, int group, uint8_t *q,
                            uint16_t *s, uint16_t *z, cudaStream_t stream);

cudaError_t launch_route(const float *logits, int M, int E, int k, int32_t *ids, float *w,
                         cudaStream_t stream);

__host__ __device__ size_t align_smem_bytes(int E, int nw);
cudaError_t launch_align(const int32_t *ids, int M, int k, int E, int block_m, int64_t cap,
                         int32_t *sorted_ids, int32_t *block_expert, int32_t *offsets,
                         int32_t *num_padded, int32_t *dev_status, cudaStream_t stream);

// xg[slot] = x[sorted_ids[slot] / k] in fp16 block order (zero for padding)
// for slots below *num_padded.
cudaError_t launch_gather(const uint16_t *x, int M, int d, int k, int64_t cap,
                          const int32_t *sorted_ids, const int32_t *num_padded, uint16_t *xg,
                          int32_t *dev_status, cudaStream_t stream);

// Alignment and gather in one launch (every CTA aligns in shared memory).
size_t align_gather_smem_bytes(int M, int k, int E, int num_sms);
cudaError_t launch_align_gather(const int32_t *ids, int M, int k, int E, int block_m, int64_t cap,
                                int32_t *sorted_ids, int32_t *block_expert, int32_t *offsets,
                                int32_t *num_padded, int32_t *dev_status, const uint16_t *x,
                                int d, uint16_t *xg, int num_sms, cudaStream_t stream);

// Router + alignment + gather in one launch, from the logits: ids and w are
// written as by launch_route.  Only for shapes route_align_gather_fits()
// accepts (E <= 128, M <= 512); cudaErrorInvalidValue otherwise.
bool route_align_gather_fits(int M, int k, int E, int num_sms);
cudaError_t launch_route_align_gather(const float *logits, int M, int k, int E, int block_m,
                                      int64_t cap, int32_t *ids, float *w, int32_t *sorted_ids,
                                      int32_t *block_expert, int32_t *offsets,
                                      int32_t *num_padded, int32_t *dev_status,
                                      const uint16_t *x, int d, uint16_t *xg, int num_sms,
                                      cudaStream_t stream);

cudaError_t launch_rmsnorm(const uint16_t *x, const uint16_t *w, int M, int d, float eps,
                           uint16_t *y, cudaStream_t stream);
size_t sampler_workspace_bytes(int M, int64_t V);
cudaError_t launch_sampler(const float *logits, int M, int64_t V, uint64_t seed, uint64_t offset,
                           float *entropy, int64_t *sample, int64_t *amax, void *workspace,
                           cudaStream_t stream);
cudaError_t launch_identity_align_gather(const uint16_t *x, int M, int d, int padded,
                                         int32_t *sorted_ids, int32_t *offsets, uint16_t *xg,
                                         cudaStream_t stream);
cudaError_t launch_combine(const float *y, const int32_t *ids, const float *w, int M, int k,
                           int d, int E, uint16_t *out, cudaStream_t stream);
// Sets the counters [M, d/128] of the combine folded into the down GEMM
// and zeroes the out rows of tokens without a valid expert id.
cudaError_t launch_combine_prepare(const int32_t *ids, int M, int k, int E, int d, int32_t *cnt,
                                   uint16_t *out, cudaStream_t stream);

// Grouped W4A16 GEMM (tcgen05).  gate_up=true: xg fp16 -> h fp16 with the
// gated activation; gate_up=false: h fp16 -> y fp32.
struct GroupedGemmProblem {
    bool gate_up;
    const uint16_t *act;        // xg or h, [cap, K] fp16 in block order
    const uint8_t *wq;          // [E, R, K/2]
    const uint16_t *ws, *wz;    // [E, R, K/group]
    const int32_t *sorted_ids;  // [cap]
    const int32_t *expert_offsets;  // [E+1]
    void *out;                  // h [cap, m] fp16 or y [A, d] fp32
    int32_t *dev_status;
    int M, k, E, K, R, group;
    int out_cols;               // m (gate_up) or d (down)
    int64_t cap;
    // true only when the kernel that wrote sorted_ids / expert_offsets is at
    // least two launches back in the stream and the launch in between waits
    // for it before triggering (the layer's align -> gate_up -> down order):
    // down may then read its schedule, and stream its weights, before its
    // grid-dependency wait.  Activations are read only after that wait.
    bool early_schedule = false;
    // The layer's fixed-order combine folded into the down launch (both
    // launches get comb_cnt; NULL: neither does anything of it).  gate_up
    // sets the counters [M][comb_d/128] and zeroes the out rows of tokens
    // without a valid expert id; down writes out [M, comb_d] bf16 =
    // sum_j w_j y_j (bit-identical to launch_combine) as tokens complete.
    const int32_t *topk_ids = nullptr;   // [M, k]
    const float *topk_w = nullptr;       // [M, k] (down)
    int32_t *comb_cnt = nullptr;
    uint16_t *comb_out = nullptr;
    int comb_d = 0;
    // test hooks (w4_test_pipeline_hooks): the pipeline wait limit, and
    // withholding the first unit's scale/zero copy so that waits run out
    uint64_t wait_ns = 1000000000ull;
    bool test_withhold_sz = false;
};

// The test hooks of the calling thread, applied to its grouped GEMM launches.
struct PipelineTestHooks {
    uint64_t wait_ns = 1000000000ull;
    bool withhold_sz = false;
};
PipelineTestHooks &pipeline_test_hooks();

// The dense W4A16 GEMM (dense_gemm.cu): y [M, N] bf16 = xg [Mpad, K] fp16
// (block order, rows past M zero) . deq(W)^T, W [N, K/2] u8 with s, z
// [N, K/group] fp16.  partials: fp32 [splits, M, N] when the contraction is
// split (dense_gemm_partial_bytes > 0), else unused.
struct DenseGemmProblem {
    const uint16_t *xg;
    const uint8_t *q;
    const uint16_t *s, *z;
    uint16_t *y;
    float *partials;
    int32_t *dev_status;
    int M, N, K, group;
};
bool dense_gemm_supported(int M, int N, int K, int group);
int dense_gemm_splits(int M, int N, int K);
size_t dense_gemm_partial_bytes(int M, int N, int K);
cudaError_t launch_dense_gemm(const DenseGemmProblem &p, cudaStream_t stream, const char **why);

// Whether the grouped GEMM's shared memory (code, activation and scale/zero
// stages, schedule) fits the current device for contraction dim K with
// this group and expert count; launch_grouped_gemm rejects what does not.
bool grouped_gemm_fits(bool gate_up, int K, int group, int E);

// Returns cudaSuccess, or an error; *why receives a static description when
// the problem is rejected before launch (shape or resource limits).
cudaError_t launch_grouped_gemm(const GroupedGemmProblem &p, cudaStream_t stream,
                                const char **why);

// W4_OK when the current device is an sm_103 part, else W4_ERR_NO_DEVICE or
// W4_ERR_CUDA with the detail recorded (the argument checks of every entry
// point call it before launching).
int check_device_sm103();

// Records `detail` as the text w4_last_error_detail() returns on this thread
// and passes `status` through.
int set_error_detail(int status, const char *detail);

// Launch `kern` as a programmatic dependent of the preceding kernel in the
// stream.  Every kernel launched this way calls pdl_wait() before it reads
// anything an earlier kernel wrote and pdl_trigger() only after that wait,
// so at most two adjacent kernels of a stream overlap and, while the later
// one runs ahead of its wait, every kernel before the earlier one is done.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace w4
