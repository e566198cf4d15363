/*
 * w4moe.h -- C ABI of libw4moe.so, a GB300 (sm_103a) library for the W4A16
 * routed mixture-of-experts layer of a block-diffusion LM's denoising forward.
 *
 * The layer (per token t with routed experts e_j and weights w_j, j < k):
 *     g, u  = x_t . deq(Wgu[e_j])^T        gate rows [0, m), up rows [m, 2m)
 *     h     = gelu_tanh(g) * u
 *     y_j   = h . deq(Wdn[e_j])^T
 *     out_t = sum_{j = 0..k-1, in order} w_j * y_j
 * with deq(W)[r, c] = s[r, c/group] * (q[r, c] - z[r, c/group]), q a uint4
 * code, s and z fp16 ("diffusiongemma-26B-A4B-w4a16" -- Checkpoint format;
 * "Inference: Making every denoising pass fast" -- The first constraint was
 * capacity, Quantisation alone leaves a sparse execution problem;
 * "dg-w4-kernels" -- Grouped MoE).  The gated activation is not named on the
 * pages; this library uses gelu_tanh(gate) * up.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer owned by the caller, except
 *     where stated.  The library never allocates device memory, never
 *     synchronises the device and never reads device data on the host, so a
 *     sequence of calls can be captured in a CUDA graph.
 *   - Every call is asynchronous on `stream` (0 = the legacy default stream).
 *   - The return value reports argument and launch errors only (w4_status).
 *     On a nonzero return nothing was launched.  w4_last_error_detail() gives
 *     a one-line description of the last failure on the calling thread.
 *   - Errors found on the device (an expert id outside [0, E), a pipeline
 *     wait that ran past its time limit) are OR-ed into *dev_status as the
 *     W4_DEV_* bits below; the kernels never trap.  dev_status may be NULL
 *     where the signature allows it, in which case such errors are dropped.
 *   - Dtypes: bf16 and fp16 values travel as uint16_t bit patterns.
 *   - Pointers to data read with 16-byte vector loads or TMA must be 16-byte
 *     aligned (W4_ERR_MISALIGNED otherwise); allocations from cudaMalloc or
 *     PyTorch always are.
 *   - Shapes are int; products that exceed 2^31 are not supported.
 */
#ifndef W4MOE_H
#define W4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define W4MOE_ABI_VERSION 9

/* Opaque CUDA stream; ABI-identical to cudaStream_t / CUstream. */
typedef struct CUstream_st *w4_stream_t;

typedef enum {
    W4_OK = 0,
    W4_ERR_INVALID_ARG = 1,       /* NULL pointer, negative size, bad option   */
    W4_ERR_UNSUPPORTED_SHAPE = 2, /* a shape the kernels do not handle         */
    W4_ERR_MISALIGNED = 3,        /* a pointer is not 16-byte aligned          */
    W4_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed      */
    W4_ERR_NO_DEVICE = 5,         /* no sm_103 device, or a driver entry point
                                     the library needs is missing              */
    W4_ERR_WORKSPACE = 6          /* workspace NULL or smaller than required   */
} w4_status;

/* Bits OR-ed into *dev_status by the kernels. */
#define W4_DEV_BAD_EXPERT_ID 0x1      /* an id outside [0, E); it was skipped   */
#define W4_DEV_PIPELINE_TIMEOUT 0x2   /* a pipeline wait exceeded ~1 s; the
                                         kernel stopped and its outputs are
                                         incomplete                              */
#define W4_DEV_TOO_MANY_JOBS 0x4      /* internal job list overflow (cannot
                                         happen for shapes the host accepted)   */
#define W4_DEV_FP16_RANGE 0x8         /* an activation (x, or h after the gated
                                         activation) lay outside fp16's finite
                                         range and was saturated to +-65504:
                                         the GEMMs' operands are fp16           */
#define W4_DEV_OUT_OF_BOUNDS 0x10     /* a range check of a data-dependent
                                         global store failed and the store was
                                         skipped (only in a library built with
                                         -DW4_CHECK_BOUNDS, a test build)       */

/* Human-readable name of a w4_status value (static string). */
const char *w4_status_string(int status);

/* Description of the last failure on the calling thread (static per thread). */
const char *w4_last_error_detail(void);

/* W4MOE_ABI_VERSION of the loaded library. */
int w4_abi_version(void);

/* --------------------------------------------------------------------------
 * w4_quantize -- quantize_w4, the checkpoint packer
 * ("diffusiongemma-26B-A4B-w4a16" -- Checkpoint format: 4-bit unsigned
 *  codes with an fp16 scale and zero point per group, packed low nibble
 *  first; -- Benchmarks: min/max round-to-nearest with no calibration;
 *  "dg-w4-kernels" -- W4A16: the packer's Python call, quantize_w4).
 *
 *   W   [E, N, K] fp32, row-major (contraction dim K innermost)
 *   q   [E, N, K/2] uint8 out, two codes per byte, low nibble first
 *   s,z [E, N, K/group] fp16 out
 * Per group of `group` consecutive elements of a row, in fp32:
 *   s = (max - min) / 15, stored fp16 (a zero fp16 scale becomes 1.0);
 *   z = -min / s16, stored fp16 (fractional zero point);
 *   q = clamp(round_half_even(w / s16 + z16), 0, 15), no fused multiply-add.
 * group must be 64, 128 or 256 and divide K.  W must be 16-byte aligned.
 * Offline, one-time; not part of the timed layer.
 * ------------------------------------------------------------------------ */
int w4_quantize(const float *W, int E, int N, int K, int group,
                uint8_t *q, uint16_t *s, uint16_t *z, w4_stream_t stream);

/* --------------------------------------------------------------------------
 * w4_moe_route -- router: softmax over E logits, top-k, renormalise
 * ("Inference: Making every denoising pass fast" -- Quantisation alone leaves
 *  a sparse execution problem: a router scores the experts per token and the
 *  token runs through the 8 best of 128).
 *
 *   logits        [M, E] fp32
 *   topk_ids      [M, k] int32 out: the k largest logits, ties to the lower
 *                 index, in descending order
 *   topk_weights  [M, k] fp32 out: exp(l_j - l_max) / sum_i exp(l_i - l_max)
 *                 over the k selected (= softmax renormalised over the k)
 * Requires 1 <= k <= 32, k <= E <= 1024.
 * ------------------------------------------------------------------------ */
int w4_moe_route(const float *logits, int M, int E, int k,
                 int32_t *topk_ids, float *topk_weights, w4_stream_t stream);

/* --------------------------------------------------------------------------
 * w4_moe_align -- sync-free token-to-expert alignment
 * ("Inference: Making every denoising pass fast" -- Quantisation alone leaves
 *  a sparse execution problem: sort assignments by expert, pad into regular
 *  blocks; "dg-w4-kernels" -- Grouped MoE: sync-free, CUDA-graph safe).
 *
 * Flat assignment index a = t*k + j (A = M*k).  With c_e the number of
 * assignments to expert e and bm = block_m:
 *   expert_offsets [E+1] out: o_0 = 0, o_{e+1} = o_e + ceil(c_e/bm)*bm
 *   sorted_ids     [cap] out: slot o_e + r holds the r-th smallest a routed
 *                  to e (stable); padding slots and slots >= o_E hold A
 *   block_expert   [cap/bm] out: owning expert of block b, -1 past o_E
 *   num_padded     [1] out: o_E (stays on the device)
 * where cap = w4_moe_align_capacity(M, k, E, block_m).  ids outside [0, E)
 * are skipped and set W4_DEV_BAD_EXPERT_ID in *dev_status (may be NULL).
 * block_m must be 16, 32, 64, 128 or 256; E <= 1024.  One CTA, no atomics
 * on global memory, no host synchronisation.
 * ------------------------------------------------------------------------ */
int64_t w4_moe_align_capacity(int M, int k, int E, int block_m);
int w4_moe_align(const int32_t *topk_ids, int M, int k, int E, int block_m,
                 int32_t *sorted_ids, int32_t *block_expert, int32_t *expert_offsets,
                 int32_t *num_padded, int32_t *dev_status, w4_stream_t stream);

/* --------------------------------------------------------------------------
 * Contraction order of the grouped GEMMs ("block order")
 * The GEMMs expand eight packed codes at a time into fp16 pairs
 * (q0,q4) (q1,q5) (q2,q6) (q3,q7), so inside every block of 8 columns of an
 * activation row, column p holds element k(p) = (p >> 1) + 4 * (p & 1), i.e.
 * the order 0,4,1,5,2,6,3,7.  Gathered activations (xg) and h use this
 * order; it is an implementation layout, not part of the checkpoint format.
 *
 * Group sums.  Every xg and h row ends in one block of 64 fp16 columns of
 * sums of its own fp16 values: xg column d + g holds the sum of group g (128
 * consecutive elements of x), h column m + 4 g + i the sum of quarter i (16
 * intermediates) of group g of 64; the columns past the last sum, up to a
 * multiple of 16, hold zero, and the rest of the block is not written.  The GEMMs multiply them by the part of each
 * group's dequantisation constant -z*s that its fp16 rounding dropped, so
 * every dequantised weight is exact to its own fp16 rounding.  Hence
 * d <= 8192 and m <= 1024.
 *
 * w4_gather_activations -- the gate_up GEMM's input in slot order:
 *   xg [cap, d + 64] fp16 out: for every slot < num_padded, the row of token
 *   sorted_ids[slot] / k of x converted to fp16 in block order, then its
 *   group sums, or zeros for a padding slot; rows >= num_padded are not
 *   written.
 * x [M, d] bf16; sorted_ids / num_padded from w4_moe_align with the same k,
 * E, block_m.  bf16 -> fp16 rounds to nearest even: exact for magnitudes in
 * [2^-14, 65504], within 2^-25 below that (fp16 subnormals); larger
 * magnitudes (and inf, NaN) do not fit: they saturate to +-65504 (NaN stays
 * NaN) and set W4_DEV_FP16_RANGE in *dev_status (may be NULL), as does a
 * group sum beyond that range.  Requires d % 128 == 0, d <= 8192, x and xg
 * 16-byte aligned.
 * ------------------------------------------------------------------------ */
int w4_gather_activations(const uint16_t *x, int M, int d, int k, int E, int block_m,
                          const int32_t *sorted_ids, const int32_t *num_padded, uint16_t *xg,
                          int32_t *dev_status, w4_stream_t stream);

/* w4_moe_align_gather -- w4_moe_align and w4_gather_activations in one launch:
 * every CTA counts all assignments per expert in its own shared memory (so no
 * CTA waits on another), places the assignments of its own range of tokens
 * and copies those tokens' rows to their slots; the grid writes the padding
 * slots and block owners.  The first launch of w4_moe_layer.  Arguments and
 * outputs as in those two calls, except that the xg rows of padding slots
 * are NOT written (their contents are unspecified; the GEMMs discard or
 * zero what they produce for padding slots).  Activations outside fp16's
 * range set W4_DEV_FP16_RANGE. */
int w4_moe_align_gather(const int32_t *topk_ids, const uint16_t *x, int M, int d, int k, int E,
                        int block_m, int32_t *sorted_ids, int32_t *block_expert,
                        int32_t *expert_offsets, int32_t *num_padded, uint16_t *xg,
                        int32_t *dev_status, w4_stream_t stream);

/* --------------------------------------------------------------------------
 * w4_moe_route_align_gather -- w4_moe_route, w4_moe_align and
 * w4_gather_activations from the router logits.  For small batches it is one
 * launch: every CTA routes every token (the same arithmetic as w4_moe_route,
 * so topk_ids and topk_weights are bit-identical to it) into shared memory,
 * computes the alignment there and gathers its own tokens' rows.  Routing
 * every token in every CTA costs more than a second launch once the batch
 * has more than a few tokens per warp, so beyond that the router runs as its
 * own launch and w4_moe_align_gather follows it (same results).  The first
 * step of w4_moe_layer_from_logits.
 *
 *   logits [M, E] fp32 in; topk_ids [M, k] int32 and topk_weights [M, k]
 *   fp32 out, as w4_moe_route; the other arguments and outputs as
 *   w4_moe_align_gather.
 * One launch for E <= 128 and M <= 16; two launches otherwise.
 * Requires what w4_moe_route and w4_moe_align_gather require.
 * ------------------------------------------------------------------------ */
int w4_moe_route_align_gather(const float *logits, const uint16_t *x, int M, int d, int k, int E,
                              int block_m, int32_t *topk_ids, float *topk_weights,
                              int32_t *sorted_ids, int32_t *block_expert,
                              int32_t *expert_offsets, int32_t *num_padded, uint16_t *xg,
                              int32_t *dev_status, w4_stream_t stream);

/* --------------------------------------------------------------------------
 * w4_grouped_gemm_gate_up -- grouped W4A16 gate_up GEMM with the gated
 * activation in its epilogue
 * ("dg-w4-kernels" -- Grouped MoE: one launch for all experts, activation
 *  folded into the first GEMM's epilogue; "diffusiongemma-26B-A4B-w4a16" --
 *  Checkpoint format: gate_up groups of 128 along the contraction dim).
 *
 *   xg             [cap, d + 64] fp16 from w4_gather_activations (slot order,
 *                  values then group sums)
 *   gu_q           [E, 2m, d/2] uint8 (w4_quantize layout), gu_s/gu_z
 *                  [E, 2m, d/group] fp16; rows [0, m) gate, [m, 2m) up
 *   sorted_ids, expert_offsets   from w4_moe_align with the same block_m
 *   h              [cap, m + 64] fp16 out, row = alignment slot: m values in
 *                  block order, h[slot] = gelu_tanh(g) * u for the token of
 *                  sorted_ids[slot], then the quarter sums of h's groups of
 *                  64 (see "Group sums"); zero rows for padding slots inside
 *                  an expert's range (whatever xg holds there); rows at slots
 *                  >= num_padded are not written.  A value of h (or a sum)
 *                  beyond fp16's range saturates to +-65504 and sets
 *                  W4_DEV_FP16_RANGE.
 * Weights are dequantised in registers to fp16 as q * s + fp16(-z * s) (one
 * fused rounding; scaled by a power of two per weight row, undone exactly in
 * fp32), multiplied on the tensor cores (tcgen05, fp16 x fp16 -> fp32), and
 * the part of -z * s lost to its fp16 rounding is added back through the
 * group sums; h is rounded to fp16 with saturation at +-65504.
 * The work runs as units of (job, 128 weight rows), a job being up to 32
 * consecutive slots of one expert, or up to 64 when M * k >= 64 * E; the
 * fp32 summation order follows from the shape alone, so results are
 * bit-identical from run to run.
 * Requires d % 128 == 0, d <= 8192, m % 64 == 0, m <= 1024, group == 128,
 * and that a unit's scales and zeros fit shared memory beside the code and
 * activation stages: d up to about 3584 at E = 128 (2688 at E = 1024);
 * W4_ERR_UNSUPPORTED_SHAPE beyond, before anything is launched.
 * dev_status may be NULL.
 * ------------------------------------------------------------------------ */
int w4_grouped_gemm_gate_up(const uint16_t *xg, int M, int d, int m, int E, int k, int block_m,
                            const uint8_t *gu_q, const uint16_t *gu_s, const uint16_t *gu_z,
                            int group, const int32_t *sorted_ids,
                            const int32_t *expert_offsets, uint16_t *h,
                            int32_t *dev_status, w4_stream_t stream);

/* --------------------------------------------------------------------------
 * w4_grouped_gemm_down -- grouped W4A16 down GEMM, contraction dim m (704 on
 * the pages) with groups of 64
 * ("diffusiongemma-26B-A4B-w4a16" -- Checkpoint format: down_proj groups of
 *  64 because 128 does not divide 704).
 *
 *   h              [cap, m + 64] fp16 from w4_grouped_gemm_gate_up (values in
 *                  block order, then quarter sums)
 *   dn_q           [E, d, m/2] uint8, dn_s/dn_z [E, d, m/group] fp16
 *   y              [M*k, d] fp32 out, row a = flat assignment index
 *                  (y[a] = h[slot of a] . deq(Wdn[e])^T); rows of skipped
 *                  (invalid-id) assignments are not written
 * Same dequantisation and correction as gate_up.
 * Requires d % 128 == 0, d <= 8192, m % 64 == 0, m <= 1024, group == 64.
 * dev_status may be NULL.
 * ------------------------------------------------------------------------ */
int w4_grouped_gemm_down(const uint16_t *h, int M, int d, int m, int E, int k, int block_m,
                         const uint8_t *dn_q, const uint16_t *dn_s, const uint16_t *dn_z,
                         int group, const int32_t *sorted_ids,
                         const int32_t *expert_offsets, float *y,
                         int32_t *dev_status, w4_stream_t stream);

/* --------------------------------------------------------------------------
 * w4_moe_combine_fixed_order -- atomics-free weighted combine
 * ("Inference: Making every denoising pass fast" -- Quantisation alone leaves
 *  a sparse execution problem: a token's eight outputs are reduced in a fixed
 *  order, never with index_add_ atomics, so reruns are bit-identical).
 *
 *   out[t, c] = bf16_rn( fma-chain over j = 0..k-1 in order, starting at 0,
 *                        of topk_weights[t, j] * y[t*k + j, c] )  in fp32;
 *   slots whose id is outside [0, E) contribute nothing.
 *   y [M*k, d] fp32, topk_ids/topk_weights [M, k], out [M, d] bf16.
 * Requires d % 4 == 0.
 * ------------------------------------------------------------------------ */
int w4_moe_combine_fixed_order(const float *y, const int32_t *topk_ids,
                               const float *topk_weights, int M, int k, int d, int E,
                               uint16_t *out, w4_stream_t stream);

/* --------------------------------------------------------------------------
 * w4_grouped_gemm_down_combine -- w4_grouped_gemm_down with
 * w4_moe_combine_fixed_order folded into its epilogue: one launch for both
 * ("dg-w4-kernels" -- Grouped MoE: one fused launch; "Inference: Making every
 *  denoising pass fast" -- Quantisation alone leaves a sparse execution
 *  problem: the fixed-order, atomics-free reduction of a token's outputs).
 *
 *   h, dn_q/dn_s/dn_z, sorted_ids, expert_offsets, y   as w4_grouped_gemm_down
 *                  (y is still written: it holds the terms of the combine)
 *   topk_ids/topk_weights [M, k]   as w4_moe_combine_fixed_order
 *   counters       [M, d/128] int32, set by w4_moe_combine_prepare with
 *                  the same topk_ids, M, k, E, d and out (earlier on the
 *                  stream, after any earlier use of the same counters);
 *                  consumed by this call
 *   out            [M, d] bf16 out, 8-byte aligned: bit-identical to
 *                  w4_grouped_gemm_down followed by
 *                  w4_moe_combine_fixed_order
 * After its last unit each CTA counts one arrival per slot of each of its
 * units on the (token, 128-column panel) counter; the warp whose arrival
 * completes a counter computes those 128 columns of out[t] from the token's
 * k rows of y in assignment order (the combine's fp32 fma chain), so no
 * element of out is written twice and none depends on arrival order.  The
 * counter atomics are the only atomics; they decide who combines, never
 * what.  The counting and the combines run after each CTA's last unit, so
 * the CTAs that finish last take most of them: one launch fewer than down
 * followed by w4_moe_combine_fixed_order, but at M = 256, d = 2816, top-8
 * about 13 us slower per layer, which is why w4_moe_layer does not use it.
 * Same requirements as w4_grouped_gemm_down.
 * ------------------------------------------------------------------------ */
int w4_grouped_gemm_down_combine(const uint16_t *h, int M, int d, int m, int E, int k,
                                 int block_m, const uint8_t *dn_q, const uint16_t *dn_s,
                                 const uint16_t *dn_z, int group, const int32_t *sorted_ids,
                                 const int32_t *expert_offsets, const int32_t *topk_ids,
                                 const float *topk_weights, int32_t *counters, float *y,
                                 uint16_t *out, int32_t *dev_status, w4_stream_t stream);

/* w4_moe_combine_prepare -- sets the counters of w4_grouped_gemm_down_combine:
 * counters[t, p, q] = k - (number of ids of token t inside [0, E)), and
 * writes the zero out row of every token with no such id (the combine of no
 * terms).  topk_ids [M, k], counters [M, d/128] int32, out [M, d] bf16
 * (8-byte aligned).  Requires d % 128 == 0.  One launch. */
int w4_moe_combine_prepare(const int32_t *topk_ids, int M, int k, int E, int d,
                           int32_t *counters, uint16_t *out, w4_stream_t stream);

/* --------------------------------------------------------------------------
 * w4_moe_layer -- the whole routed-expert layer: alignment fused with the
 * activation gather, gate_up + activation, down, fixed-order combine, as
 * four launches on one stream (each a programmatic dependent of the one
 * before, so their starts and ends overlap)
 * ("dg-w4-kernels" -- Grouped MoE: out = fused_moe_w4_v2(hidden, experts,
 *  topk_ids, topk_weights)).
 *
 * workspace: caller-owned device buffer of at least
 * w4_moe_layer_workspace_size(...) bytes, 256-byte aligned; it holds the
 * alignment outputs, the gathered activations, h and y.  Its contents on return are the intermediates
 * of this call (layout: see the implementation; not part of the ABI).
 * Same shape rules as the individual calls; dev_status may be NULL.
 * ------------------------------------------------------------------------ */
size_t w4_moe_layer_workspace_size(int M, int d, int m, int E, int k, int block_m);
int w4_moe_layer(const uint16_t *x, const int32_t *topk_ids, const float *topk_weights,
                 int M, int d, int m, int E, int k, int block_m,
                 const uint8_t *gu_q, const uint16_t *gu_s, const uint16_t *gu_z, int gu_group,
                 const uint8_t *dn_q, const uint16_t *dn_s, const uint16_t *dn_z, int dn_group,
                 void *workspace, size_t workspace_bytes, uint16_t *out,
                 int32_t *dev_status, w4_stream_t stream);

/* --------------------------------------------------------------------------
 * w4_moe_layer_host -- w4_moe_layer with the step's activations, routing
 * and output in host memory: on `stream` it copies x [M, d] bf16, topk_ids
 * [M, k] and topk_weights [M, k] from the host into staging buffers in the
 * workspace (one cudaMemcpyAsync each), runs the layer's four launches and
 * copies out [M, d] bf16 back to out_host.  Everything is enqueued
 * asynchronously: with page-locked host buffers the copies overlap other
 * streams' work, and the call returns before they finish, so synchronise
 * the stream before reading out_host or changing the host inputs.  Calls on
 * different streams with different workspaces may run concurrently.
 *
 * workspace: device buffer of at least w4_moe_layer_host_workspace_size(...)
 * bytes, 256-byte aligned: the layer's workspace followed by the staging
 * buffers.  Weights, dev_status and the shape rules as w4_moe_layer; a host
 * pointer that is NULL while M > 0 is W4_ERR_INVALID_ARG; M = 0 does nothing.
 * ------------------------------------------------------------------------ */
size_t w4_moe_layer_host_workspace_size(int M, int d, int m, int E, int k, int block_m);
int w4_moe_layer_host(const uint16_t *x_host, const int32_t *topk_ids_host,
                      const float *topk_weights_host, int M, int d, int m, int E, int k,
                      int block_m,
                      const uint8_t *gu_q, const uint16_t *gu_s, const uint16_t *gu_z, int gu_group,
                      const uint8_t *dn_q, const uint16_t *dn_s, const uint16_t *dn_z, int dn_group,
                      void *workspace, size_t workspace_bytes, uint16_t *out_host,
                      int32_t *dev_status, w4_stream_t stream);

/* --------------------------------------------------------------------------
 * w4_moe_layer_from_logits -- w4_moe_layer with the router in its first
 * launch: from the router logits [M, E] fp32 instead of topk_ids and
 * topk_weights, which it writes (caller-owned [M, k] int32 / fp32 outputs,
 * as w4_moe_route) and then uses for the combine.  Same workspace as
 * w4_moe_layer (w4_moe_layer_workspace_size); out is bit-identical to
 * w4_moe_route followed by w4_moe_layer.
 * ------------------------------------------------------------------------ */
int w4_moe_layer_from_logits(const uint16_t *x, const float *logits, int M, int d, int m, int E,
                             int k, int block_m, const uint8_t *gu_q, const uint16_t *gu_s,
                             const uint16_t *gu_z, int gu_group, const uint8_t *dn_q,
                             const uint16_t *dn_s, const uint16_t *dn_z, int dn_group,
                             void *workspace, size_t workspace_bytes, int32_t *topk_ids,
                             float *topk_weights, uint16_t *out, int32_t *dev_status,
                             w4_stream_t stream);

/* --------------------------------------------------------------------------
 * w4_moe_layer_static_scratch -- w4_moe_layer without a workspace argument.
 * The paper has no counterpart: this is a library convenience for callers
 * that cannot allocate device memory when they call the layer, e.g. a plain
 * C host with no device allocator of its own, or a server that reserves its
 * memory at start-up and must not call cudaMalloc/cudaFree (which
 * synchronise the device) or re-enter its allocator afterwards.
 *
 * The intermediates live in one library-owned device array of
 * W4_STATIC_SCRATCH_BYTES (64 MiB) per device; that holds the M = 256,
 * d = 2816, m = 704, E = 128, k = 8 layer at block_m = 16 (about 51 MB).
 * Shapes whose w4_moe_layer_workspace_size(...) exceeds it are rejected with
 * W4_ERR_WORKSPACE before anything is launched.  Nothing is allocated: no
 * cudaMalloc, no cudaFree, no allocating library routine.  Nothing in the
 * array needs to start at zero.
 *
 * Every call looks up the array's device address on the current device
 * (cudaGetSymbolAddress, host-only), so the address always belongs to the
 * current context, also after a cudaDeviceReset.  The first call on a device
 * may load the library's module onto it; make that first call before any
 * stream capture.
 *
 * Every call on a device shares the one array: calls whose GPU work overlaps
 * (different streams, or different host threads with different streams)
 * race and corrupt each other's results.  Issue them on one stream.
 * Arguments, outputs, shape rules and errors otherwise as w4_moe_layer.
 * ------------------------------------------------------------------------ */
#define W4_STATIC_SCRATCH_BYTES (64u << 20)
int w4_moe_layer_static_scratch(const uint16_t *x, const int32_t *topk_ids,
                                const float *topk_weights,
                                int M, int d, int m, int E, int k, int block_m,
                                const uint8_t *gu_q, const uint16_t *gu_s, const uint16_t *gu_z,
                                int gu_group,
                                const uint8_t *dn_q, const uint16_t *dn_s, const uint16_t *dn_z,
                                int dn_group, uint16_t *out, int32_t *dev_status,
                                w4_stream_t stream);

/* --------------------------------------------------------------------------
 * w4_w4a16_linear -- the dense W4A16 linear: y = x . deq(W)^T
 * ("dg-w4-kernels" -- W4A16: w4a16_linear(x, qw, scale, zero) equals
 *  F.linear(x, dequant(W)), reading packed nibbles and dequantising inline;
 *  "Inference: Making every denoising pass fast" -- Dense W4 everywhere:
 *  attention, the shared MLP and the LM head as dense W4A16 layers).
 *
 *   x          [M, K] bf16 in
 *   q          [N, K/2] uint8, w4_quantize's layout; s, z [N, K/group] fp16
 *   y          [M, N] bf16 out
 *   workspace  device scratch of w4_w4a16_linear_workspace_size(M, K, N,
 *              group) bytes, 256-byte aligned; contents need no initialisation
 * The rows are converted to fp16 in the GEMMs' operand order (one launch),
 * then multiplied by the dequantised weight: fp16 x fp16 tcgen05 MMA with
 * fp32 accumulation, rows rounded to bf16 once.  Each 128-row panel of W is
 * dequantised once per pass of up to 256 token rows, and narrow outputs
 * split the contraction (fp32 partial sums in the workspace, added in split
 * order by one more launch; the split depends on the shape only, so results
 * are the same on every GPU).  Two or three launches.
 * Requires group 64 or 128, K >= 256 a multiple of the group and of 64 with
 * K / group <= 32, N a multiple of 128.  dev_status may be NULL.
 * ------------------------------------------------------------------------ */
size_t w4_w4a16_linear_workspace_size(int M, int K, int N, int group);
int w4_w4a16_linear(const uint16_t *x, int M, int K, int N, const uint8_t *q, const uint16_t *s,
                    const uint16_t *z, int group, void *workspace, size_t workspace_bytes,
                    uint16_t *y, int32_t *dev_status, w4_stream_t stream);

/* ==========================================================================
 * Beside the layer: the per-step kernels of the denoising loop
 * ========================================================================== */

/* --------------------------------------------------------------------------
 * w4_rmsnorm -- fused_rmsnorm: y = x / sqrt(mean(x^2) + eps) * weight over
 * the last axis, one kernel
 * ("dg-w4-kernels" -- RMSNorm; "Inference: Making every denoising pass
 *  fast" -- RMSNorm: each activation rescaled by its root-mean-square
 *  magnitude).
 *
 *   x       [M, d] bf16 in (16-byte aligned)
 *   weight  [d] bf16 in (16-byte aligned); multiplies as is (no 1 + weight)
 *   y       [M, d] bf16 out (16-byte aligned; may equal x)
 * Arithmetic in fp32 (sum of squares, reciprocal square root, two products),
 * y rounded to bf16 once.  One warp per row with the row in registers for
 * d <= 4096; wider rows take a CTA per row.  Requires d % 8 == 0, eps >= 0.
 * ------------------------------------------------------------------------ */
int w4_rmsnorm(const uint16_t *x, const uint16_t *weight, int M, int d, float eps, uint16_t *y,
               w4_stream_t stream);

/* --------------------------------------------------------------------------
 * w4_sample_logits -- fused_entropy and gumbel_argmax_sample in one
 * streaming pass over vocabulary logits
 * ("dg-w4-kernels" -- Sampler: the entropy of Categorical(logits) in one
 *  pass instead of a logsumexp/sub/exp/mul/sum chain; a Gumbel-max draw from
 *  the same Categorical with Philox noise made inline, and the plain argmax
 *  from the same reduction).
 *
 *   logits   [M, V] fp32 in; -inf entries are masked out; a row needs one
 *            finite entry (an all -inf row gives a NaN entropy)
 *   seed, offset  the noise stream: Philox4x32-10 (Salmon et al., SC 2011)
 *            with key (seed lo, seed hi) and counter (c / 4, t, offset lo,
 *            offset hi) for row t, column c, which takes output word c % 4;
 *            a word r gives g = -ln(-ln(1 - v)), v = (r + 1/2) 2^-32
 *   entropy  [M] fp32 out, -sum p ln p in nats, or NULL to skip
 *   sample   [M] int64 out, argmax_c (logit + g), or NULL to skip
 *   argmax   [M] int64 out, argmax_c logit, or NULL to skip
 *   workspace  device scratch of w4_sample_logits_workspace_size(M, V)
 *            bytes (partials per row segment); contents need no initialisation
 * Ties go to the lower column.  Results do not depend on scheduling: every
 * reduction runs in a fixed order.  Quads of logits that cannot win the draw
 * (their largest logit + 23 below the running best; g < 22.9 always) skip
 * their noise, which changes no result.  Two launches: persistent CTAs
 * stream equal spans of the rows laid end to end and write one partial per
 * row segment, then one warp per row merges them.  The split depends on the
 * GPU's SM count, so results are bit-identical run to run on one GPU model.
 * Requires 0 < V < 2^31.
 * ------------------------------------------------------------------------ */
size_t w4_sample_logits_workspace_size(int M, int64_t V);
int w4_sample_logits(const float *logits, int M, int64_t V, uint64_t seed, uint64_t offset,
                     float *entropy, int64_t *sample, int64_t *argmax, void *workspace,
                     size_t workspace_bytes, w4_stream_t stream);

/* fused_entropy: w4_sample_logits with only the entropy. */
int w4_fused_entropy(const float *logits, int M, int64_t V, float *entropy, void *workspace,
                     size_t workspace_bytes, w4_stream_t stream);

/* gumbel_argmax_sample: w4_sample_logits with the sample and the argmax. */
int w4_gumbel_argmax_sample(const float *logits, int M, int64_t V, uint64_t seed,
                            uint64_t offset, int64_t *sample, int64_t *argmax, void *workspace,
                            size_t workspace_bytes, w4_stream_t stream);

/* --------------------------------------------------------------------------
 * w4_test_pipeline_hooks -- a test hook of the grouped GEMMs (not for
 * production use): for later w4_grouped_gemm_gate_up / _down / _down_combine
 * calls and the layer's GEMMs made from the calling thread, every pipeline
 * wait gives up after wait_limit_ns (0: back to the default of one second)
 * and, if withhold_first_scales is nonzero, each CTA withholds the copy of
 * its first unit's scales and zeros, so that its waits run out: the kernel
 * then sets W4_DEV_PIPELINE_TIMEOUT, lets its own copies land, drains its
 * MMAs, frees its tensor memory and exits, leaving its outputs incomplete
 * and the context usable.  Returns W4_OK.
 * ------------------------------------------------------------------------ */
int w4_test_pipeline_hooks(uint64_t wait_limit_ns, int withhold_first_scales);

#ifdef __cplusplus
}
#endif

#endif /* W4MOE_H */
