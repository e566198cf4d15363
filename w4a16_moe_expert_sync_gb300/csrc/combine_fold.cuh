// combine_fold.cuh -- the fixed-order combine folded into the down GEMM:
// per-(token, 128-column panel) arrival counters.
//
// The combine of token t needs the y rows of all its valid assignments,
// which different CTAs of the down GEMM produce in no fixed order.  Once a
// CTA has stored one assignment's 128 y columns of a panel it counts one
// arrival on counter (t, panel); the warp that brings the counter to k
// computes those 128 columns of out[t] from all k rows in assignment order
// (the same fp32 fma chain as the standalone combine), so the result does
// not depend on which CTA finishes last and no output element is written
// twice.  A counter starts at k minus the token's number of valid
// assignments; a token with none gets its zero out row when the counters
// are set.
#pragma once

#include <cstdint>

namespace w4 {

// Counters of token t: [d / 128 panels] int32.
__host__ __device__ inline int64_t fold_counter_index(int t, int panels, int panel)
{
    return static_cast<int64_t>(t) * panels + panel;
}

// Sets token t's counters, by one warp (all 32 lanes call it).  out [M, d]
// bf16 rows are 8-byte aligned (d % 128 == 0, out 8-byte aligned).
__device__ __forceinline__ void fold_prepare_token(int t, int lane, const int32_t *topk_ids,
                                                   int k, int E, int d, int32_t *cnt,
                                                   uint16_t *out)
{
    const unsigned full = 0xffffffffu;
    int nvalid = 0;
    for (int j0 = 0; j0 < k; j0 += 32) {
        const int j = j0 + lane;
        const int e = j < k ? __ldg(topk_ids + static_cast<int64_t>(t) * k + j) : -1;
        nvalid += __popc(__ballot_sync(full, e >= 0 && e < E));
    }
    const int panels = d / 128;
    int32_t *c = cnt + fold_counter_index(t, panels, 0);
    for (int i = lane; i < panels; i += 32)
        c[i] = k - nvalid;
    if (nvalid == 0) {
        uint2 *o = reinterpret_cast<uint2 *>(out + static_cast<int64_t>(t) * d);
        for (int i = lane; i < d / 4; i += 32)
            o[i] = make_uint2(0, 0);
    }
}

}  // namespace w4
