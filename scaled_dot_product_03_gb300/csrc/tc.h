// tc.h -- launchers of the tcgen05 (tensor-core) kernels (internal).
#pragma once

#include "launch.h"

namespace gbattn {

// Whether the tensor-core kernels cover this element type and head dim.
bool uses_tc_fwd(int dtype, int D);
bool uses_tc_bwd(int dtype, int D);
// Whether the single-pass backward (fp32 dQ accumulator) covers them.
bool uses_tc_bwd_fused(int dtype, int D);

cudaError_t launch_tc_fwd(int dtype, const FwdArgs &a, int max_lq, int max_lkv, cudaStream_t st);
// The backward launchers encode every tensor map they need first, then
// enqueue the row-term preprocess (over q_rows query rows) and their kernels,
// so a refused map enqueues nothing.
cudaError_t launch_tc_bwd(int dtype, const BwdArgs &a, int max_lq, int max_lkv, int q_rows,
                          cudaStream_t st);
// Single-pass backward: a.dq_acc (fp32, laid out like LSE with D columns per
// row) is cleared by the preprocess; writes dk, dv and then dq.
cudaError_t launch_tc_bwd_fused(int dtype, const BwdArgs &a, int max_lkv, int q_rows, cudaStream_t st);
// The head-dim-64 form of the single-pass backward.
cudaError_t launch_tc_bwd_fused64(int dtype, const BwdArgs &a, int max_lkv, int q_rows, cudaStream_t st);
// dk, dv from the fp32 partials of split query heads (a.dkv_part), D = 64 or 128.
cudaError_t launch_dkv_reduce(int dtype, const BwdArgs &a, cudaStream_t st);
// dq = scale * accumulator, in dq's element type and strides (D = 64 or 128).
cudaError_t launch_dq_convert(int dtype, const BwdArgs &a, cudaStream_t st);

// One kernel that waits on an mbarrier nothing arrives on, gives up after
// `limit_ns`, and records the timeout in *err.
cudaError_t launch_watchdog_selftest(unsigned *err, uint64_t limit_ns, cudaStream_t st);

}  // namespace gbattn
