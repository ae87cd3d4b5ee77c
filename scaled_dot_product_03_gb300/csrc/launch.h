// launch.h -- host-side launchers of the library's kernels (internal).
#pragma once

#include <utility>

#include "common.cuh"

namespace gbattn {

struct FwdArgs {
    Geometry g;
    View q, k, v;
    MutView o;
    float *lse;
    unsigned *err;        // device error word (watchdog)
    uint64_t watchdog_ns;
};

struct BwdArgs {
    Geometry g;
    View q, k, v, o, dout;
    const float *lse;
    MutView dq, dk, dv;
    const float *dlse;    // optional gradient of the loss w.r.t. LSE (LSE layout)
    float *delta;         // workspace: row terms <dO_i, O_i> - dLSE_i, laid out like LSE
    float *dq_acc;        // fp32 dq accumulator laid out like LSE with D columns
                          // per row, cleared by the preprocess kernel; null when
                          // the backward does not use one
    float *dkv_part = nullptr;  // single pass with the query heads of a group split
                          // over nsplit CTAs: fp32 partial dK, dV per split,
                          // [nsplit][2][key rows][Hkv][D] (null: no split)
    int nsplit = 1;       // query-head splits per key tile (1: none)
    int acc_d = 0;        // floats per row of dq_acc and of the partials (the
                          // tensor-core head dim, tc_dim(D))
    unsigned *work_ctr = nullptr;  // persistent single pass: items taken after
                          // each CTA's first, zeroed by the preprocess kernel
    unsigned *err;
    uint64_t watchdog_ns;
};

struct MergeArgs {
    int B, S, H, D;
    View o1, o2;
    MutView out;
    const float *lse1, *lse2;
    float *lse_out;
};

// Streaming multiprocessors of the current device (queried once per device).
cudaError_t device_sm_count(int *out);

// Launches kern on st with programmatic stream serialization: the grid may
// begin while the previous kernel on the stream is finishing (once that
// kernel's CTAs have issued griddep_launch), so kern must griddep_wait
// before it reads anything the previous kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// dtype: 0 = fp16, 1 = bf16, 2 = fp32 (same values as attn_dtype).
cudaError_t launch_simt_fwd(int dtype, const FwdArgs &a, int max_lq, cudaStream_t st);
// Preprocess (q_rows query rows), then the FFMA dq and dk/dv kernels.
cudaError_t launch_simt_bwd(int dtype, const BwdArgs &a, int max_lq, int max_lkv, int q_rows,
                            cudaStream_t st);
cudaError_t launch_bwd_preprocess(int dtype, const BwdArgs &a, int rows, cudaStream_t st);
cudaError_t launch_merge(int dtype, const MergeArgs &a, cudaStream_t st);

struct MergeBwdArgs {
    int B, S, H, D;
    View o1, o2, dout;
    MutView do1, do2;
    const float *lse1, *lse2, *dlse;  // dlse may be null
    float *dlse1, *dlse2;
};
cudaError_t launch_merge_bwd(int dtype, const MergeBwdArgs &a, cudaStream_t st);
// THD row sums of the emulated context-parallel backward: mode 0 adds the
// rows of v inside a sequence into acc, mode 2 copies them there, mode 1
// writes acc into v (0 outside every sequence).  acc: [T, H, D] fp32
// contiguous.
cudaError_t launch_thd_rows(int dtype, int mode, int T, int H, int D, const MutView &v, float *acc, const int *cu,
                            const int *pad, int B, cudaStream_t st);
cudaError_t launch_partitioned_indices(const int *pad, int B, int world, int rank, int n_out, int *out,
                                       cudaStream_t st);

}  // namespace gbattn
