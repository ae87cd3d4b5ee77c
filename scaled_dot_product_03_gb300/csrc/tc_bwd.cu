// tc_bwd.cu -- tcgen05 backward kernels (fp16/bf16).
#include "ptx.cuh"
#include "tc.h"

namespace gbattn {

bool uses_tc_bwd(int dtype, int D) { return false; }

cudaError_t launch_tc_bwd(int dtype, const BwdArgs &a, int max_lq, int max_lkv, int q_rows,
                          cudaStream_t st) {
    return cudaErrorNotSupported;
}

}  // namespace gbattn
