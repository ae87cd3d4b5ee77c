// tc_fwd.cu -- tcgen05 forward kernel (fp16/bf16).
#include "ptx.cuh"
#include "tc.h"

namespace gbattn {

bool uses_tc_fwd(int dtype, int D) { return false; }

cudaError_t launch_tc_fwd(int dtype, const FwdArgs &a, int max_lq, int max_lkv, cudaStream_t st) {
    return cudaErrorNotSupported;
}

}  // namespace gbattn
