// prof.h -- per-launch timing hook (internal).  While the calling thread has
// profiling enabled (attn_profile_begin), launchers bracket each kernel with
// prof_before / prof_after, which record CUDA events on the launch stream.
#pragma once

#include <cuda_runtime.h>

namespace gbattn {

// Kernel kinds reported by attn_profile_read (same values as in gbattn.h).
enum ProfKind {
    kProfFwd = 0,
    kProfBwdPreprocess = 1,
    kProfBwdDkDv = 2,
    kProfBwdDq = 3,
    kProfMerge = 4,
    kProfSimtFwd = 5,
    kProfSimtBwdDq = 6,
    kProfSimtBwdDkDv = 7,
    kProfBwdFused = 8,
    kProfBwdDqConvert = 9,
    kProfMergeBwd = 10,
    kProfBwdDkvReduce = 11,
    kProfThdRows = 12,
};

void prof_before(cudaStream_t st, int kind);
void prof_after(cudaStream_t st);

}  // namespace gbattn
