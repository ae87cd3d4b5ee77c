// noalloc.cu -- attn_bwd_noalloc: the backward pass with its scratch memory
// in a fixed device array owned by this library, for callers that cannot
// allocate device memory themselves.
//
// The scratch lives in the file-scope device array below.  Host code cannot
// use its name as a device address (on the host the name denotes a
// host-side stand-in), so the address is looked up with
// cudaGetSymbolAddress, once per device, with that device current, and
// handed to the kernels as an ordinary pointer.
#include <cstdio>
#include <mutex>

#include "gbattn.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[GBATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];

// Device address of g_bwd_scratch on the current device (looked up on the
// first call for that device).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_bwd_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

namespace gbattn {
// Records the calling thread's error message (defined with the C ABI).
attn_status record_error(attn_status st, const char *msg);
}  // namespace gbattn

extern "C" attn_status attn_bwd_noalloc(const attn_params *p, attn_tensor q, attn_tensor k,
                                        attn_tensor v, attn_tensor o, attn_tensor dout,
                                        const float *lse, attn_tensor dq, attn_tensor dk,
                                        attn_tensor dv, attn_stream_t stream) {
    const size_t need = attn_bwd_workspace_size(p);
    if (need > (size_t)GBATTN_NOALLOC_SCRATCH_BYTES) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "attn_bwd_noalloc: this problem needs %zu bytes of scratch, the library's "
                 "static scratch holds %zu; use attn_bwd with a caller-owned workspace",
                 need, (size_t)GBATTN_NOALLOC_SCRATCH_BYTES);
        return gbattn::record_error(ATTN_ERR_UNSUPPORTED, msg);
    }
    void *scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        char msg[200];
        snprintf(msg, sizeof msg, "attn_bwd_noalloc: address of the static scratch: %s",
                 cudaGetErrorString(e));
        return gbattn::record_error(ATTN_ERR_CUDA, msg);
    }
    // invalid parameters are reported by attn_bwd's own checks
    return attn_bwd(p, q, k, v, o, dout, lse, dq, dk, dv, scratch,
                    (size_t)GBATTN_NOALLOC_SCRATCH_BYTES, stream);
}
