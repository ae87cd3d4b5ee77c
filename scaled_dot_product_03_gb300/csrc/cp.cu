// cp.cu -- token partition of a padded THD buffer for context parallelism.
//
// "[PyTorch] Add support for cuDNN FusedAttention + THD + CP": with THD
// inputs, each sequence is cut into 2 x CP chunks and every rank holds two
// of them, so that causal work is balanced; the thread's code selects a
// rank's tokens with thd_get_partitioned_indices(cu_seqlens_padded,
// total_tokens, world_size, rank).  Rank r holds chunk r and the mirrored
// chunk 2 CP - 1 - r of every sequence (early chunks see few keys under a
// causal mask, late ones many; each pair sums to the same work).  Output
// position p of rank r lists, sequence by sequence, the buffer rows of
// chunk r then of chunk 2 CP - 1 - r.
#include "gbattn.h"
#include "launch.h"

namespace gbattn {
namespace {

__global__ void __launch_bounds__(256)
    partitioned_indices_kernel(const int *__restrict__ pad, int B, int world, int rank, int n_out,
                               int *__restrict__ out) {
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < n_out; p += gridDim.x * blockDim.x) {
        // sequence b owns local positions [pad[b] / world, pad[b + 1] / world)
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) / 2;
            if (__ldg(pad + mid) / world <= p) lo = mid; else hi = mid - 1;
        }
        const int start = __ldg(pad + lo);
        const int c = (__ldg(pad + lo + 1) - start) / (2 * world);  // chunk length
        const int u = p - start / world;                              // position in the rank's share
        out[p] = u < c ? start + rank * c + u : start + (2 * world - 1 - rank) * c + (u - c);
    }
}

}  // namespace

cudaError_t launch_partitioned_indices(const int *pad, int B, int world, int rank, int n_out, int *out,
                                       cudaStream_t st) {
    if (n_out <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    int blocks = (n_out + 255) / 256;
    if (blocks > sms * 4) blocks = sms * 4;  // grid-stride loop beyond four blocks per SM
    partitioned_indices_kernel<<<blocks, 256, 0, st>>>(pad, B, world, rank, n_out, out);
    return cudaGetLastError();
}

}  // namespace gbattn
