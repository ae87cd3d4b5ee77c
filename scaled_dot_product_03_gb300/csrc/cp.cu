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
// chunk r then of chunk 2 CP - 1 - r.  Also the row sums the emulated
// ring's backward accumulates its per-step gradients with.
#include "gbattn.h"
#include "launch.h"
#include "prof.h"

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

// Sums of the ring's per-step gradients (the backward of the ring: every
// step's attention backward, taken with the merged O and LSE, yields dQ of
// the rank's query chunk and dK, dV of the key/value chunk it holds, and the
// gradient is their sum over the steps).  One thread per 8 consecutive
// elements of a (row, head); rows inside a sequence are row pad[b] + i,
// i < L_b.  mode 0: acc += src (src in the element type); mode 2: acc = src;
// mode 1: dst = acc converted to the element type, and 0 on rows outside
// every sequence.  acc is [T, H, D] fp32, contiguous.
template <typename T>
__device__ __forceinline__ void load8(const T *p, float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const T *e = reinterpret_cast<const T *>(&u);
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = to_f32(e[i]);
}
template <>
__device__ __forceinline__ void load8<float>(const float *p, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
template <typename T>
__device__ __forceinline__ void store8(T *p, const float (&x)[8]) {
    uint4 u;
    T *e = reinterpret_cast<T *>(&u);
#pragma unroll
    for (int i = 0; i < 8; ++i) e[i] = from_f32<T>(x[i]);
    *reinterpret_cast<uint4 *>(p) = u;
}
template <>
__device__ __forceinline__ void store8<float>(float *p, const float (&x)[8]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}

template <typename T>
__global__ void __launch_bounds__(256)
    thd_rows_kernel(int mode, int64_t n_chunks, int H, int cpr, MutView v, float *__restrict__ acc,
                    const int *__restrict__ cu, const int *__restrict__ pad, int B) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_chunks;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t pair = i / cpr;  // (row, head)
        const int c = (int)(i - pair * cpr);
        const int64_t r = pair / H;
        const int h = (int)(pair - r * H);
        const bool in_seq = thd_row_in_sequence(cu, pad, B, (int)r);
        float *a = acc + pair * (int64_t)(cpr * 8) + c * 8;
        T *e = (T *)v.ptr + r * v.ss + (int64_t)h * v.sh + c * 8;
        float x[8];
        if (mode == 0) {
            if (!in_seq) continue;
            float y[8];
            load8<float>(a, x);
            load8<T>(e, y);
#pragma unroll
            for (int k = 0; k < 8; ++k) x[k] += y[k];
            store8<float>(a, x);
        } else if (mode == 2) {
            if (!in_seq) continue;
            load8<T>(e, x);
            store8<float>(a, x);
        } else {
            if (in_seq) {
                load8<float>(a, x);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) x[k] = 0.f;
            }
            store8<T>(e, x);
        }
    }
}

}  // namespace

cudaError_t launch_thd_rows(int dtype, int mode, int T_, int H, int D, const MutView &v, float *acc, const int *cu,
                            const int *pad, int B, cudaStream_t st) {
    const int64_t n_chunks = (int64_t)T_ * H * (D / 8);
    if (n_chunks <= 0) return cudaSuccess;
    int sms = 0;
    cudaError_t e = device_sm_count(&sms);
    if (e != cudaSuccess) return e;
    int64_t blocks = (n_chunks + 255) / 256;
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;  // grid-stride beyond eight blocks per SM
    prof_before(st, kProfThdRows);
    switch (dtype) {
        case 0: thd_rows_kernel<__half><<<(unsigned)blocks, 256, 0, st>>>(mode, n_chunks, H, D / 8, v, acc, cu, pad, B); break;
        case 1: thd_rows_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, st>>>(mode, n_chunks, H, D / 8, v, acc, cu, pad, B); break;
        case 2: thd_rows_kernel<float><<<(unsigned)blocks, 256, 0, st>>>(mode, n_chunks, H, D / 8, v, acc, cu, pad, B); break;
        default: prof_after(st); return cudaErrorInvalidValue;
    }
    prof_after(st);
    return cudaGetLastError();
}

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
