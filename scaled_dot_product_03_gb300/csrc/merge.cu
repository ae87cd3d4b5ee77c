// merge.cu -- LSE merge of two partial attentions over disjoint key sets,
// and its backward.
//
// Restates merge_attn of "Significant Accuracy Difference between Compiled
// and Eager Flex Attention": with m = max(lse1, lse2), e_k = exp(lse_k - m),
//   o = (o1 e1 + o2 e2) / (e1 + e2),   lse = m + log(e1 + e2),
// in fp32, guarding the case where both sides saw no key (m = -inf).
//
// Streaming kernel, bound by HBM bandwidth: each row (b, s, h) is handled by
// a power-of-two group of lanes inside one warp, each lane moving 16-byte
// vectors of the row, so rows never straddle warps and an in-place update of
// the LSE (lse_out == lse1) is ordered after every lane has read it.
#include "launch.h"
#include "prof.h"

namespace gbattn {
namespace {

template <typename T, int VEC>
struct alignas(sizeof(T) * VEC) Vec {
    T v[VEC];
};

template <typename T, int VEC>
__global__ void __launch_bounds__(256) merge_kernel(MergeArgs a, int tpr) {
    const int lane = threadIdx.x & 31;
    const int rows_per_warp = 32 / tpr;
    const int sub = lane / tpr, c0 = lane % tpr;
    const int vpr = a.D / VEC;  // vectors per row
    const int64_t rows = (int64_t)a.B * a.S * a.H;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
         w * rows_per_warp < rows; w += warps) {
        const int64_t r = w * rows_per_warp + sub;  // row = ((b * H) + h) * S + s
        const bool active = r < rows;
        float l1 = -INFINITY, l2 = -INFINITY;
        int b = 0, h = 0, s = 0;
        if (active) {
            l1 = a.lse1[r];
            l2 = a.lse2[r];
            s = (int)(r % a.S);
            h = (int)((r / a.S) % a.H);
            b = (int)(r / ((int64_t)a.S * a.H));
        }
        const float mx = fmaxf(l1, l2);
        float w1 = 0.f, w2 = 0.f, lse = -INFINITY;
        if (mx != -INFINITY) {
            const float e1 = expf(l1 - mx), e2 = expf(l2 - mx);
            const float inv = 1.f / (e1 + e2);
            w1 = e1 * inv;
            w2 = e2 * inv;
            lse = mx + logf(e1 + e2);
        }
        if (active) {
            const T *p1 = (const T *)a.o1.ptr + b * a.o1.sb + s * a.o1.ss + h * a.o1.sh;
            const T *p2 = (const T *)a.o2.ptr + b * a.o2.sb + s * a.o2.ss + h * a.o2.sh;
            T *po = (T *)a.out.ptr + b * a.out.sb + s * a.out.ss + h * a.out.sh;
            for (int c = c0; c < vpr; c += tpr) {
                const Vec<T, VEC> x1 = ((const Vec<T, VEC> *)p1)[c];
                const Vec<T, VEC> x2 = ((const Vec<T, VEC> *)p2)[c];
                Vec<T, VEC> y;
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    y.v[e] = from_f32<T>(to_f32(x1.v[e]) * w1 + to_f32(x2.v[e]) * w2);
                ((Vec<T, VEC> *)po)[c] = y;
            }
        }
        __syncwarp();
        if (active && c0 == 0) a.lse_out[r] = lse;
    }
}

// Backward of the merge for upstream gradients dO (and dLSE) of the merged
// row.  With w_k = exp(lse_k - lse) the merged o = w1 o1 + w2 o2, so
//   dO_k = w_k dO,   dLSE_k = w_k (<dO, o_k - o> + dLSE)
// where <dO, o1 - o> = w2 <dO, o1 - o2> and <dO, o2 - o> = -w1 <dO, o1 - o2>:
// one pass over the row accumulates <dO, o1 - o2> while writing dO_1, dO_2.
template <typename T, int VEC>
__global__ void __launch_bounds__(256) merge_bwd_kernel(MergeBwdArgs a, int tpr) {
    const int lane = threadIdx.x & 31;
    const int rows_per_warp = 32 / tpr;
    const int sub = lane / tpr, c0 = lane % tpr;
    const int vpr = a.D / VEC;
    const int64_t rows = (int64_t)a.B * a.S * a.H;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
         w * rows_per_warp < rows; w += warps) {
        const int64_t r = w * rows_per_warp + sub;  // row = ((b * H) + h) * S + s
        const bool active = r < rows;
        float l1 = -INFINITY, l2 = -INFINITY, g = 0.f;
        int b = 0, h = 0, s = 0;
        if (active) {
            l1 = a.lse1[r];
            l2 = a.lse2[r];
            if (a.dlse) g = a.dlse[r];
            s = (int)(r % a.S);
            h = (int)((r / a.S) % a.H);
            b = (int)(r / ((int64_t)a.S * a.H));
        }
        const float mx = fmaxf(l1, l2);
        float w1 = 0.f, w2 = 0.f;
        if (mx != -INFINITY) {
            const float e1 = expf(l1 - mx), e2 = expf(l2 - mx);
            const float inv = 1.f / (e1 + e2);
            w1 = e1 * inv;
            w2 = e2 * inv;
        }
        float acc = 0.f;  // <dO, o1 - o2>
        if (active) {
            const T *p1 = (const T *)a.o1.ptr + b * a.o1.sb + s * a.o1.ss + h * a.o1.sh;
            const T *p2 = (const T *)a.o2.ptr + b * a.o2.sb + s * a.o2.ss + h * a.o2.sh;
            const T *pd = (const T *)a.dout.ptr + b * a.dout.sb + s * a.dout.ss + h * a.dout.sh;
            T *q1 = (T *)a.do1.ptr + b * a.do1.sb + s * a.do1.ss + h * a.do1.sh;
            T *q2 = (T *)a.do2.ptr + b * a.do2.sb + s * a.do2.ss + h * a.do2.sh;
            for (int c = c0; c < vpr; c += tpr) {
                const Vec<T, VEC> x1 = ((const Vec<T, VEC> *)p1)[c];
                const Vec<T, VEC> x2 = ((const Vec<T, VEC> *)p2)[c];
                const Vec<T, VEC> y = ((const Vec<T, VEC> *)pd)[c];
                Vec<T, VEC> z1, z2;
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float dy = to_f32(y.v[e]);
                    acc = fmaf(dy, to_f32(x1.v[e]) - to_f32(x2.v[e]), acc);
                    z1.v[e] = from_f32<T>(w1 * dy);
                    z2.v[e] = from_f32<T>(w2 * dy);
                }
                ((Vec<T, VEC> *)q1)[c] = z1;
                ((Vec<T, VEC> *)q2)[c] = z2;
            }
        }
        for (int off = tpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (active && c0 == 0) {
            a.dlse1[r] = w1 * fmaf(w2, acc, g);
            a.dlse2[r] = w2 * fmaf(-w1, acc, g);
        }
    }
}

template <typename T, int VEC>
cudaError_t merge_bwd_typed(const MergeBwdArgs &a, cudaStream_t st) {
    const int vpr = a.D / VEC;
    int tpr = 1;
    while (tpr < vpr && tpr < 32) tpr *= 2;
    const int64_t rows = (int64_t)a.B * a.S * a.H;
    const int64_t warps_needed = (rows + (32 / tpr) - 1) / (32 / tpr);
    int64_t blocks = (warps_needed + 7) / 8;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    prof_before(st, kProfMergeBwd);
    merge_bwd_kernel<T, VEC><<<(int)blocks, 256, 0, st>>>(a, tpr);
    prof_after(st);
    return cudaGetLastError();
}

template <typename T, int VEC>
cudaError_t merge_typed(const MergeArgs &a, cudaStream_t st) {
    const int vpr = a.D / VEC;
    int tpr = 1;
    while (tpr < vpr && tpr < 32) tpr *= 2;
    const int64_t rows = (int64_t)a.B * a.S * a.H;
    const int64_t warps_needed = (rows + (32 / tpr) - 1) / (32 / tpr);
    int64_t blocks = (warps_needed + 7) / 8;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    prof_before(st, kProfMerge);
    merge_kernel<T, VEC><<<(int)blocks, 256, 0, st>>>(a, tpr);
    prof_after(st);
    return cudaGetLastError();
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

template <typename V>
bool view_vec_ok(const V &v, int vec) {
    return aligned16(v.ptr) && (v.sb % vec) == 0 && (v.ss % vec) == 0 && (v.sh % vec) == 0;
}

}  // namespace

cudaError_t launch_merge(int dtype, const MergeArgs &a, cudaStream_t st) {
    const size_t elt = dtype == 2 ? 4 : 2;
    const int vec = (int)(16 / elt);
    bool vec_ok = (a.D % vec) == 0 && aligned16(a.o1.ptr) && aligned16(a.o2.ptr) &&
                  aligned16(a.out.ptr);
    const View *vs[2] = {&a.o1, &a.o2};
    for (const View *v : vs)
        vec_ok = vec_ok && (v->sb % vec) == 0 && (v->ss % vec) == 0 && (v->sh % vec) == 0;
    vec_ok = vec_ok && (a.out.sb % vec) == 0 && (a.out.ss % vec) == 0 && (a.out.sh % vec) == 0;
    switch (dtype) {
        case 0: return vec_ok ? merge_typed<__half, 8>(a, st) : merge_typed<__half, 1>(a, st);
        case 1: return vec_ok ? merge_typed<__nv_bfloat16, 8>(a, st)
                              : merge_typed<__nv_bfloat16, 1>(a, st);
        case 2: return vec_ok ? merge_typed<float, 4>(a, st) : merge_typed<float, 1>(a, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_merge_bwd(int dtype, const MergeBwdArgs &a, cudaStream_t st) {
    const size_t elt = dtype == 2 ? 4 : 2;
    const int vec = (int)(16 / elt);
    const bool vec_ok = (a.D % vec) == 0 && view_vec_ok(a.o1, vec) && view_vec_ok(a.o2, vec) &&
                        view_vec_ok(a.dout, vec) && view_vec_ok(a.do1, vec) && view_vec_ok(a.do2, vec);
    switch (dtype) {
        case 0: return vec_ok ? merge_bwd_typed<__half, 8>(a, st) : merge_bwd_typed<__half, 1>(a, st);
        case 1: return vec_ok ? merge_bwd_typed<__nv_bfloat16, 8>(a, st)
                              : merge_bwd_typed<__nv_bfloat16, 1>(a, st);
        case 2: return vec_ok ? merge_bwd_typed<float, 4>(a, st) : merge_bwd_typed<float, 1>(a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gbattn
