// merge.cu -- LSE merge of two partial attentions over disjoint key sets,
// and its backward.
//
// Restates merge_attn of "Significant Accuracy Difference between Compiled
// and Eager Flex Attention": with m = max(lse1, lse2), e_k = exp(lse_k - m),
//   o = (o1 e1 + o2 e2) / (e1 + e2),   lse = m + log(e1 + e2),
// in fp32, guarding the case where both sides saw no key (m = -inf).
//
// Streaming kernels, bound by HBM bandwidth: each row (b, s, h) is handled by
// a power-of-two group of lanes inside one warp, each lane moving 16-byte
// vectors of the row, so rows never straddle warps and an in-place update of
// the LSE (lse_out == lse1) is ordered after every lane has read it.  Each
// warp keeps several rows of loads in flight.
#include "launch.h"
#include "prof.h"

namespace gbattn {
namespace {

template <typename T, int VEC>
struct alignas(sizeof(T) * VEC) Vec {
    T v[VEC];
};

// Rows are visited in the order (b, s, h), the memory order of the usual
// (b, s, h, d) views, so consecutive warps stream consecutive rows of o; the
// LSE of row (b, s, h) sits at (b H + h) S + s, and the LSE arrays (4 bytes
// per row) are small enough to stay in L2 across their scattered accesses.
struct RowIdx {
    unsigned b, s, h, lse;
};
__device__ __forceinline__ RowIdx row_idx(unsigned q, const FastDiv &fS, const FastDiv &fH) {
    RowIdx x;
    const unsigned bs = fH.div(q);
    x.h = q - bs * fH.d;
    x.b = fS.div(bs);
    x.s = bs - x.b * fS.d;
    x.lse = (x.b * fH.d + x.h) * fS.d + x.s;
    return x;
}

// Row weights of the merge, exp(lse_k - m) normalised, with the hardware
// base-2 exponential (the weights enter an fp32 or narrower result).
__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
template <typename V>
__device__ __forceinline__ int64_t row_off(const V &v, const RowIdx &x) {
    return (int64_t)x.b * v.sb + (int64_t)x.s * v.ss + (int64_t)x.h * v.sh;
}

// A row is covered by tpr lanes (a power of two), each moving NV vectors of
// it: vector c0 + j tpr for j < NV (consecutive lanes, consecutive vectors).
// All loads of the row are issued before any store: the only overlap the
// interface allows (o_out == o1 or o2) is of the same element, which each
// lane reads before it writes.  NV = 0 is the fallback for long rows (lanes
// loop over the row's vectors).  32-bit index arithmetic (the launcher
// guarantees fewer than 2^31 rows).
template <typename T, int VEC, int NV>
__global__ void __launch_bounds__(256) merge_kernel(MergeArgs a, int tpr, FastDiv fS, FastDiv fH) {
    using Vt = Vec<T, VEC>;
    constexpr int NR = NV > 0 ? NV : 1;
    const int lane = threadIdx.x & 31;
    const int rows_per_warp = 32 / tpr;
    const int sub = lane / tpr, c0 = lane % tpr;
    const int vpr = a.D / VEC;  // vectors per row
    const unsigned rows = (unsigned)a.B * a.S * a.H;
    const unsigned nwarps = gridDim.x * (blockDim.x / 32);
    const unsigned step = nwarps * rows_per_warp;
    for (unsigned q = (blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * rows_per_warp + sub;
         q - sub < rows; q += step) {
        const bool act = q < rows;
        const RowIdx x = row_idx(act ? q : 0, fS, fH);
        float l1 = -INFINITY, l2 = -INFINITY;
        Vt x1[NR], x2[NR];
        if (act) {
            l1 = a.lse1[x.lse];
            l2 = a.lse2[x.lse];
            if (NV > 0) {
                const Vt *p1 = (const Vt *)((const T *)a.o1.ptr + row_off(a.o1, x));
                const Vt *p2 = (const Vt *)((const T *)a.o2.ptr + row_off(a.o2, x));
#pragma unroll
                for (int j = 0; j < NR; ++j) {
                    const int c = c0 + j * tpr;
                    if (c < vpr) {
                        x1[j] = p1[c];
                        x2[j] = p2[c];
                    }
                }
            }
        }
        const float mx = fmaxf(l1, l2);
        float w1 = 0.f, w2 = 0.f, lse = -INFINITY;
        if (mx != -INFINITY) {
            const float e1 = ex2f((l1 - mx) * kLog2e), e2 = ex2f((l2 - mx) * kLog2e);
            const float inv = __frcp_rn(e1 + e2);
            w1 = e1 * inv;
            w2 = e2 * inv;
            lse = mx + __log2f(e1 + e2) * kLn2;
        }
        if (act) {
            Vt *po = (Vt *)((T *)a.out.ptr + row_off(a.out, x));
            auto mix = [&](const Vt &y1, const Vt &y2) {
                Vt y;
#pragma unroll
                for (int e = 0; e < VEC; ++e) y.v[e] = from_f32<T>(to_f32(y1.v[e]) * w1 + to_f32(y2.v[e]) * w2);
                return y;
            };
            if (NV > 0) {
#pragma unroll
                for (int j = 0; j < NR; ++j) {
                    const int c = c0 + j * tpr;
                    if (c < vpr) po[c] = mix(x1[j], x2[j]);
                }
            } else {
                const Vt *p1 = (const Vt *)((const T *)a.o1.ptr + row_off(a.o1, x));
                const Vt *p2 = (const Vt *)((const T *)a.o2.ptr + row_off(a.o2, x));
                for (int c = c0; c < vpr; c += tpr) {
                    const Vt y1 = p1[c], y2 = p2[c];
                    po[c] = mix(y1, y2);
                }
            }
        }
        // every lane of the row has read lse1 / lse2 before one writes the
        // (possibly aliased) output
        __syncwarp();
        if (act && c0 == 0) a.lse_out[x.lse] = lse;
    }
}

// Backward of the merge for upstream gradients dO (and dLSE) of the merged
// row.  With w_k = exp(lse_k - lse) the merged o = w1 o1 + w2 o2, so
//   dO_k = w_k dO,   dLSE_k = w_k (<dO, o_k - o> + dLSE)
// where <dO, o1 - o> = w2 <dO, o1 - o2> and <dO, o2 - o> = -w1 <dO, o1 - o2>:
// one pass over the row accumulates <dO, o1 - o2> while writing dO_1, dO_2.
template <typename T, int VEC, int NV>
__global__ void __launch_bounds__(256) merge_bwd_kernel(MergeBwdArgs a, int tpr, FastDiv fS, FastDiv fH) {
    using Vt = Vec<T, VEC>;
    constexpr int NR = NV > 0 ? NV : 1;
    const int lane = threadIdx.x & 31;
    const int rows_per_warp = 32 / tpr;
    const int sub = lane / tpr, c0 = lane % tpr;
    const int vpr = a.D / VEC;
    const unsigned rows = (unsigned)a.B * a.S * a.H;
    const unsigned nwarps = gridDim.x * (blockDim.x / 32);
    const unsigned step = nwarps * rows_per_warp;
    for (unsigned q = (blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * rows_per_warp + sub;
         q - sub < rows; q += step) {
        const bool act = q < rows;
        const RowIdx x = row_idx(act ? q : 0, fS, fH);
        float l1 = -INFINITY, l2 = -INFINITY, gl = 0.f;
        Vt x1[NR], x2[NR], y[NR];
        if (act) {
            l1 = a.lse1[x.lse];
            l2 = a.lse2[x.lse];
            if (a.dlse) gl = a.dlse[x.lse];
            if (NV > 0) {
                const Vt *p1 = (const Vt *)((const T *)a.o1.ptr + row_off(a.o1, x));
                const Vt *p2 = (const Vt *)((const T *)a.o2.ptr + row_off(a.o2, x));
                const Vt *pd = (const Vt *)((const T *)a.dout.ptr + row_off(a.dout, x));
#pragma unroll
                for (int j = 0; j < NR; ++j) {
                    const int c = c0 + j * tpr;
                    if (c < vpr) {
                        x1[j] = p1[c];
                        x2[j] = p2[c];
                        y[j] = pd[c];
                    }
                }
            }
        }
        const float mx = fmaxf(l1, l2);
        float w1 = 0.f, w2 = 0.f;
        if (mx != -INFINITY) {
            const float e1 = ex2f((l1 - mx) * kLog2e), e2 = ex2f((l2 - mx) * kLog2e);
            const float inv = __frcp_rn(e1 + e2);
            w1 = e1 * inv;
            w2 = e2 * inv;
        }
        float acc = 0.f;  // <dO, o1 - o2>
        if (act) {
            Vt *q1 = (Vt *)((T *)a.do1.ptr + row_off(a.do1, x));
            Vt *q2 = (Vt *)((T *)a.do2.ptr + row_off(a.do2, x));
            auto one = [&](const Vt &v1, const Vt &v2, const Vt &dy, int c) {
                Vt z1, z2;
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float d = to_f32(dy.v[e]);
                    acc = fmaf(d, to_f32(v1.v[e]) - to_f32(v2.v[e]), acc);
                    z1.v[e] = from_f32<T>(w1 * d);
                    z2.v[e] = from_f32<T>(w2 * d);
                }
                q1[c] = z1;
                q2[c] = z2;
            };
            if (NV > 0) {
#pragma unroll
                for (int j = 0; j < NR; ++j) {
                    const int c = c0 + j * tpr;
                    if (c < vpr) one(x1[j], x2[j], y[j], c);
                }
            } else {
                const Vt *p1 = (const Vt *)((const T *)a.o1.ptr + row_off(a.o1, x));
                const Vt *p2 = (const Vt *)((const T *)a.o2.ptr + row_off(a.o2, x));
                const Vt *pd = (const Vt *)((const T *)a.dout.ptr + row_off(a.dout, x));
                for (int c = c0; c < vpr; c += tpr) one(p1[c], p2[c], pd[c], c);
            }
        }
        for (int off = tpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (act && c0 == 0) {
            a.dlse1[x.lse] = w1 * fmaf(w2, acc, gl);
            a.dlse2[x.lse] = w2 * fmaf(-w1, acc, gl);
        }
    }
}

// Lanes per row and vectors per lane for rows of vpr vectors: four vectors
// per lane when that leaves a power-of-two lane count of at most 32, else
// two, else one vector per lane (spare lanes idle), else (rows longer than
// 32 vectors of an odd count) lanes looping over the row.
struct RowSplit {
    int tpr, nv;
};
inline bool pow2_le32(int x) { return x >= 1 && x <= 32 && (x & (x - 1)) == 0; }
inline RowSplit row_split(int vpr) {
    if (vpr % 4 == 0 && pow2_le32(vpr / 4)) return {vpr / 4, 4};
    if (vpr % 2 == 0 && pow2_le32(vpr / 2)) return {vpr / 2, 2};
    int t = 1;
    while (t < vpr && t < 32) t *= 2;
    return {t, vpr <= t ? 1 : 0};
}

template <typename T, int VEC, typename Args, typename K1, typename K2, typename K4, typename K0>
cudaError_t launch_rows(const Args &a, int kind, K1 k1, K2 k2, K4 k4, K0 k0, cudaStream_t st) {
    const RowSplit rs = row_split(a.D / VEC);
    const int64_t rows = (int64_t)a.B * a.S * a.H;
    if (rows >= ((int64_t)1 << 31)) return cudaErrorInvalidConfiguration;
    int sms = 0;
    cudaError_t e = device_sm_count(&sms);
    if (e != cudaSuccess) return e;
    const int64_t per_warp = 32 / rs.tpr;
    const int64_t warps_needed = (rows + per_warp - 1) / per_warp;
    int64_t blocks = (warps_needed + 7) / 8;
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    if (blocks < 1) blocks = 1;
    const FastDiv fS(a.S), fH(a.H);
    prof_before(st, kind);
    switch (rs.nv) {
        case 4: k4<<<(int)blocks, 256, 0, st>>>(a, rs.tpr, fS, fH); break;
        case 2: k2<<<(int)blocks, 256, 0, st>>>(a, rs.tpr, fS, fH); break;
        case 1: k1<<<(int)blocks, 256, 0, st>>>(a, rs.tpr, fS, fH); break;
        default: k0<<<(int)blocks, 256, 0, st>>>(a, rs.tpr, fS, fH); break;
    }
    prof_after(st);
    return cudaGetLastError();
}

template <typename T, int VEC>
cudaError_t merge_bwd_typed(const MergeBwdArgs &a, cudaStream_t st) {
    return launch_rows<T, VEC>(a, kProfMergeBwd, merge_bwd_kernel<T, VEC, 1>, merge_bwd_kernel<T, VEC, 2>,
                               merge_bwd_kernel<T, VEC, 4>, merge_bwd_kernel<T, VEC, 0>, st);
}

template <typename T, int VEC>
cudaError_t merge_typed(const MergeArgs &a, cudaStream_t st) {
    return launch_rows<T, VEC>(a, kProfMerge, merge_kernel<T, VEC, 1>, merge_kernel<T, VEC, 2>,
                               merge_kernel<T, VEC, 4>, merge_kernel<T, VEC, 0>, st);
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
