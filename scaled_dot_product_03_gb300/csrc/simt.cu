// simt.cu -- FFMA (CUDA-core) attention kernels.
//
// This is the fp32 path: "Significant Accuracy Difference between Compiled
// and Eager Flex Attention" traces its fp32 error to kernels that used
// tensor cores "by default" for fp32 inputs, so fp32 inputs are computed
// here with plain fp32 fused multiply-adds and never reach a tensor core.
// Every kernel also accepts fp16/bf16 inputs (converted to fp32 on load).
//
// Forward: one lane per query row and the rows' keys split over the CTA's
// warps, each with an online softmax over its key blocks (an exact rewrite of
// the two-pass softmax), the warps' partial results combined at the end.
// Backward: the row term delta_i = <dO_i, O_i> first, then one kernel for dq
// (lane per query row, keys split over warps) and one for dk/dv (four threads
// per key, the query blocks of the group's heads split over thread groups),
// each recomputing P from the saved LSE and summing partials in shared
// memory.
#include "launch.h"
#include "prof.h"

namespace gbattn {
namespace {

constexpr int kThreads = 128;

// Barrier among `n` threads (a multiple of 32) on named barrier `id` (1-15).
__device__ __forceinline__ void ptx_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <typename T>
__device__ __forceinline__ const T *row_ptr(const View &v, int b, int row, int h) {
    return (const T *)v.ptr + (int64_t)b * v.sb + (int64_t)row * v.ss + (int64_t)h * v.sh;
}
template <typename T>
__device__ __forceinline__ T *row_ptr(const MutView &v, int b, int row, int h) {
    return (T *)v.ptr + (int64_t)b * v.sb + (int64_t)row * v.ss + (int64_t)h * v.sh;
}

// ---------------------------------------------------------------------------
// Work split of the query-row kernels (forward and dq): a CTA takes kRows
// query rows (lane = row) and kSplits warps; warp w walks key blocks
// w, w + kSplits, ... of the rows' key range, staging each block of BN keys
// in its own slice of shared memory, and the warps' partial results are
// combined through shared memory at the end.  Splitting the keys over warps
// (rather than one thread per row over all keys) puts kSplits times more
// warps on short problems such as the page-3 workload.
constexpr int kRows = 32;
constexpr int kSplits = 8;
constexpr int kSplitThreads = kRows * kSplits;
constexpr int kBN = 16;  // keys per block and warp

// Forward.  grid (ceil(max Lq / kRows), Hq, B), kSplitThreads threads.
// smem: Q^T [D][kRows] (lane-consecutive reads), per warp a K and a V block
// [kBN][D]; afterwards the partial (m, l, o) of every warp.  Each warp keeps
// an online softmax over its blocks (an exact rewrite of the two-pass
// softmax); the combination rescales the partials by exp2(m_w - max m).
template <typename T, int D>
__global__ void __launch_bounds__(kSplitThreads) simt_fwd_kernel(FwdArgs a) {
    extern __shared__ float smem[];
    float *Qs = smem, *KV = Qs + D * kRows;
    const Geometry &g = a.g;
    const int b = blockIdx.z, h = blockIdx.y, m0 = blockIdx.x * kRows, tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;
    const SeqInfo s = seq_info(g, b);
    if (blockIdx.x == gridDim.x - 1 && tid == 0) report_uncovered(a.err, g, s.Lq, gridDim.x * kRows, kErrSeqlenQ);
    if (m0 >= s.Lq) return;
    const int hk = h / g.G, i = m0 + lane;
    for (int e = tid; e < kRows * D; e += kSplitThreads) {
        const int r = e / D, d = e % D;
        float x = 0.f;
        if (m0 + r < s.Lq) x = to_f32(row_ptr<T>(a.q, b, s.q0 + m0 + r, h)[d]);
        Qs[d * kRows + r] = x;
    }
    int jlo, jhi;
    key_range(m0, min(m0 + kRows, s.Lq), s.Lkv, g.wl, g.wr, jlo, jhi);
    const int nblk = (jhi - jlo + kBN - 1) / kBN;
    __syncthreads();
    float *Ks = KV + warp * 2 * kBN * D, *Vs = Ks + kBN * D;
    float m = -INFINITY, l = 0.f, o[D];
#pragma unroll
    for (int d = 0; d < D; ++d) o[d] = 0.f;
    for (int bi = warp; bi < nblk; bi += kSplits) {
        const int j0 = jlo + bi * kBN;
        __syncwarp();
        for (int e = lane; e < kBN * D; e += 32) {
            const int r = e / D, d = e % D, j = j0 + r;
            float kx = 0.f, vx = 0.f;
            if (j < jhi) {
                kx = to_f32(row_ptr<T>(a.k, b, s.kv0 + j, hk)[d]);
                vx = to_f32(row_ptr<T>(a.v, b, s.kv0 + j, hk)[d]);
            }
            Ks[e] = kx;
            Vs[e] = vx;
        }
        __syncwarp();
        float sc[kBN];
#pragma unroll
        for (int jj = 0; jj < kBN; ++jj) sc[jj] = 0.f;
#pragma unroll 4
        for (int d = 0; d < D; ++d) {
            const float qd = Qs[d * kRows + lane];
#pragma unroll
            for (int jj = 0; jj < kBN; ++jj) sc[jj] = fmaf(qd, Ks[jj * D + d], sc[jj]);
        }
        float mx = m;
#pragma unroll
        for (int jj = 0; jj < kBN; ++jj) {
            const int j = j0 + jj;
            const bool vis = i < s.Lq && j < jhi && visible(i, j, s.Lkv, g.wl, g.wr);
            if (!vis) sc[jj] = -INFINITY;
            else mx = fmaxf(mx, sc[jj] * g.scale_log2);
        }
        if (mx == -INFINITY) continue;  // nothing visible yet for this row
        const float alpha = exp2f(m - mx);
        l *= alpha;
#pragma unroll
        for (int d = 0; d < D; ++d) o[d] *= alpha;
#pragma unroll
        for (int jj = 0; jj < kBN; ++jj) {
            const float p = sc[jj] == -INFINITY ? 0.f : exp2f(fmaf(sc[jj], g.scale_log2, -mx));
            l += p;
            sc[jj] = p;
        }
#pragma unroll
        for (int jj = 0; jj < kBN; ++jj) {
#pragma unroll
            for (int d = 0; d < D; ++d) o[d] = fmaf(sc[jj], Vs[jj * D + d], o[d]);
        }
        m = mx;
    }
    // partials of every warp: o^T [kSplits][D][kRows], m and l [kSplits][kRows]
    __syncthreads();
    float *Op = KV, *Mp = Op + kSplits * D * kRows, *Lp = Mp + kSplits * kRows;
#pragma unroll
    for (int d = 0; d < D; ++d) Op[(warp * D + d) * kRows + lane] = o[d];
    Mp[warp * kRows + lane] = m;
    Lp[warp * kRows + lane] = l;
    __syncthreads();
    // thread (warp, lane): row lane, head dims [warp D / kSplits, (warp + 1) D / kSplits)
    float mt = -INFINITY;
#pragma unroll
    for (int w = 0; w < kSplits; ++w) mt = fmaxf(mt, Mp[w * kRows + lane]);
    float wt[kSplits], lt = 0.f;
#pragma unroll
    for (int w = 0; w < kSplits; ++w) {
        const float mw = Mp[w * kRows + lane];
        wt[w] = mw == -INFINITY ? 0.f : exp2f(mw - mt);
        lt = fmaf(Lp[w * kRows + lane], wt[w], lt);
    }
    if (i < s.Lq) {
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        T *orow = row_ptr<T>(a.o, b, s.q0 + i, h);
        constexpr int DS = D / kSplits;
#pragma unroll 8
        for (int e = 0; e < DS; ++e) {
            const int d = warp * DS + e;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < kSplits; ++w) acc = fmaf(Op[(w * D + d) * kRows + lane], wt[w], acc);
            orow[d] = from_f32<T>(acc * inv);
        }
        if (warp == 0) a.lse[lse_index(g, s, b, h, i)] = lt > 0.f ? (mt + log2f(lt)) * kLn2 : -INFINITY;
    }
}

// ---------------------------------------------------------------------------
// Lanes that share one row: the largest power of two (the group is reduced
// with xor shuffles and must tile the warp) not above the row's chunks,
// at most 32; lanes loop over the remaining chunks.
__host__ __device__ inline int lanes_per_row(int chunks) {
    int t = 1;
    while (t * 2 <= chunks && t < 32) t *= 2;
    return t;
}

// Backward preprocess: delta = <dO, O> - dLSE per (row, head) (dLSE = 0 when
// no LSE gradient is given).  A group of up to 32
// lanes (power of two) covers one (row, head), each lane VEC elements at a
// time.  Also clears the fp32 dq accumulator (laid out like LSE, D floats per
// row) and the work counter of the persistent single pass when the backward
// uses them.
template <typename T, int VEC>
__global__ void bwd_preprocess_kernel(BwdArgs a, int rows) {
    struct alignas(sizeof(T) * VEC) Vt { T v[VEC]; };
    const Geometry &g = a.g;
    // (launched as a dependent of the previous kernel: wait for it, then let
    // the backward's next kernel begin launching)
    griddep_wait();
    griddep_launch();
    if (a.work_ctr && blockIdx.x == 0 && threadIdx.x == 0) *a.work_ctr = 0u;
    const int D = g.D;
    const int chunks = D / VEC;
    const int tpr = lanes_per_row(chunks);
    const int lane = threadIdx.x & 31, sub = lane / tpr, c0 = lane % tpr;
    const int per_warp = 32 / tpr;
    const int64_t pairs = (int64_t)rows * g.Hq;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
         w * per_warp < pairs; w += nwarps) {
        const int64_t pr = w * per_warp + sub;
        const bool active = pr < pairs;
        float acc = 0.f;
        int64_t idx = 0;
        if (active) {
            const int r = (int)(pr / g.Hq), h = (int)(pr % g.Hq);
            int b = 0, row = r;
            if (g.thd) {
                idx = (int64_t)h * g.Tq + r;
            } else {
                b = r / g.Sq;
                row = r % g.Sq;
                idx = ((int64_t)b * g.Hq + h) * g.Sq + row;
            }
            const Vt *o = reinterpret_cast<const Vt *>(row_ptr<T>(a.o, b, row, h));
            const Vt *d_o = reinterpret_cast<const Vt *>(row_ptr<T>(a.dout, b, row, h));
            // (the accumulator rows are acc_d floats apart; columns past D
            // are padding that is never read)
            float *acc_row = a.dq_acc ? a.dq_acc + idx * a.acc_d : nullptr;
            for (int c = c0; c < chunks; c += tpr) {
                const Vt x = o[c], y = d_o[c];
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc = fmaf(to_f32(x.v[e]), to_f32(y.v[e]), acc);
                if (acc_row) {
                    if (VEC % 4 == 0) {
#pragma unroll
                        for (int e = 0; e < VEC; e += 4)
                            *reinterpret_cast<float4 *>(acc_row + c * VEC + e) = make_float4(0.f, 0.f, 0.f, 0.f);
                    } else {
#pragma unroll
                        for (int e = 0; e < VEC; ++e) acc_row[c * VEC + e] = 0.f;
                    }
                }
            }
        }
        for (int off = tpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        // a gradient reaching LSE adds P_ij dLSE_i to dS_ij, i.e. lowers the
        // row term by dLSE_i
        if (active && c0 == 0) a.delta[idx] = a.dlse ? acc - a.dlse[idx] : acc;
    }
}

// The same for 16-bit O and dO with the head dim fixed at compile time: a
// row is covered by LPR lanes moving one 16-byte vector of O and of dO each
// (LPR = D / 8 rounded up to a power of two; the spare lanes of D = 96 idle),
// and every warp keeps U row groups in flight before it reduces any, so each
// lane has U pairs of loads outstanding.  Index arithmetic is 32-bit (the
// launcher guarantees fewer than 2^31 (row, head) pairs).
template <typename T, int D, int U>
__global__ void __launch_bounds__(256) bwd_preprocess16_kernel(BwdArgs a, int rows, FastDiv fHq, FastDiv fSq) {
    constexpr int NV = D / 8;                              // 16-byte vectors per row
    constexpr int LPR = NV <= 4 ? 4 : NV <= 8 ? 8 : 16;   // lanes per row
    constexpr int RPW = 32 / LPR;                         // rows per warp and group
    const Geometry &g = a.g;
    griddep_wait();
    griddep_launch();
    if (a.work_ctr && blockIdx.x == 0 && threadIdx.x == 0) *a.work_ctr = 0u;
    const int lane = threadIdx.x & 31, sub = lane / LPR, c = lane % LPR;
    const unsigned pairs = (unsigned)rows * (unsigned)g.Hq;
    const unsigned nwarps = gridDim.x * (blockDim.x / 32);
    for (unsigned base = (blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * (RPW * U); base < pairs;
         base += nwarps * (RPW * U)) {
        uint4 x[U], y[U];
        unsigned idx[U];
        bool act[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const unsigned pr = base + u * RPW + sub;
            act[u] = pr < pairs;
            x[u] = y[u] = make_uint4(0, 0, 0, 0);
            idx[u] = 0;
            if (act[u]) {
                const unsigned r = fHq.div(pr), h = pr - r * (unsigned)g.Hq;
                unsigned b = 0, row = r;
                if (g.thd) {
                    idx[u] = h * (unsigned)g.Tq + r;
                } else {
                    b = fSq.div(r);
                    row = r - b * (unsigned)g.Sq;
                    idx[u] = (b * (unsigned)g.Hq + h) * (unsigned)g.Sq + row;
                }
                if (c < NV) {
                    x[u] = reinterpret_cast<const uint4 *>(row_ptr<T>(a.o, b, row, h))[c];
                    y[u] = reinterpret_cast<const uint4 *>(row_ptr<T>(a.dout, b, row, h))[c];
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const T *xv = reinterpret_cast<const T *>(&x[u]);
            const T *yv = reinterpret_cast<const T *>(&y[u]);
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc = fmaf(to_f32(xv[e]), to_f32(yv[e]), acc);
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (act[u]) {
                if (a.dq_acc && c < NV) {
                    float4 *z = reinterpret_cast<float4 *>(a.dq_acc + (size_t)idx[u] * a.acc_d + c * 8);
                    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
                    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                // a gradient reaching LSE adds P_ij dLSE_i to dS_ij, i.e.
                // lowers the row term by dLSE_i
                if (c == 0) a.delta[idx[u]] = a.dlse ? acc - a.dlse[idx[u]] : acc;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Backward dq, with the work split of the forward: grid (ceil(max Lq /
// kRows), Hq, B), kSplitThreads threads; lane = query row, warps split the
// keys; smem Q^T and dO^T [D][kRows], per warp a K and a V block, then the
// warps' partial dq [kSplits][D][kRows], summed at the end.
template <typename T, int D>
__global__ void __launch_bounds__(kSplitThreads) simt_bwd_dq_kernel(BwdArgs a) {
    extern __shared__ float smem[];
    float *Qs = smem, *Os = Qs + D * kRows, *KV = Os + D * kRows;
    const Geometry &g = a.g;
    const int b = blockIdx.z, h = blockIdx.y, m0 = blockIdx.x * kRows, tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;
    const SeqInfo s = seq_info(g, b);
    if (blockIdx.x == gridDim.x - 1 && tid == 0) report_uncovered(a.err, g, s.Lq, gridDim.x * kRows, kErrSeqlenQ);
    if (m0 >= s.Lq) return;
    const int hk = h / g.G, i = m0 + lane;
    for (int e = tid; e < kRows * D; e += kSplitThreads) {
        const int r = e / D, d = e % D;
        float x = 0.f, y = 0.f;
        if (m0 + r < s.Lq) {
            x = to_f32(row_ptr<T>(a.q, b, s.q0 + m0 + r, h)[d]);
            y = to_f32(row_ptr<T>(a.dout, b, s.q0 + m0 + r, h)[d]);
        }
        Qs[d * kRows + r] = x;
        Os[d * kRows + r] = y;  // dO^T
    }
    float lse_l2 = 0.f, delta = 0.f;
    if (i < s.Lq) {
        const int64_t li = lse_index(g, s, b, h, i);
        lse_l2 = a.lse[li] * kLog2e;
        delta = a.delta[li];
    }
    int jlo, jhi;
    key_range(m0, min(m0 + kRows, s.Lq), s.Lkv, g.wl, g.wr, jlo, jhi);
    const int nblk = (jhi - jlo + kBN - 1) / kBN;
    __syncthreads();
    float *Ks = KV + warp * 2 * kBN * D, *Vs = Ks + kBN * D;
    float dq[D];
#pragma unroll
    for (int d = 0; d < D; ++d) dq[d] = 0.f;
    for (int bi = warp; bi < nblk; bi += kSplits) {
        const int j0 = jlo + bi * kBN;
        __syncwarp();
        for (int e = lane; e < kBN * D; e += 32) {
            const int r = e / D, d = e % D, j = j0 + r;
            float kx = 0.f, vx = 0.f;
            if (j < jhi) {
                kx = to_f32(row_ptr<T>(a.k, b, s.kv0 + j, hk)[d]);
                vx = to_f32(row_ptr<T>(a.v, b, s.kv0 + j, hk)[d]);
            }
            Ks[e] = kx;
            Vs[e] = vx;
        }
        __syncwarp();
        float sc[kBN], dp[kBN];
#pragma unroll
        for (int jj = 0; jj < kBN; ++jj) sc[jj] = dp[jj] = 0.f;
#pragma unroll 4
        for (int d = 0; d < D; ++d) {
            const float qd = Qs[d * kRows + lane], od = Os[d * kRows + lane];
#pragma unroll
            for (int jj = 0; jj < kBN; ++jj) {
                sc[jj] = fmaf(qd, Ks[jj * D + d], sc[jj]);
                dp[jj] = fmaf(od, Vs[jj * D + d], dp[jj]);
            }
        }
#pragma unroll
        for (int jj = 0; jj < kBN; ++jj) {
            const int j = j0 + jj;
            float ds = 0.f;
            if (i < s.Lq && j < jhi && visible(i, j, s.Lkv, g.wl, g.wr)) {
                const float p = exp2f(fmaf(sc[jj], g.scale_log2, -lse_l2));
                ds = p * (dp[jj] - delta);
            }
            sc[jj] = ds;
        }
#pragma unroll
        for (int jj = 0; jj < kBN; ++jj) {
#pragma unroll
            for (int d = 0; d < D; ++d) dq[d] = fmaf(sc[jj], Ks[jj * D + d], dq[d]);
        }
    }
    __syncthreads();
    float *Qp = KV;  // [kSplits][D][kRows]
#pragma unroll
    for (int d = 0; d < D; ++d) Qp[(warp * D + d) * kRows + lane] = dq[d];
    __syncthreads();
    if (i < s.Lq) {
        T *row = row_ptr<T>(a.dq, b, s.q0 + i, h);
        constexpr int DS = D / kSplits;
#pragma unroll 8
        for (int e = 0; e < DS; ++e) {
            const int d = warp * DS + e;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < kSplits; ++w) acc += Qp[(w * D + d) * kRows + lane];
            row[d] = from_f32<T>(acc * g.scale);
        }
    }
}

// ---------------------------------------------------------------------------
// Backward dk, dv: four threads per key (thread part p owns d = p, p + 4,
// ...), kKeys keys per CTA, and kGroups groups of such threads that split
// the (query head, query block) pairs of the keys' group between them, each
// staging its own query blocks of kQB rows; the groups' partial dk and dv
// are summed through shared memory at the end.
constexpr int kKeys = 16;
constexpr int kGroups = 4;
constexpr int kQB = 16;
constexpr int kKvThreads = kKeys * 4 * kGroups;

template <typename T, int D>
__global__ void __launch_bounds__(kKvThreads) simt_bwd_dkdv_kernel(BwdArgs a) {
    constexpr int DP = D / 4;
    constexpr int kGroupFloats = 2 * kQB * D + 2 * kQB;  // Q, dO, lse, delta of one group
    extern __shared__ float smem[];
    const Geometry &g = a.g;
    const int b = blockIdx.z, hk = blockIdx.y, n0 = blockIdx.x * kKeys, tid = threadIdx.x;
    const int grp = tid / (kKeys * 4), gt = tid % (kKeys * 4);
    float *Qs = smem + grp * kGroupFloats, *Os = Qs + kQB * D, *Ls = Os + kQB * D, *Ds = Ls + kQB;
    const SeqInfo s = seq_info(g, b);
    if (blockIdx.x == gridDim.x - 1 && tid == 0)
        report_uncovered(a.err, g, s.Lkv, gridDim.x * kKeys, kErrSeqlenKv);
    if (n0 >= s.Lkv) return;
    const int kt = gt / 4, part = gt % 4, j = n0 + kt;
    float kr[DP], vr[DP], dk[DP], dv[DP];
#pragma unroll
    for (int t = 0; t < DP; ++t) {
        kr[t] = vr[t] = dk[t] = dv[t] = 0.f;
        if (j < s.Lkv) {
            kr[t] = to_f32(row_ptr<T>(a.k, b, s.kv0 + j, hk)[4 * t + part]);
            vr[t] = to_f32(row_ptr<T>(a.v, b, s.kv0 + j, hk)[4 * t + part]);
        }
    }
    int ilo, ihi;
    query_range(n0, min(n0 + kKeys, s.Lkv), s.Lq, g.wl, g.wr, ilo, ihi);
    const int nqb = (ihi - ilo + kQB - 1) / kQB;
    const int n_pairs = nqb * g.G;
    for (int t0 = grp; t0 < n_pairs; t0 += kGroups) {
        const int h = hk * g.G + t0 / nqb, i0 = ilo + (t0 % nqb) * kQB;
        ptx_bar_sync(1 + grp, kKeys * 4);  // the group's previous block is read
        for (int e = gt; e < kQB * D; e += kKeys * 4) {
            const int r = e / D, d = e % D, i = i0 + r;
            float x = 0.f, y = 0.f;
            if (i < ihi) {
                x = to_f32(row_ptr<T>(a.q, b, s.q0 + i, h)[d]);
                y = to_f32(row_ptr<T>(a.dout, b, s.q0 + i, h)[d]);
            }
            Qs[e] = x;
            Os[e] = y;
        }
        for (int r = gt; r < kQB; r += kKeys * 4) {
            const int i = i0 + r;
            float lv = 0.f, dv_ = 0.f;
            if (i < ihi) {
                const int64_t li = lse_index(g, s, b, h, i);
                lv = a.lse[li] * kLog2e;
                dv_ = a.delta[li];
            }
            Ls[r] = lv;
            Ds[r] = dv_;
        }
        ptx_bar_sync(1 + grp, kKeys * 4);
        for (int r = 0; r < kQB; ++r) {
            const int i = i0 + r;
            float sp = 0.f, dpp = 0.f;
#pragma unroll
            for (int t = 0; t < DP; ++t) {
                sp = fmaf(Qs[r * D + 4 * t + part], kr[t], sp);
                dpp = fmaf(Os[r * D + 4 * t + part], vr[t], dpp);
            }
            sp += __shfl_xor_sync(0xffffffffu, sp, 1);
            sp += __shfl_xor_sync(0xffffffffu, sp, 2);
            dpp += __shfl_xor_sync(0xffffffffu, dpp, 1);
            dpp += __shfl_xor_sync(0xffffffffu, dpp, 2);
            if (i < ihi && visible(i, j, s.Lkv, g.wl, g.wr)) {
                const float p = exp2f(fmaf(sp, g.scale_log2, -Ls[r]));
                const float ds = p * (dpp - Ds[r]);
#pragma unroll
                for (int t = 0; t < DP; ++t) {
                    dv[t] = fmaf(p, Os[r * D + 4 * t + part], dv[t]);
                    dk[t] = fmaf(ds, Qs[r * D + 4 * t + part], dk[t]);
                }
            }
        }
    }
    // partials of every group: dk and dv [kGroups][kKeys][D]
    __syncthreads();
    float *Kp = smem, *Vp = Kp + kGroups * kKeys * D;
#pragma unroll
    for (int t = 0; t < DP; ++t) {
        Kp[(grp * kKeys + kt) * D + 4 * t + part] = dk[t];
        Vp[(grp * kKeys + kt) * D + 4 * t + part] = dv[t];
    }
    __syncthreads();
    for (int e = tid; e < kKeys * D; e += kKvThreads) {
        const int key = e / D, d = e % D, jj = n0 + key;
        if (jj >= s.Lkv) continue;
        float sk = 0.f, sv = 0.f;
#pragma unroll
        for (int w = 0; w < kGroups; ++w) {
            sk += Kp[(w * kKeys + key) * D + d];
            sv += Vp[(w * kKeys + key) * D + d];
        }
        row_ptr<T>(a.dk, b, s.kv0 + jj, hk)[d] = from_f32<T>(sk * g.scale);
        row_ptr<T>(a.dv, b, s.kv0 + jj, hk)[d] = from_f32<T>(sv);
    }
}

template <int D> constexpr size_t fwd_smem() {
    // Q^T, then the larger of the warps' K / V blocks and their partials
    return sizeof(float) * (D * kRows + (kSplits * D * kRows + 2 * kSplits * kRows > kSplits * 2 * kBN * D
                                             ? kSplits * D * kRows + 2 * kSplits * kRows
                                             : kSplits * 2 * kBN * D));
}
template <int D> constexpr size_t dq_smem() {
    return sizeof(float) * (2 * D * kRows + (kSplits * D * kRows > kSplits * 2 * kBN * D ? kSplits * D * kRows
                                                                                        : kSplits * 2 * kBN * D));
}
template <int D> constexpr size_t dkdv_smem() {
    constexpr size_t groups = (size_t)kGroups * (2 * kQB * D + 2 * kQB);
    constexpr size_t parts = (size_t)2 * kGroups * kKeys * D;
    return sizeof(float) * (groups > parts ? groups : parts);
}

template <typename T, int D>
cudaError_t fwd_typed(const FwdArgs &a, int max_lq, cudaStream_t st) {
    constexpr size_t smem = fwd_smem<D>();
    auto k = simt_fwd_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((max_lq + kRows - 1) / kRows, a.g.Hq, a.g.B);
    prof_before(st, kProfSimtFwd);
    k<<<grid, kSplitThreads, smem, st>>>(a);
    prof_after(st);
    return cudaGetLastError();
}

cudaError_t preprocess_any(int dtype, const BwdArgs &a, int rows, cudaStream_t st);

template <typename T, int D>
cudaError_t bwd_typed(int dtype, const BwdArgs &a, int max_lq, int max_lkv, int q_rows, cudaStream_t st) {
    constexpr size_t smem_dq = dq_smem<D>();
    constexpr size_t smem_kv = dkdv_smem<D>();
    auto kq = simt_bwd_dq_kernel<T, D>;
    auto kkv = simt_bwd_dkdv_kernel<T, D>;
    // kernel attributes first, so that a refusal enqueues nothing
    cudaError_t e;
    if (max_lq > 0 &&
        (e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_dq)) != cudaSuccess)
        return e;
    if (max_lkv > 0 &&
        (e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_kv)) != cudaSuccess)
        return e;
    if ((e = preprocess_any(dtype, a, q_rows, st)) != cudaSuccess) return e;
    if (max_lq > 0) {
        dim3 grid((max_lq + kRows - 1) / kRows, a.g.Hq, a.g.B);
        prof_before(st, kProfSimtBwdDq);
        kq<<<grid, kSplitThreads, smem_dq, st>>>(a);
        prof_after(st);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (max_lkv > 0) {
        dim3 grid((max_lkv + kKeys - 1) / kKeys, a.g.Hkv, a.g.B);
        prof_before(st, kProfSimtBwdDkDv);
        kkv<<<grid, kKvThreads, smem_kv, st>>>(a);
        prof_after(st);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace

// Head dims with a kernel: 32, 64, 96 and 128, for every element type (16-bit
// types normally take the tensor-core kernels; fp32 always comes here).
template <int D>
cudaError_t fwd_dtype(int dtype, const FwdArgs &a, int max_lq, cudaStream_t st) {
    switch (dtype) {
        case 0: return fwd_typed<__half, D>(a, max_lq, st);
        case 1: return fwd_typed<__nv_bfloat16, D>(a, max_lq, st);
        case 2: return fwd_typed<float, D>(a, max_lq, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_simt_fwd(int dtype, const FwdArgs &a, int max_lq, cudaStream_t st) {
    switch (a.g.D) {
        case 32: return fwd_dtype<32>(dtype, a, max_lq, st);
        case 64: return fwd_dtype<64>(dtype, a, max_lq, st);
        case 96: return fwd_dtype<96>(dtype, a, max_lq, st);
        case 128: return fwd_dtype<128>(dtype, a, max_lq, st);
    }
    return cudaErrorInvalidValue;
}

namespace {
bool rows_aligned16(const View &v, size_t es) {
    return ((uintptr_t)v.ptr % 16) == 0 && (v.sb * es) % 16 == 0 && (v.ss * es) % 16 == 0 &&
           (v.sh * es) % 16 == 0;
}
template <typename T, int VEC>
void preprocess_typed(const BwdArgs &a, int rows, cudaStream_t st) {
    const int tpr = lanes_per_row(a.g.D / VEC);
    const int64_t warps = ((int64_t)rows * a.g.Hq + (32 / tpr) - 1) / (32 / tpr);
    int64_t blocks = (warps + 7) / 8;
    int sms = 0;
    if (device_sm_count(&sms) != cudaSuccess) sms = 1;
    if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;  // grid-stride beyond 16 blocks per SM
    if (blocks < 1) blocks = 1;
    prof_before(st, kProfBwdPreprocess);
    bwd_preprocess_kernel<T, VEC><<<(unsigned)blocks, 256, 0, st>>>(a, rows);
    prof_after(st);
}
}  // namespace

namespace {
cudaError_t preprocess_any(int dtype, const BwdArgs &a, int rows, cudaStream_t st) {
    return launch_bwd_preprocess(dtype, a, rows, st);
}
}  // namespace

namespace {
template <typename T, int D>
cudaError_t preprocess16_typed(const BwdArgs &a, int rows, cudaStream_t st) {
    constexpr int U = 4;
    constexpr int NV = D / 8;
    constexpr int LPR = NV <= 4 ? 4 : NV <= 8 ? 8 : 16;
    const int64_t pairs = (int64_t)rows * a.g.Hq;
    int sms = 0;
    cudaError_t e = device_sm_count(&sms);
    if (e != cudaSuccess) return e;
    // warps needed, U row groups of 32 / LPR rows each; at most 8 blocks of
    // 256 threads per SM, the rest by the grid-stride loop
    const int64_t warps = (pairs + (32 / LPR) * U - 1) / ((32 / LPR) * U);
    int64_t blocks = (warps + 7) / 8;
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    if (blocks < 1) blocks = 1;
    prof_before(st, kProfBwdPreprocess);
    cudaError_t le = launch_pdl(bwd_preprocess16_kernel<T, D, U>, dim3((unsigned)blocks), dim3(256), 0, st, a, rows,
                                FastDiv(a.g.Hq), FastDiv(a.g.Sq > 0 ? a.g.Sq : 1));
    prof_after(st);
    return le != cudaSuccess ? le : cudaGetLastError();
}

template <typename T>
cudaError_t preprocess16_any(const BwdArgs &a, int rows, cudaStream_t st) {
    switch (a.g.D) {
        case 32: return preprocess16_typed<T, 32>(a, rows, st);
        case 64: return preprocess16_typed<T, 64>(a, rows, st);
        case 96: return preprocess16_typed<T, 96>(a, rows, st);
        case 128: return preprocess16_typed<T, 128>(a, rows, st);
    }
    return cudaErrorInvalidValue;
}
}  // namespace

cudaError_t launch_bwd_preprocess(int dtype, const BwdArgs &a, int rows, cudaStream_t st) {
    // 32-bit index arithmetic in the 16-bit kernel
    const bool idx32 = (int64_t)rows * a.g.Hq < ((int64_t)1 << 31);
    switch (dtype) {
        case 0:
            if (idx32) return preprocess16_any<__half>(a, rows, st);
            preprocess_typed<__half, 8>(a, rows, st);
            break;
        case 1:
            if (idx32) return preprocess16_any<__nv_bfloat16>(a, rows, st);
            preprocess_typed<__nv_bfloat16, 8>(a, rows, st);
            break;
        case 2:
            if (rows_aligned16(a.o, 4) && rows_aligned16(a.dout, 4))
                preprocess_typed<float, 4>(a, rows, st);
            else
                preprocess_typed<float, 1>(a, rows, st);
            break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <int D>
cudaError_t bwd_dtype(int dtype, const BwdArgs &a, int max_lq, int max_lkv, int q_rows, cudaStream_t st) {
    switch (dtype) {
        case 0: return bwd_typed<__half, D>(dtype, a, max_lq, max_lkv, q_rows, st);
        case 1: return bwd_typed<__nv_bfloat16, D>(dtype, a, max_lq, max_lkv, q_rows, st);
        case 2: return bwd_typed<float, D>(dtype, a, max_lq, max_lkv, q_rows, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_simt_bwd(int dtype, const BwdArgs &a, int max_lq, int max_lkv, int q_rows,
                            cudaStream_t st) {
    switch (a.g.D) {
        case 32: return bwd_dtype<32>(dtype, a, max_lq, max_lkv, q_rows, st);
        case 64: return bwd_dtype<64>(dtype, a, max_lq, max_lkv, q_rows, st);
        case 96: return bwd_dtype<96>(dtype, a, max_lq, max_lkv, q_rows, st);
        case 128: return bwd_dtype<128>(dtype, a, max_lq, max_lkv, q_rows, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gbattn
