// common.cuh -- types shared by the library's translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gbattn {

// log2(e) and ln(2), for moving between natural-log and base-2 softmax.
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// A tensor view: base pointer and element strides of (b, s, h); the d
// stride is 1.  THD views have sb = 0 and carry the sequence start in the
// row offset instead.
struct View {
    const void *ptr;
    int64_t sb, ss, sh;
};

struct MutView {
    void *ptr;
    int64_t sb, ss, sh;
};

// Everything a kernel needs to locate sequence b.
struct Geometry {
    int B, Sq, Skv, Hq, Hkv, D, G;
    int thd;              // 1: packed THD, 0: dense
    int Tq;               // THD: total query rows (LSE row pitch)
    const int *cu_q, *cu_kv;
    const int *pad_q, *pad_kv;  // THD: first row of each sequence when the
                                // buffer is padded (null: cu_q / cu_kv)
    int wl, wr;           // window, -1 = unbounded
    float scale;
    float scale_log2;     // scale * log2(e)
};

// Head dim the tensor-core kernels compute with for a head dim D of 32, 64,
// 96 or 128: 32 runs on the 64-wide kernels and 96 on the 128-wide ones.
// Tensor maps keep the real D as their inner extent, so the loads fill the
// columns past D with zeros (which add nothing to any product) and the
// stores drop them; row-by-row stores stop at D.
__host__ __device__ constexpr int tc_dim(int D) { return D <= 64 ? 64 : 128; }

struct SeqInfo {
    int q0, kv0;  // first row of the sequence (THD), 0 for dense
    int Lq, Lkv;  // lengths
};

__device__ __forceinline__ SeqInfo seq_info(const Geometry &g, int b) {
    SeqInfo s;
    if (g.thd) {
        const int q_lo = __ldg(g.cu_q + b), kv_lo = __ldg(g.cu_kv + b);
        s.Lq = __ldg(g.cu_q + b + 1) - q_lo;
        s.Lkv = __ldg(g.cu_kv + b + 1) - kv_lo;
        s.q0 = g.pad_q ? __ldg(g.pad_q + b) : q_lo;
        s.kv0 = g.pad_kv ? __ldg(g.pad_kv + b) : kv_lo;
    } else {
        s.q0 = 0;
        s.kv0 = 0;
        s.Lq = g.Sq;
        s.Lkv = g.Skv;
    }
    return s;
}

// Whether token row `row` of a THD buffer lies inside a sequence (rows of
// the tail, or in the gaps of a padded buffer, do not): the last sequence
// starting at or before the row must still extend over it.
__device__ __forceinline__ bool thd_row_in_sequence(const int *cu, const int *pad, int B, int row) {
    if (B <= 0) return false;
    const int *start = pad ? pad : cu;
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (__ldg(start + mid) <= row) lo = mid; else hi = mid - 1;
    }
    const int len = __ldg(cu + lo + 1) - __ldg(cu + lo);
    return row >= __ldg(start + lo) && row < __ldg(start + lo) + len;
}

// Index of LSE / row-term element of query row i of head h in sequence b.
__device__ __forceinline__ int64_t lse_index(const Geometry &g, const SeqInfo &s,
                                             int b, int h, int i) {
    return g.thd ? (int64_t)h * g.Tq + s.q0 + i
                 : ((int64_t)b * g.Hq + h) * g.Sq + i;
}

// Bits of the device error word other than the watchdog codes (which stay
// below 2^16).  THD launches size their grids from max_seqlen_q / _kv; a
// sequence longer than that would be left partly unprocessed, so the CTA of
// each sequence's last grid tile reports it with one of these bits.
constexpr unsigned kErrSeqlenQ = 1u << 30;
constexpr unsigned kErrSeqlenKv = 1u << 29;

__device__ __forceinline__ void report_uncovered(unsigned *err, const Geometry &g, int len, int covered,
                                                 unsigned bit) {
    if (g.thd && len > covered) atomicOr(err, bit);
}

__device__ __forceinline__ bool visible(int i, int j, int Lkv, int wl, int wr) {
    return j >= 0 && j < Lkv && (wl < 0 || j >= i - wl) && (wr < 0 || j <= i + wr);
}

// Range [lo, hi) of keys visible to at least one of query rows [i0, i1).
__device__ __forceinline__ void key_range(int i0, int i1, int Lkv, int wl, int wr,
                                          int &lo, int &hi) {
    lo = wl < 0 ? 0 : max(0, i0 - wl);
    hi = wr < 0 ? Lkv : min(Lkv, i1 - 1 + wr + 1);
    if (hi < lo) hi = lo;
}

// Range [lo, hi) of query rows that see at least one of keys [j0, j1).
__device__ __forceinline__ void query_range(int j0, int j1, int Lq, int wl, int wr,
                                            int &lo, int &hi) {
    lo = wr < 0 ? 0 : max(0, j0 - wr);
    hi = wl < 0 ? Lq : min(Lq, j1 - 1 + wl + 1);
    if (hi < lo) hi = lo;
}

// Work order of the tensor-core kernels.  Work index w covers nt tiles of
// each of nbh (batch, head) pairs.  Heads are grouped in bands of `band`
// pairs: the work in flight at one time then touches a few heads' tensors
// (they stay in L2), and inside a band the tiles go by rank 0 (heaviest)
// first, each rank across the band's heads, so dispatch stays close to
// longest-first.  Measured: 8 suits the forward and the two-kernel
// backward; the single-pass backward, whose fp32 dQ sums also live in L2,
// prefers fewer heads per band.
constexpr int kHeadBand = 8;

__device__ __forceinline__ void banded_order(int w, int nt, int nbh, int &bh, int &rank,
                                             int band = kHeadBand) {
    const int per_band = band * nt;
    const int bi = w / per_band, r = w % per_band;
    const int h0 = bi * band;
    const int bs = min(band, nbh - h0);
    rank = r / bs;
    bh = h0 + r % bs;
}

// Unsigned 32-bit division by a divisor fixed for a launch, as a multiply
// and shifts (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994, the round-up method for N-bit unsigned operands):
// with 2^(l-1) < d <= 2^l and m = floor(2^32 (2^l - d) / d) + 1,
//   t = umulhi(m, n),  n / d = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0)
// for every 32-bit n.  Built on the host, used by the streaming kernels whose
// per-row index arithmetic would otherwise be dominated by divisions.
struct FastDiv {
    uint32_t d, m, s1, s2;
    FastDiv() = default;
    __host__ explicit FastDiv(uint32_t div) : d(div) {
        uint32_t l = 0;
        while (l < 32 && ((uint64_t)1 << l) < div) ++l;
        m = (uint32_t)((((uint64_t)1 << 32) * (((uint64_t)1 << l) - div)) / div + 1);
        s1 = l < 1 ? l : 1;
        s2 = l > 0 ? l - 1 : 0;
    }
    __host__ __device__ __forceinline__ uint32_t div(uint32_t n) const {
#ifdef __CUDA_ARCH__
        const uint32_t t = __umulhi(m, n);
#else
        const uint32_t t = (uint32_t)(((uint64_t)m * n) >> 32);
#endif
        return (t + ((n - t) >> s1)) >> s2;
    }
};

// Programmatic dependent launch.  griddep_wait: wait until the grids this
// one depends on have completed and their writes are visible (returns at
// once for a grid launched without the dependency).  griddep_launch: let the
// grid that depends on this one begin launching once every CTA of this grid
// has issued it (or exited).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

}  // namespace gbattn
