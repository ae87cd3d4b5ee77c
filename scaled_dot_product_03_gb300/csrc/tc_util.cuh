// tc_util.cuh -- small device helpers shared by the single-pass backward
// kernels (internal).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace gbattn {
namespace tcu {

// Byte offset of k-step kk (16 elements along K) in a K-major 128B-swizzled
// tile of `rows` rows (64-element atoms of rows x 128 B).
__device__ __forceinline__ constexpr uint32_t kmaj_off(int kk, int rows) {
    return (kk / 4) * (rows * 128) + (kk % 4) * 32;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T> __device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Element-wise product of two packed pairs, rounded to nearest.
template <typename T> __device__ __forceinline__ uint32_t mul2(uint32_t a, uint32_t b);
template <> __device__ __forceinline__ uint32_t mul2<__nv_bfloat16>(uint32_t a, uint32_t b) {
    const __nv_bfloat162 r =
        __hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&a), *reinterpret_cast<const __nv_bfloat162 *>(&b));
    return *reinterpret_cast<const uint32_t *>(&r);
}
template <> __device__ __forceinline__ uint32_t mul2<__half>(uint32_t a, uint32_t b) {
    const __half2 r = __hmul2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b));
    return *reinterpret_cast<const uint32_t *>(&r);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// Adds a box of fp32 from shared memory into the tensor at (x, y, z).
__device__ __forceinline__ void tma_reduce_add_3d(uint32_t src, const CUtensorMap *map, int x, int y, int z) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            map),
        "r"(x), "r"(y), "r"(z), "r"(src)
        : "memory");
}

// Writes 32 fp32 values (times mul) of one row as the element type.
template <typename T>
__device__ __forceinline__ void store_row32(T *dst, const uint32_t (&v)[32], float mul) {
    uint4 pk[4];
    uint32_t *pw = reinterpret_cast<uint32_t *>(pk);
#pragma unroll
    for (int e = 0; e < 16; ++e)
        pw[e] = pack2<T>(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int e = 0; e < 4; ++e) d4[e] = pk[e];
}

// Writes 32 fp32 values of one row (16-byte stores).
__device__ __forceinline__ void store_f32_row32(float *dst, const uint32_t (&v)[32]) {
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int e = 0; e < 8; ++e) d4[e] = make_uint4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
}

// One work item of a persistent single-pass backward: the BK keys of key
// tile kt of a (batch, key/value head, query-head split), decoded from its
// index w in the banded, heaviest-first order.
struct BwdItem {
    SeqInfo s;
    int b, hk, sp, kt;
    int n0, nkeys;   // first key, keys in the tile (<= 0: the tile is past the sequence)
    int h0, nh;      // query heads [h0, h0 + nh)
    int ilo, nqb;    // first query row seeing the tile, query blocks per head
    int n_it;        // blocks: nqb * nh
};

__device__ __forceinline__ BwdItem bwd_item(int w, const Geometry &g, int nsplit, int n_ktiles, int bk, int bq,
                                            int band) {
    BwdItem it;
    int bhs;
    banded_order(w, n_ktiles, g.Hkv * g.B * nsplit, bhs, it.kt, band);
    it.sp = bhs % nsplit;
    const int bh = bhs / nsplit;
    it.hk = bh % g.Hkv;
    it.b = bh / g.Hkv;
    it.s = seq_info(g, it.b);
    it.n0 = it.kt * bk;
    it.nkeys = min(bk, it.s.Lkv - it.n0);
    const int gs = (g.G + nsplit - 1) / nsplit;
    it.h0 = it.hk * g.G + it.sp * gs;
    it.nh = max(0, min(gs, g.G - it.sp * gs));
    int ihi = 0;
    it.ilo = 0;
    if (it.nkeys > 0) query_range(it.n0, it.n0 + it.nkeys, it.s.Lq, g.wl, g.wr, it.ilo, ihi);
    it.nqb = (ihi - it.ilo + bq - 1) / bq;
    it.n_it = it.nkeys > 0 ? it.nqb * it.nh : 0;
    return it;
}

}  // namespace tcu
}  // namespace gbattn
