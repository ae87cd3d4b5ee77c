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

}  // namespace tcu
}  // namespace gbattn
