// tc_bwd.cu -- tcgen05 backward attention for fp16 / bf16 (head dim 64, 128).
//
// One CTA owns a tile of 128 keys of one (batch, key/value head).  K and V
// stay in shared memory while the CTA walks every 64-row query block of every
// query head of the group that sees any of its keys.  Per block (q rows i,
// keys j, all fp32 accumulation in tensor memory):
//
//   S^T  = K Q^T            (keys x queries)
//   dP^T = V dO^T
//   P^T  = exp(scale S^T - LSE)       recomputed from the forward's LSE
//   dS^T = P^T o (dP^T - delta)       delta_i = <dO_i, O_i> (preprocess kernel)
//   dV  += P^T dO           P^T rounded to the input type, read from TMEM
//   dK  += dS^T Q           dS^T read from TMEM
//   dQ^T = K^T dS^T         dS^T also written to shared memory; the result is
//                           staged in shared memory and added to an fp32 dq
//                           accumulator in global memory by one bulk
//                           reduction per block
//
// (dK and dQ are scaled once at the end.)  Warp roles (448 threads): warps
// 0-7 compute P and dS (thread = key row; warps 0-3 take query columns 0-31,
// warps 4-7 columns 32-63) and store dK (0-3) and dV (4-7) at the end; warps
// 8-11 drain dQ^T from TMEM into the global accumulator (thread = head dim);
// warp 12 issues the loads (query blocks run QS stages ahead); warp 13
// allocates TMEM and issues the MMAs.
//
// TMEM columns: dK [0, D), dV [D, 2D), S/P double buffer 2 x 64, dP/dS 64,
// dQ^T 64 (M = 128 rows; for D = 64 the upper 64 rows multiply a zero tile).
// P and dS overwrite S and dP in place, packed two per column: query columns
// 0-31 into columns 0-15, 32-63 into 32-47.
#include <type_traits>

#include "ptx.cuh"
#include "tc.h"
#include "tmap.h"

namespace gbattn {
namespace {

using namespace ptx;

constexpr int BN = 128;   // keys per CTA
constexpr int BMQ = 64;   // query rows per block
constexpr int kMaxQS = 4;
constexpr int kThreads = 448;
constexpr int kCompute = 256;  // threads of the P / dS role
constexpr int kDrainWarp0 = 8;
constexpr int kProdWarp = 12;
constexpr int kMmaWarp = 13;

template <int D>
struct BwdCfg {
    static constexpr int QS = D == 128 ? 3 : 4;        // query-block pipeline stages
    static constexpr int kKVBytes = BN * D * 2;        // one K or V tile
    static constexpr int kQBytes = BMQ * D * 2;        // one Q or dO block
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKOff + kKVBytes;
    static constexpr int kQOff = kVOff + kKVBytes;
    static constexpr int kDOOff = kQOff + QS * kQBytes;
    static constexpr int kDSOff = kDOOff + QS * kQBytes;     // dS^T [128 keys][64 q]
    static constexpr int kZeroOff = kDSOff + BN * BMQ * 2;   // zero tile (D = 64 only)
    static constexpr int kDQOff = kZeroOff + (D == 64 ? BN * 128 : 0);  // fp32 [64 q][D]
    static constexpr int kStatOff = kDQOff + BMQ * D * 4;
    static constexpr int kBarOff = kStatOff + QS * BMQ * 2 * 4;
    static constexpr int kSmemBytes = kBarOff + 256 + 1024;
    // TMEM columns
    static constexpr int kTmDK = 0, kTmDV = D, kTmS = 2 * D, kTmDP = 2 * D + 128,
                         kTmDQ = 2 * D + 192;
};

struct Bars {
    uint64_t kv_full;
    uint64_t q_full[kMaxQS], q_empty[kMaxQS];
    uint64_t s_full, dp_full, ds_full, dk_done, it_done, dq_empty;
    uint32_t tmem_base;
    int abort_flag;
};

// TMEM column of k-step kk (16 query rows) of packed P / dS: each half of
// 32 query columns packs its rows into the first 16 of its own 32 columns,
// so no half overwrites values the other half has yet to read.
__device__ __forceinline__ constexpr uint32_t pcol(int kk) { return (kk / 2) * 32 + (kk % 2) * 8; }

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

// global[0 .. bytes) += shared[0 .. bytes) (fp32), as one bulk operation.
__device__ __forceinline__ void bulk_reduce_add_f32(float *gdst, const void *ssrc, uint32_t bytes) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
                     gdst),
                 "r"(smem_u32(ssrc)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  BwdArgs a, int n_ktiles) {
    using C = BwdCfg<D>;
    constexpr int QS = C::QS;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Bars &bar = *reinterpret_cast<Bars *>(smem + C::kBarOff);
    float *s_lse = reinterpret_cast<float *>(smem + C::kStatOff);      // [QS][64], log2 units
    float *s_delta = s_lse + QS * BMQ;                                  // [QS][64]
    const Geometry &g = a.g;

    const int bh = blockIdx.x % (g.Hkv * g.B);
    const int kt = blockIdx.x / (g.Hkv * g.B);
    const int hk = bh % g.Hkv, b = bh / g.Hkv;
    const SeqInfo s = seq_info(g, b);
    const int n0 = kt * BN;
    if (n0 >= s.Lkv) return;
    const int nkeys = min(BN, s.Lkv - n0);

    int ilo, ihi;
    query_range(n0, n0 + nkeys, s.Lq, g.wl, g.wr, ilo, ihi);
    const int nqb = (ihi - ilo + BMQ - 1) / BMQ;  // query blocks per head
    const int n_it = nqb * g.G;                   // iterations

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        mbar_init(&bar.kv_full, 1);
        for (int i = 0; i < QS; ++i) {
            mbar_init(&bar.q_full[i], 32);
            mbar_init(&bar.q_empty[i], 1);
        }
        mbar_init(&bar.s_full, 1);
        mbar_init(&bar.dp_full, 1);
        mbar_init(&bar.ds_full, kCompute);
        mbar_init(&bar.dk_done, 1);
        mbar_init(&bar.it_done, 1);
        mbar_init(&bar.dq_empty, 128);
        bar.abort_flag = 0;
        fence_mbar_init();
    }
    if (D == 64) {  // zero tile standing in for head dims 64..127 of K^T
        uint4 *z = reinterpret_cast<uint4 *>(smem + C::kZeroOff);
        for (int e = threadIdx.x; e < BN * 128 / 16; e += kThreads) z[e] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bar.tmem_base, 512);
        tmem_relinquish();
    }
    if (warp == kProdWarp && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem_base;
    const Watchdog wd{a.watchdog_ns, a.err, &bar.abort_flag};
    const int cb = g.thd ? 0 : b;  // TMA batch coordinate

    if (warp == kProdWarp) {
        // ------------------------------------------------------------ loads
        if (n_it > 0) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&bar.kv_full, 2 * C::kKVBytes);
                for (int c = 0; c < D / 64; ++c) {
                    tma_load_4d(smem + C::kKOff + c * BN * 128, &tm_k, &bar.kv_full, c * 64,
                                s.kv0 + n0, hk, cb);
                    tma_load_4d(smem + C::kVOff + c * BN * 128, &tm_v, &bar.kv_full, c * 64,
                                s.kv0 + n0, hk, cb);
                }
            }
            for (int t = 0; t < n_it; ++t) {
                const int st = t % QS;
                const uint32_t ph = (t / QS) & 1;
                const int h = hk * g.G + t / nqb;
                const int i0 = ilo + (t % nqb) * BMQ;
                // LSE (in log2 units) and delta of the block's rows, fetched
                // while the stage is still in use
                float lv[2], dv[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int i = i0 + lane + 32 * u;
                    lv[u] = dv[u] = 0.f;
                    if (i < s.Lq) {
                        const int64_t li = lse_index(g, s, b, h, i);
                        lv[u] = a.lse[li] * kLog2e;
                        dv[u] = a.delta[li];
                    }
                }
                if (!__all_sync(0xffffffffu, mbar_wait(&bar.q_empty[st], ph ^ 1, wd, 0x40))) break;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    s_lse[st * BMQ + lane + 32 * u] = lv[u];
                    s_delta[st * BMQ + lane + 32 * u] = dv[u];
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bar.q_full[st], 2 * C::kQBytes);
                    for (int c = 0; c < D / 64; ++c) {
                        tma_load_4d(smem + C::kQOff + st * C::kQBytes + c * BMQ * 128, &tm_q,
                                    &bar.q_full[st], c * 64, s.q0 + i0, h, cb);
                        tma_load_4d(smem + C::kDOOff + st * C::kQBytes + c * BMQ * 128, &tm_do,
                                    &bar.q_full[st], c * 64, s.q0 + i0, h, cb);
                    }
                } else {
                    mbar_arrive(&bar.q_full[st]);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA
        if (lane == 0 && n_it > 0) {
            const uint32_t sK = smem_u32(smem + C::kKOff), sV = smem_u32(smem + C::kVOff);
            const uint32_t sQ = smem_u32(smem + C::kQOff), sDO = smem_u32(smem + C::kDOOff);
            const uint32_t sDS = smem_u32(smem + C::kDSOff);
            constexpr uint32_t idSP = idesc_f16(128, BMQ, kBf16, 0, 0);   // S^T, dP^T
            constexpr uint32_t idKV = idesc_f16(128, D, kBf16, 0, 1);     // dV, dK
            constexpr uint32_t idQ = idesc_f16(128, BMQ, kBf16, 1, 1);    // dQ^T
            // K^T as an MN-major operand: atoms of 64 head dims, the second one
            // is the zero tile when D = 64
            constexpr uint32_t kLboKT = D == 128 ? BN * 128 : C::kZeroOff - C::kKOff;
            // Descriptors are formed once (per stage); each MMA adds a
            // compile-time offset to the start address.
            const uint64_t dK = smem_desc_sw128(sK, 16, 1024);       // K, K-major
            const uint64_t dV = smem_desc_sw128(sV, 16, 1024);       // V, K-major
            const uint64_t dKT = smem_desc_sw128(sK, kLboKT, 1024);  // K^T, MN-major
            const uint64_t dDS = smem_desc_sw128(sDS, BN * 128, 1024);
            auto kmaj_off = [](int kk, int rows) { return (kk / 4) * (rows * 128) + (kk % 4) * 32; };
            auto issue_s = [&](int t) {
                const uint64_t db = smem_desc_sw128(sQ + (t % QS) * C::kQBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + C::kTmS + (t & 1) * BMQ, desc_add(dK, kmaj_off(kk, BN)),
                           desc_add(db, kmaj_off(kk, BMQ)), idSP, kk > 0);
                mma_commit(&bar.s_full);
            };
            bool ok = mbar_wait(&bar.kv_full, 0, wd, 0x50);
            if (ok) ok = mbar_wait(&bar.q_full[0], 0, wd, 0x51);
            if (ok) {
                tc_fence_after();
                issue_s(0);
            }
            for (int t = 0; ok && t < n_it; ++t) {
                const int st = t % QS;
                const uint32_t sq = sQ + st * C::kQBytes, sdo = sDO + st * C::kQBytes;
                const uint64_t dDOk = smem_desc_sw128(sdo, 16, 1024);         // dO, K-major
                const uint64_t dDOm = smem_desc_sw128(sdo, BMQ * 128, 1024);  // dO, MN-major
                const uint64_t dQm = smem_desc_sw128(sq, BMQ * 128, 1024);    // Q, MN-major
                // dP^T into the dP buffer, free once iteration t-1's dK finished
                if (t > 0 && !(ok = mbar_wait(&bar.dk_done, (t - 1) & 1, wd, 0x52))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + C::kTmDP, desc_add(dV, kmaj_off(kk, BN)),
                           desc_add(dDOk, kmaj_off(kk, BMQ)), idSP, kk > 0);
                mma_commit(&bar.dp_full);
                // S^T of the next block runs while P and dS of this one are made
                // (its buffer held P of block t-1, whose dV finished before dk_done)
                if (t + 1 < n_it) {
                    if (!(ok = mbar_wait(&bar.q_full[(t + 1) % QS], ((t + 1) / QS) & 1, wd, 0x55)))
                        break;
                    tc_fence_after();
                    issue_s(t + 1);
                }
                if (!(ok = mbar_wait(&bar.ds_full, t & 1, wd, 0x53))) break;
                tc_fence_after();
                // dV += P^T dO, dK += dS^T Q  (B operands MN-major: N = head dim)
#pragma unroll
                for (int kk = 0; kk < BMQ / 16; ++kk)
                    mma_ts(tmem + C::kTmDV, tmem + C::kTmS + (t & 1) * BMQ + pcol(kk),
                           desc_add(dDOm, kk * 16 * 128), idKV, (t > 0 || kk > 0));
#pragma unroll
                for (int kk = 0; kk < BMQ / 16; ++kk)
                    mma_ts(tmem + C::kTmDK, tmem + C::kTmDP + pcol(kk), desc_add(dQm, kk * 16 * 128),
                           idKV, (t > 0 || kk > 0));
                mma_commit(&bar.q_empty[st]);
                mma_commit(&bar.dk_done);
                // dQ^T = K^T dS^T into the dQ buffer, free once drained
                if (t > 0 && !(ok = mbar_wait(&bar.dq_empty, (t - 1) & 1, wd, 0x54))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ss(tmem + C::kTmDQ, desc_add(dKT, kk * 16 * 128), desc_add(dDS, kk * 16 * 128),
                           idQ, kk > 0);
                mma_commit(&bar.it_done);
            }
        }
    } else if (warp < 8) {
        // ------------------------------------------ P, dS (thread = key row)
        const int half = warp / 4;           // query columns [32 half, 32 half + 32)
        const int c0 = half * 32;
        const int j = (warp % 4) * 32 + lane;  // key within the tile
        const int key = n0 + j;
        const uint32_t lane_off = (uint32_t)((warp % 4) * 32) << 16;
        const float c2 = g.scale_log2;
        uint8_t *dsrow = smem + C::kDSOff + j * 128;
        bool ok = true;
        for (int t = 0; t < n_it; ++t) {
            const int st = t % QS;
            const int i0 = ilo + (t % nqb) * BMQ + c0;  // first query row of this half
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.s_full, t & 1, wd, 0x60));
            if (!ok) break;
            tc_fence_after();
            uint32_t pr[32];
            const uint32_t tS = tmem + C::kTmS + (t & 1) * BMQ + lane_off;
            tmem_ld32(tS + c0, pr);
            // LSE / delta of this stage are in shared memory once q_full completed
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.q_full[st], (t / QS) & 1, wd, 0x61));
            if (!ok) break;
            const float4 *lse4 = reinterpret_cast<const float4 *>(s_lse + st * BMQ + c0);
            const bool full = (i0 + 31 < s.Lq) && (n0 + BN - 1 < s.Lkv) &&
                              (g.wr < 0 || n0 + BN - 1 <= i0 + g.wr) &&
                              (g.wl < 0 || n0 >= i0 + 31 - g.wl);
            float p[32];
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 l4 = lse4[q4];
                const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = 4 * q4 + e;
                    p[c] = ex2(fmaf(__uint_as_float(pr[c]), c2, -lv[e]));
                }
            }
            if (!full) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int i = i0 + c;
                    if (!(i < s.Lq && visible(i, key, s.Lkv, g.wl, g.wr))) p[c] = 0.f;
                }
            }
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) pk[c] = pack2<T>(p[2 * c], p[2 * c + 1]);
            tmem_st16(tS + c0, pk);  // packed into the first 16 of this half's columns
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.dp_full, t & 1, wd, 0x62));
            if (!ok) break;
            tc_fence_after();
            const uint32_t tP = tmem + C::kTmDP + lane_off;
            tmem_ld32(tP + c0, pr);
            const float4 *dl4 = reinterpret_cast<const float4 *>(s_delta + st * BMQ + c0);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 d4 = dl4[q4];
                const float d0 = p[4 * q4] * (__uint_as_float(pr[4 * q4]) - d4.x);
                const float d1 = p[4 * q4 + 1] * (__uint_as_float(pr[4 * q4 + 1]) - d4.y);
                const float d2 = p[4 * q4 + 2] * (__uint_as_float(pr[4 * q4 + 2]) - d4.z);
                const float d3 = p[4 * q4 + 3] * (__uint_as_float(pr[4 * q4 + 3]) - d4.w);
                pk[2 * q4] = pack2<T>(d0, d1);
                pk[2 * q4 + 1] = pack2<T>(d2, d3);
            }
            tmem_st16(tP + c0, pk);
            // dS^T row j, this half's 4 chunks of the swizzled MN-major tile
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int chunk = c0 / 8 + q;
                uint4 v = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                *reinterpret_cast<uint4 *>(dsrow + ((chunk ^ (j & 7)) * 16)) = v;
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar.ds_full);
        }
        // epilogue: dK (scaled) from warps 0-3, dV from warps 4-7
        if (ok && n_it > 0)
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.it_done, (n_it - 1) & 1, wd, 0x63));
        tc_fence_after();
        const bool valid = j < nkeys;
        const MutView &ov = half == 0 ? a.dk : a.dv;
        T *dst = (T *)ov.ptr + (int64_t)b * ov.sb + (int64_t)(s.kv0 + key) * ov.ss +
                 (int64_t)hk * ov.sh;
        const float mul = half == 0 ? g.scale : 1.f;
        const uint32_t base = tmem + (half == 0 ? C::kTmDK : C::kTmDV) + lane_off;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t v[32];
            if (n_it > 0) {
                tmem_ld32(base + cc * 32, v);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0u;
            }
            if (valid) {
                uint4 pk4[4];
                uint32_t *pw = reinterpret_cast<uint32_t *>(pk4);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pw[e] = pack2<T>(__uint_as_float(v[2 * e]) * mul,
                                     __uint_as_float(v[2 * e + 1]) * mul);
                uint4 *d4 = reinterpret_cast<uint4 *>(dst + cc * 32);
#pragma unroll
                for (int e = 0; e < 4; ++e) d4[e] = pk4[e];
            }
        }
    } else {
        // ------------------------------------- dQ^T drain (thread = head dim)
        // dq accumulator layout: [Hq][rows][D] fp32, so the block's rows of one
        // head are contiguous and go out as a single bulk reduction.
        const int wq = warp % 4;
        const int d = wq * 32 + lane;
        const uint32_t tQ = tmem + C::kTmDQ + ((uint32_t)(wq * 32) << 16);
        const bool has = wq * 32 < D;  // D = 64: lanes 64..127 hold zeros
        const bool leader = threadIdx.x == kDrainWarp0 * 32;
        float *sdq = reinterpret_cast<float *>(smem + C::kDQOff);
        const int64_t rows_total = g.thd ? (int64_t)g.Tq : (int64_t)g.B * g.Sq;
        const int64_t row_base = g.thd ? s.q0 : (int64_t)b * g.Sq;
        for (int t = 0; t < n_it; ++t) {
            const int h = hk * g.G + t / nqb;
            const int i0 = ilo + (t % nqb) * BMQ;
            if (!__all_sync(0xffffffffu, mbar_wait(&bar.it_done, t & 1, wd, 0x70))) break;
            tc_fence_after();
            uint32_t v[BMQ];
            if (has) {
                tmem_ld32(tQ, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                tmem_ld32(tQ + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            }
            tc_fence_before();
            mbar_arrive(&bar.dq_empty);
            if (leader) bulk_wait_read0();  // previous block's staging tile was read
            named_bar_sync(1, 128);
            if (has) {
#pragma unroll
                for (int c = 0; c < BMQ; ++c) sdq[c * D + d] = __uint_as_float(v[c]);
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (leader) {
                const int nrow = min(BMQ, s.Lq - i0);
                float *dst = a.dq_acc + ((int64_t)h * rows_total + row_base + i0) * D;
                bulk_reduce_add_f32(dst, sdq, (uint32_t)(nrow * D * 4));
                bulk_commit();
            }
        }
        if (leader) bulk_wait0();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// dq = scale * dq_acc ([Hq][rows][D] fp32), converted and written through
// dq's strides.
template <typename T>
__global__ void dq_convert_kernel(BwdArgs a, int rows) {
    const Geometry &g = a.g;
    const int D = g.D;
    const int64_t n = (int64_t)rows * g.Hq * (D / 8);
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int c8 = (int)(e % (D / 8));
        const int64_t hr = e / (D / 8);  // h * rows + r
        const int r = (int)(hr % rows);
        const int h = (int)(hr / rows);
        int b = 0, row = r;
        if (!g.thd) {
            b = r / g.Sq;
            row = r % g.Sq;
        }
        const float4 *src = reinterpret_cast<const float4 *>(a.dq_acc + hr * D + c8 * 8);
        const float4 x = src[0], y = src[1];
        uint4 o;
        o.x = pack2<T>(x.x * g.scale, x.y * g.scale);
        o.y = pack2<T>(x.z * g.scale, x.w * g.scale);
        o.z = pack2<T>(y.x * g.scale, y.y * g.scale);
        o.w = pack2<T>(y.z * g.scale, y.w * g.scale);
        T *dst = (T *)a.dq.ptr + (int64_t)b * a.dq.sb + (int64_t)row * a.dq.ss + (int64_t)h * a.dq.sh +
                 c8 * 8;
        *reinterpret_cast<uint4 *>(dst) = o;
    }
}

template <typename T, int D>
cudaError_t launch_typed(const BwdArgs &a, int max_lq, int max_lkv, int q_rows, cudaStream_t st) {
    const int dt = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;
    const Geometry &g = a.g;
    const uint64_t es = 2;
    const uint64_t nb = g.thd ? 1 : (uint64_t)g.B;
    uint64_t dq[4] = {(uint64_t)D, (uint64_t)g.Sq, (uint64_t)g.Hq, nb};
    uint64_t dk[4] = {(uint64_t)D, (uint64_t)g.Skv, (uint64_t)g.Hkv, nb};
    auto strides = [&](const View &v, const uint64_t dims[4], uint64_t out[3]) {
        const int64_t el[3] = {v.ss, v.sh, g.thd ? 0 : v.sb};
        for (int i = 0; i < 3; ++i)
            out[i] = (dims[i + 1] == 1 && el[i] == 0) ? 16 : (uint64_t)el[i] * es;
    };
    uint64_t sq[3], sk[3], sv[3], sd[3];
    strides(a.q, dq, sq);
    strides(a.k, dk, sk);
    strides(a.v, dk, sv);
    strides(a.dout, dq, sd);
    CUtensorMap tq, tk, tv, tdo;
    cudaError_t e;
    if ((e = make_tmap_16bit(&tq, a.q.ptr, dt, dq, sq, BMQ)) != cudaSuccess) return e;
    if ((e = make_tmap_16bit(&tk, a.k.ptr, dt, dk, sk, BN)) != cudaSuccess) return e;
    if ((e = make_tmap_16bit(&tv, a.v.ptr, dt, dk, sv, BN)) != cudaSuccess) return e;
    if ((e = make_tmap_16bit(&tdo, a.dout.ptr, dt, dq, sd, BMQ)) != cudaSuccess) return e;
    if (max_lkv > 0) {
        const int smem = BwdCfg<D>::kSmemBytes;
        auto kern = tc_bwd_kernel<T, D>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
            cudaSuccess)
            return e;
        const int n_ktiles = (max_lkv + BN - 1) / BN;
        const int64_t grid = (int64_t)n_ktiles * g.Hkv * g.B;
        if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
        kern<<<(unsigned)grid, kThreads, smem, st>>>(tq, tk, tv, tdo, a, n_ktiles);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (q_rows > 0) {
        const int64_t n = (int64_t)q_rows * g.Hq * (D / 8);
        const int64_t blocks = std::min<int64_t>((n + 255) / 256, 152 * 16);
        dq_convert_kernel<T><<<(unsigned)blocks, 256, 0, st>>>(a, q_rows);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

bool uses_tc_bwd(int dtype, int D) { return (dtype == 0 || dtype == 1) && (D == 64 || D == 128); }

cudaError_t launch_tc_bwd(int dtype, const BwdArgs &a, int max_lq, int max_lkv, int q_rows,
                          cudaStream_t st) {
    switch (dtype * 2 + (a.g.D == 128)) {
        case 0: return launch_typed<__half, 64>(a, max_lq, max_lkv, q_rows, st);
        case 1: return launch_typed<__half, 128>(a, max_lq, max_lkv, q_rows, st);
        case 2: return launch_typed<__nv_bfloat16, 64>(a, max_lq, max_lkv, q_rows, st);
        case 3: return launch_typed<__nv_bfloat16, 128>(a, max_lq, max_lkv, q_rows, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gbattn
