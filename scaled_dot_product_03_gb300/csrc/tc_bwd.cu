// tc_bwd.cu -- tcgen05 backward attention for fp16 / bf16 (head dim 64, 128).
//
// Two kernels, each the only writer of its outputs, so nothing is
// accumulated across CTAs and the result does not depend on scheduling:
//
// dK/dV kernel: one CTA per 128 keys of a (batch, key/value head).  K and V
// stay in shared memory while the CTA walks every 128-row query block of
// every query head of the group that sees its keys (keys j, queries i):
//   S^T  = K Q^T,  dP^T = V dO^T          (A and B from shared memory)
//   P^T  = exp(scale S^T - LSE)           recomputed from the forward's LSE
//   dS^T = P^T o (dP^T - delta)           delta_i = <dO_i, O_i> (preprocess)
//   dV  += P^T dO,  dK += dS^T Q          (P^T, dS^T read from TMEM)
// dQ kernel: one CTA per 128 query rows of a (batch, query head).  Q and dO
// sit in TMEM as MMA operands while the CTA walks the key blocks its rows see:
//   S = Q K^T,  dP = dO V^T,  P, dS as above (thread = query row),
//   dQ += dS K                            (dS read from TMEM)
// dK and dQ are scaled once at the end.
//
// In both kernels warps 0-7 compute P and dS for one row each (warps 0-3
// take columns 0-63 of the block, warps 4-7 columns 64-127) and store the
// results at the end, warp 8 issues TMA loads and warp 9 allocates TMEM and
// issues the MMAs.  P and dS overwrite S and dP in TMEM, packed two per
// column: columns 0-63 of the block into TMEM columns 0-31, 64-127 into
// 64-95, so neither half overwrites values the other half has yet to read.
#include <algorithm>
#include <type_traits>

#include "ptx.cuh"
#include "tc.h"
#include "prof.h"
#include "tmap.h"

namespace gbattn {
namespace {

using namespace ptx;

constexpr int BLK = 128;   // rows of every tile: keys (dK/dV) or queries (dQ)
constexpr int kThreads = 320;
constexpr int kCompute = 256;
constexpr int kProdWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kMaxStages = 3;

// TMEM column of k-step kk (16 rows of the block) of packed P / dS.
__device__ __forceinline__ constexpr uint32_t pcol(int kk) { return (kk / 4) * 64 + (kk % 4) * 8; }
// Byte offset of k-step kk (16 head dims) in a K-major tile of `rows` rows.
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

// ===================================================================== dK dV
template <int D>
struct KVCfg {
    static constexpr int QS = D == 128 ? 2 : 3;           // query-block stages
    static constexpr int kTile = BLK * D * 2;             // one 128 x D tile
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKOff + kTile;
    static constexpr int kQOff = kVOff + kTile;
    static constexpr int kDOOff = kQOff + QS * kTile;
    static constexpr int kStatOff = kDOOff + QS * kTile;  // [QS][128] lse2, [QS][128] delta
    static constexpr int kBarOff = kStatOff + QS * BLK * 2 * 4;
    static constexpr int kSmemBytes = kBarOff + 256 + 1024;
    static constexpr int kTmDK = 0, kTmDV = D, kTmS = 2 * D, kTmDP = 2 * D + 128;
};

struct KVBars {
    uint64_t kv_full;
    uint64_t q_full[kMaxStages], q_empty[kMaxStages];
    uint64_t s_full, dp_full, p_full, ds_full, acc_done;
    uint32_t tmem_base;
    int abort_flag;
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       BwdArgs a, int n_ktiles) {
    using C = KVCfg<D>;
    constexpr int QS = C::QS;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    KVBars &bar = *reinterpret_cast<KVBars *>(smem + C::kBarOff);
    float *s_lse = reinterpret_cast<float *>(smem + C::kStatOff);  // log2 units
    float *s_delta = s_lse + QS * BLK;
    const Geometry &g = a.g;

    // banded work order; rank 0 = the first key tiles (seen by the most
    // queries when causal)
    // (a split of the query heads of a group counts as a head of its own)
    int bhs, kt;
    banded_order(blockIdx.x, n_ktiles, g.Hkv * g.B * a.nsplit, bhs, kt);
    const int sp = bhs % a.nsplit, bh = bhs / a.nsplit;
    const int hk = bh % g.Hkv, b = bh / g.Hkv;
    const SeqInfo s = seq_info(g, b);
    const int n0 = kt * BLK;
    if (kt == n_ktiles - 1 && sp == 0 && threadIdx.x == 0)
        report_uncovered(a.err, g, s.Lkv, n_ktiles * BLK, kErrSeqlenKv);
    if (n0 >= s.Lkv) return;
    const int nkeys = min(BLK, s.Lkv - n0);
    // query heads of this CTA: [h0, h0 + nh) of the group's G
    const int gs = (g.G + a.nsplit - 1) / a.nsplit;
    const int h0 = hk * g.G + sp * gs;
    const int nh = min(gs, g.G - sp * gs);

    int ilo, ihi;
    query_range(n0, n0 + nkeys, s.Lq, g.wl, g.wr, ilo, ihi);
    const int nqb = (ihi - ilo + BLK - 1) / BLK;  // query blocks per head
    const int n_it = nqb * nh;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        mbar_init(&bar.kv_full, 1);
        for (int i = 0; i < QS; ++i) {
            mbar_init(&bar.q_full[i], 32);
            mbar_init(&bar.q_empty[i], 1);
        }
        mbar_init(&bar.s_full, 1);
        mbar_init(&bar.dp_full, 1);
        mbar_init(&bar.p_full, kCompute);
        mbar_init(&bar.ds_full, kCompute);
        mbar_init(&bar.acc_done, 1);
        bar.abort_flag = 0;
        fence_mbar_init();
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
                mbar_arrive_expect_tx(&bar.kv_full, 2 * C::kTile);
                for (int c = 0; c < D / 64; ++c) {
                    tma_load_4d(smem + C::kKOff + c * BLK * 128, &tm_k, &bar.kv_full, c * 64,
                                s.kv0 + n0, hk, cb);
                    tma_load_4d(smem + C::kVOff + c * BLK * 128, &tm_v, &bar.kv_full, c * 64,
                                s.kv0 + n0, hk, cb);
                }
            }
            for (int t = 0; t < n_it; ++t) {
                const int st = t % QS;
                const uint32_t ph = (t / QS) & 1;
                const int h = h0 + t / nqb;
                const int i0 = ilo + (t % nqb) * BLK;
                // LSE (log2 units) and delta of the block's rows, fetched while
                // the stage is still in use
                float lv[4], dv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
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
                for (int u = 0; u < 4; ++u) {
                    s_lse[st * BLK + lane + 32 * u] = lv[u];
                    s_delta[st * BLK + lane + 32 * u] = dv[u];
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bar.q_full[st], 2 * C::kTile);
                    for (int c = 0; c < D / 64; ++c) {
                        tma_load_4d(smem + C::kQOff + st * C::kTile + c * BLK * 128, &tm_q,
                                    &bar.q_full[st], c * 64, s.q0 + i0, h, cb);
                        tma_load_4d(smem + C::kDOOff + st * C::kTile + c * BLK * 128, &tm_do,
                                    &bar.q_full[st], c * 64, s.q0 + i0, h, cb);
                    }
                } else {
                    mbar_arrive(&bar.q_full[st]);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA
        // Per block t: S^T_t, dP^T_t, then dV_t (once P is written), S^T_{t+1}
        // (its TMEM held P_t, read by dV_t just before: MMAs of one thread
        // execute in issue order), dK_t (once dS is written), dP^T_{t+1}.
        // The whole warp runs the loop in step; one elected lane issues each
        // group of MMAs with its commit.
        if (n_it > 0) {
            constexpr uint32_t idSP = idesc_f16(BLK, BLK, kBf16, 0, 0);  // S^T, dP^T
            constexpr uint32_t idKV = idesc_f16(BLK, D, kBf16, 0, 1);    // dV, dK
            const uint32_t sQ = smem_u32(smem + C::kQOff), sDO = smem_u32(smem + C::kDOOff);
            const uint64_t dK = smem_desc_sw128(smem_u32(smem + C::kKOff), 16, 1024);
            const uint64_t dV = smem_desc_sw128(smem_u32(smem + C::kVOff), 16, 1024);
            auto wait = [&](uint64_t *b, uint32_t ph, unsigned code) {
                const bool r = __all_sync(0xffffffffu, mbar_wait(b, ph, wd, code));
                if (r) tc_fence_after();
                return r;
            };
            auto issue_s = [&](int t) {
                const uint64_t db = smem_desc_sw128(sQ + (t % QS) * C::kTile, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tmem + C::kTmS, desc_add(dK, kmaj_off(kk, BLK)), desc_add(db, kmaj_off(kk, BLK)),
                               idSP, kk > 0);
                    mma_commit(&bar.s_full);
                }
                __syncwarp();
            };
            auto issue_dp = [&](int t) {
                const uint64_t db = smem_desc_sw128(sDO + (t % QS) * C::kTile, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tmem + C::kTmDP, desc_add(dV, kmaj_off(kk, BLK)), desc_add(db, kmaj_off(kk, BLK)),
                               idSP, kk > 0);
                    mma_commit(&bar.dp_full);
                }
                __syncwarp();
            };
            bool ok = wait(&bar.kv_full, 0, 0x50) && wait(&bar.q_full[0], 0, 0x51);
            if (ok) {
                issue_s(0);
                issue_dp(0);
            }
            for (int t = 0; ok && t < n_it; ++t) {
                const int st = t % QS;
                const bool next = t + 1 < n_it;
                const uint32_t acc0 = t > 0 ? 1u : 0u;
                // B operands as MN-major (N = head dim) views of the Q / dO tiles
                const uint64_t dOm = smem_desc_sw128(sDO + st * C::kTile, BLK * 128, 1024);
                const uint64_t dQm = smem_desc_sw128(sQ + st * C::kTile, BLK * 128, 1024);
                if (!(ok = wait(&bar.p_full, t & 1, 0x52))) break;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BLK / 16; ++kk)
                        mma_ts(tmem + C::kTmDV, tmem + C::kTmS + pcol(kk), desc_add(dOm, kk * 16 * 128), idKV,
                               kk > 0 ? 1u : acc0);
                }
                __syncwarp();
                if (next) {
                    if (!(ok = wait(&bar.q_full[(t + 1) % QS], ((t + 1) / QS) & 1, 0x53))) break;
                    issue_s(t + 1);
                }
                if (!(ok = wait(&bar.ds_full, t & 1, 0x54))) break;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BLK / 16; ++kk)
                        mma_ts(tmem + C::kTmDK, tmem + C::kTmDP + pcol(kk), desc_add(dQm, kk * 16 * 128), idKV,
                               kk > 0 ? 1u : acc0);
                    mma_commit(&bar.q_empty[st]);
                }
                __syncwarp();
                if (next) issue_dp(t + 1);
            }
            if (ok && elect_one()) mma_commit(&bar.acc_done);
            __syncwarp();
        }
    } else {
        // --------------------------------------- P, dS (thread = key row)
        const int half = warp / 4;             // query columns [64 half, 64 half + 64)
        const int c0 = half * 64;
        const int j = (warp % 4) * 32 + lane;  // key within the tile
        const int key = n0 + j;
        const uint32_t lane_off = (uint32_t)((warp % 4) * 32) << 16;
        const uint32_t tS = tmem + C::kTmS + c0 + lane_off;
        const uint32_t tP = tmem + C::kTmDP + c0 + lane_off;
        const float c2 = g.scale_log2;
        bool ok = true;
        for (int t = 0; t < n_it; ++t) {
            const int st = t % QS;
            const int i0 = ilo + (t % nqb) * BLK + c0;  // first query row of this half
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.s_full, t & 1, wd, 0x60));
            if (!ok) break;
            tc_fence_after();
            // (LSE / delta of stage st were written before q_full completed,
            // which S^T_t itself waited for)
            const float *lse2 = s_lse + st * BLK + c0;
            const float *dlt = s_delta + st * BLK + c0;
            const bool full = (i0 + 63 < s.Lq) && (n0 + BLK - 1 < s.Lkv) &&
                              (g.wr < 0 || n0 + BLK - 1 <= i0 + g.wr) &&
                              (g.wl < 0 || n0 >= i0 + 63 - g.wl);
            float p[64];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t sr[32];
                tmem_ld32(tS + 32 * h2, sr);
                // 16-byte broadcast reads of the LSE (fewer shared memory wavefronts)
                const float4 *l4 = reinterpret_cast<const float4 *>(lse2 + 32 * h2);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 l = l4[q];
                    p[32 * h2 + 4 * q] = ex2(fmaf(__uint_as_float(sr[4 * q]), c2, -l.x));
                    p[32 * h2 + 4 * q + 1] = ex2(fmaf(__uint_as_float(sr[4 * q + 1]), c2, -l.y));
                    p[32 * h2 + 4 * q + 2] = ex2(fmaf(__uint_as_float(sr[4 * q + 2]), c2, -l.z));
                    p[32 * h2 + 4 * q + 3] = ex2(fmaf(__uint_as_float(sr[4 * q + 3]), c2, -l.w));
                }
            }
            if (!full) {
                // queries that see this key: columns [clo, chi) of this half
                int clo = 0, chi = min(64, s.Lq - i0);
                if (g.wr >= 0) clo = max(clo, key - g.wr - i0);
                if (g.wl >= 0) chi = min(chi, key + g.wl + 1 - i0);
                if (key >= s.Lkv) chi = clo;
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (c < clo || c >= chi) p[c] = 0.f;
            }
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) pk[c] = pack2<T>(p[2 * c], p[2 * c + 1]);
            tmem_st32(tS, pk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bar.p_full);
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.dp_full, t & 1, wd, 0x61));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t dr[32];
                tmem_ld32(tP + 32 * h2, dr);
                const float4 *d4 = reinterpret_cast<const float4 *>(dlt + 32 * h2);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 d = d4[q];
                    const int e = 32 * h2 + 4 * q;
                    pk[16 * h2 + 2 * q] = pack2<T>(p[e] * (__uint_as_float(dr[4 * q]) - d.x),
                                                   p[e + 1] * (__uint_as_float(dr[4 * q + 1]) - d.y));
                    pk[16 * h2 + 2 * q + 1] = pack2<T>(p[e + 2] * (__uint_as_float(dr[4 * q + 2]) - d.z),
                                                       p[e + 3] * (__uint_as_float(dr[4 * q + 3]) - d.w));
                }
            }
            tmem_st32(tP, pk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bar.ds_full);
        }
        // epilogue: dK (scaled) from warps 0-3, dV from warps 4-7
        if (ok && n_it > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bar.acc_done, 0, wd, 0x62));
        tc_fence_after();
        const MutView &ov = half == 0 ? a.dk : a.dv;
        T *dst = (T *)ov.ptr + (int64_t)b * ov.sb + (int64_t)(s.kv0 + key) * ov.ss + (int64_t)hk * ov.sh;
        const float mul = half == 0 ? g.scale : 1.f;
        const uint32_t base = tmem + (half == 0 ? C::kTmDK : C::kTmDV) + lane_off;
        // split query heads: this split's fp32 partial row instead, summed in
        // split order by a second kernel
        float *part = nullptr;
        if (a.dkv_part) {
            const int64_t krow = (g.thd ? 0 : (int64_t)b * g.Skv) + s.kv0 + key;
            const int64_t nrows = g.thd ? g.Skv : (int64_t)g.B * g.Skv;
            part = a.dkv_part + (((int64_t)(sp * 2 + half) * nrows + krow) * g.Hkv + hk) * D;
        }
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t v[32];
            if (n_it > 0) {
                tmem_ld32(base + cc * 32, v);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0u;
            }
            if (j < nkeys && (part || cc * 32 < g.D)) {
                if (part) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(part + cc * 32);
#pragma unroll
                    for (int e = 0; e < 8; ++e) d4[e] = make_uint4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                } else {
                    store_row32<T>(dst + cc * 32, v, mul);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ======================================================================= dQ
template <int D>
struct QCfg {
    static constexpr int KS = 3;  // key/value stages
    static constexpr int kTile = BLK * D * 2;
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKOff + KS * kTile;
    static constexpr int kBarOff = kVOff + KS * kTile;
    static constexpr int kSmemBytes = kBarOff + 256 + 1024;
    static constexpr int kTmQ = 0, kTmDO = D / 2, kTmS = D, kTmDP = D + 128, kTmDQ = D + 256;
};

struct QBars {
    uint64_t k_full[kMaxStages], k_empty[kMaxStages], v_full[kMaxStages], v_empty[kMaxStages];
    uint64_t qd_ready, s_full, s_free, dp_full, ds_full, dq_done;
    uint32_t tmem_base;
    int abort_flag;
};

// One unit of dQ work: 128 query rows of one (batch, query head), in the
// banded work order (rank 0 = the last query tile, most keys when causal).
struct QTile {
    int b, h, m0, nrows, jlo, nb;
    SeqInfo s;
};

__device__ __forceinline__ QTile q_tile(const Geometry &g, int w, int n_mtiles) {
    QTile t;
    int bh, rank;
    banded_order(w, n_mtiles, g.Hq * g.B, bh, rank);
    const int mt = n_mtiles - 1 - rank;
    t.h = bh % g.Hq;
    t.b = bh / g.Hq;
    t.s = seq_info(g, t.b);
    t.m0 = mt * BLK;
    t.nrows = max(0, min(BLK, t.s.Lq - t.m0));
    t.jlo = 0;
    t.nb = 0;
    if (t.nrows > 0) {
        int jhi;
        key_range(t.m0, t.m0 + t.nrows, t.s.Lkv, g.wl, g.wr, t.jlo, jhi);
        t.nb = (jhi - t.jlo + BLK - 1) / BLK;
    }
    return t;
}

// Each CTA walks work items blockIdx.x, blockIdx.x + gridDim.x, ...; barrier
// phases and pipeline stages carry over from one item to the next, so with
// fewer CTAs than items the next item's loads and MMAs overlap this item's
// epilogue.  The launcher gives one CTA per item, which balances uneven
// causal items better on this part.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     BwdArgs a, int n_mtiles) {
    using C = QCfg<D>;
    constexpr int KS = C::KS;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    QBars &bar = *reinterpret_cast<QBars *>(smem + C::kBarOff);
    const Geometry &g = a.g;
    const int n_work = n_mtiles * g.Hq * g.B;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < KS; ++i) {
            mbar_init(&bar.k_full[i], 1);
            mbar_init(&bar.k_empty[i], 1);
            mbar_init(&bar.v_full[i], 1);
            mbar_init(&bar.v_empty[i], 1);
        }
        mbar_init(&bar.qd_ready, kCompute);
        mbar_init(&bar.s_full, 1);
        mbar_init(&bar.s_free, kCompute);
        mbar_init(&bar.dp_full, 1);
        mbar_init(&bar.ds_full, kCompute);
        mbar_init(&bar.dq_done, 1);
        bar.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bar.tmem_base, 512);
        tmem_relinquish();
    }
    if (warp == kProdWarp && lane == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem_base;
    const Watchdog wd{a.watchdog_ns, a.err, &bar.abort_flag};

    if (warp == kProdWarp) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            int gb = 0;  // key blocks loaded so far (all items)
            bool ok = true;
            for (int w = blockIdx.x; ok && w < n_work; w += gridDim.x) {
                const QTile tl = q_tile(g, w, n_mtiles);
                const int cb = g.thd ? 0 : tl.b;
                const int hk = tl.h / g.G;
                const int kv_row = tl.s.kv0 + tl.jlo;
                for (int jb = 0; jb < tl.nb; ++jb, ++gb) {
                    const int st = gb % KS;
                    const uint32_t ph = (gb / KS) & 1;
                    if (!(ok = mbar_wait(&bar.k_empty[st], ph ^ 1, wd, 0x80))) break;
                    mbar_arrive_expect_tx(&bar.k_full[st], C::kTile);
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_4d(smem + C::kKOff + st * C::kTile + c * BLK * 128, &tm_k, &bar.k_full[st],
                                    c * 64, kv_row + jb * BLK, hk, cb);
                    if (!(ok = mbar_wait(&bar.v_empty[st], ph ^ 1, wd, 0x81))) break;
                    mbar_arrive_expect_tx(&bar.v_full[st], C::kTile);
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_4d(smem + C::kVOff + st * C::kTile + c * BLK * 128, &tm_v, &bar.v_full[st],
                                    c * 64, kv_row + jb * BLK, hk, cb);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA
        // Per block: S of the next block as soon as this block's S has been
        // read, dQ += dS K, then dP of the next block (its TMEM held dS, read
        // by the dQ MMA just before; MMAs of one thread run in issue order).
        // The whole warp runs the loop in step; one elected lane issues each
        // group of MMAs with its commit.
        {
            constexpr uint32_t idS = idesc_f16(BLK, BLK, kBf16, 0, 0);  // S, dP: A from TMEM
            constexpr uint32_t idQ = idesc_f16(BLK, D, kBf16, 0, 1);    // dQ: B = K, MN-major
            const uint32_t sK = smem_u32(smem + C::kKOff), sV = smem_u32(smem + C::kVOff);
            auto wait = [&](uint64_t *b, uint32_t ph, unsigned code) {
                const bool r = __all_sync(0xffffffffu, mbar_wait(b, ph, wd, code));
                if (r) tc_fence_after();
                return r;
            };
            auto commit = [&](uint64_t *b) {
                if (elect_one()) mma_commit(b);
                __syncwarp();
            };
            auto issue_s = [&](int gbk) {
                const uint64_t db = smem_desc_sw128(sK + (gbk % KS) * C::kTile, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ts(tmem + C::kTmS, tmem + C::kTmQ + kk * 8, desc_add(db, kmaj_off(kk, BLK)), idS,
                               kk > 0);
                    mma_commit(&bar.s_full);
                }
                __syncwarp();
            };
            auto issue_dp = [&](int gbk) {
                const uint64_t db = smem_desc_sw128(sV + (gbk % KS) * C::kTile, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ts(tmem + C::kTmDP, tmem + C::kTmDO + kk * 8, desc_add(db, kmaj_off(kk, BLK)), idS,
                               kk > 0);
                    mma_commit(&bar.dp_full);
                }
                __syncwarp();
            };
            int gb = 0, tn = 0;  // key blocks and non-empty items so far
            bool ok = true;
            for (int w = blockIdx.x; ok && w < n_work; w += gridDim.x) {
                const QTile tl = q_tile(g, w, n_mtiles);
                if (tl.nb == 0) continue;
                // Q and dO of this item are in TMEM (written after the previous
                // item's MMAs had all completed)
                if (!(ok = wait(&bar.qd_ready, tn & 1, 0x90))) break;
                if (!(ok = wait(&bar.k_full[gb % KS], (gb / KS) & 1, 0x91))) break;
                issue_s(gb);
                if (!(ok = wait(&bar.v_full[gb % KS], (gb / KS) & 1, 0x92))) break;
                issue_dp(gb);
                for (int jb = 0; ok && jb < tl.nb; ++jb) {
                    const int gbk = gb + jb, st = gbk % KS;
                    const bool next = jb + 1 < tl.nb;
                    const int st1 = (gbk + 1) % KS;
                    const uint32_t ph1 = ((gbk + 1) / KS) & 1;
                    if (next) {
                        if (!(ok = wait(&bar.k_full[st1], ph1, 0x93))) break;
                        if (!(ok = wait(&bar.s_free, gbk & 1, 0x94))) break;
                        issue_s(gbk + 1);
                    }
                    if (!(ok = wait(&bar.ds_full, gbk & 1, 0x95))) break;
                    const uint64_t dKm = smem_desc_sw128(sK + st * C::kTile, BLK * 128, 1024);
                    const uint32_t acc0 = jb > 0 ? 1u : 0u;
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < BLK / 16; ++kk)
                            mma_ts(tmem + C::kTmDQ, tmem + C::kTmDP + pcol(kk), desc_add(dKm, kk * 16 * 128), idQ,
                                   kk > 0 ? 1u : acc0);
                        mma_commit(&bar.k_empty[st]);
                        mma_commit(&bar.v_empty[st]);
                    }
                    __syncwarp();
                    if (next) {
                        if (!(ok = wait(&bar.v_full[st1], ph1, 0x96))) break;
                        issue_dp(gbk + 1);
                    }
                }
                if (!ok) break;
                commit(&bar.dq_done);
                gb += tl.nb;
                ++tn;
            }
        }
    } else {
        // --------------------------------------- P, dS (thread = query row)
        const int half = warp / 4;             // key columns [64 half, 64 half + 64)
        const int c0 = half * 64;
        const int r = (warp % 4) * 32 + lane;  // row within the tile
        const uint32_t lane_off = (uint32_t)((warp % 4) * 32) << 16;
        const uint32_t tS = tmem + C::kTmS + c0 + lane_off;
        const uint32_t tP = tmem + C::kTmDP + c0 + lane_off;
        const float c2 = g.scale_log2;
        int gb = 0, tn = 0;
        bool ok = true;
        // dq rows of the previous item, stored after the next item has started
        uint32_t pend[D / 2];
        T *pend_dst = nullptr;
        for (int w = blockIdx.x; ok && w < n_work; w += gridDim.x) {
            const QTile tl = q_tile(g, w, n_mtiles);
            if (tl.m0 == (n_mtiles - 1) * BLK && threadIdx.x == 0)
                report_uncovered(a.err, g, tl.s.Lq, n_mtiles * BLK, kErrSeqlenQ);
            if (tl.nrows == 0) continue;
            const int row = tl.m0 + r;
            T *dst = (T *)a.dq.ptr + (int64_t)tl.b * a.dq.sb + (int64_t)(tl.s.q0 + row) * a.dq.ss +
                     (int64_t)tl.h * a.dq.sh + half * (D / 2);
            if (tl.nb == 0) {  // no key visible to any row: dq = 0
                if (r < tl.nrows) {
                    uint32_t z[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) z[e] = 0u;
#pragma unroll
                    for (int cc = 0; cc < D / 64; ++cc)
                        if (half * (D / 2) + cc * 32 < g.D) store_row32<T>(dst + cc * 32, z, 1.f);
                }
                continue;
            }
            // Q (warps 0-3) or dO (warps 4-7) row into TMEM as an MMA operand
            {
                const View &src = half == 0 ? a.q : a.dout;
                const T *p = (const T *)src.ptr + (int64_t)tl.b * src.sb + (int64_t)(tl.s.q0 + row) * src.ss +
                             (int64_t)tl.h * src.sh;
                const uint32_t dstc = tmem + (half == 0 ? C::kTmQ : C::kTmDO) + lane_off;
#pragma unroll
                for (int cc = 0; cc < D / 64; ++cc) {
                    uint32_t v[32];
                    uint4 *v4 = reinterpret_cast<uint4 *>(v);
#pragma unroll
                    for (int e = 0; e < 8; ++e)  // (columns past the head dim: zero padding)
                        v4[e] = r < tl.nrows && cc * 64 + e * 8 < g.D ? reinterpret_cast<const uint4 *>(p + cc * 64)[e]
                                                                       : make_uint4(0, 0, 0, 0);
                    tmem_st32(dstc + cc * 32, v);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bar.qd_ready);
            }
            if (pend_dst) {  // previous item's dq, overlapping this item's first MMAs
#pragma unroll
                for (int cc = 0; cc < D / 64; ++cc)
                    if (half * (D / 2) + cc * 32 < g.D)
                        store_row32<T>(pend_dst + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&pend[cc * 32]),
                                       g.scale);
                pend_dst = nullptr;
            }
            float lse2 = 0.f, dlt = 0.f;
            if (r < tl.nrows) {
                const int64_t li = lse_index(g, tl.s, tl.b, tl.h, row);
                lse2 = a.lse[li] * kLog2e;
                dlt = a.delta[li];
            }
            const int rlo = tl.m0, rhi = tl.m0 + tl.nrows - 1;
            for (int jb = 0; jb < tl.nb; ++jb) {
                const int gbk = gb + jb;
                const int k0 = tl.jlo + jb * BLK + c0;  // first key of this half
                ok = __all_sync(0xffffffffu, mbar_wait(&bar.s_full, gbk & 1, wd, 0xa0));
                if (!ok) break;
                tc_fence_after();
                float p[64];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    uint32_t sr[32];
                    tmem_ld32(tS + 32 * h2, sr);
#pragma unroll
                    for (int c = 0; c < 32; ++c) p[32 * h2 + c] = __uint_as_float(sr[c]);
                }
                tc_fence_before();
                mbar_arrive(&bar.s_free);
                const bool full = (k0 + 63 < tl.s.Lkv) && (g.wr < 0 || k0 + 63 <= rlo + g.wr) &&
                                  (g.wl < 0 || k0 >= rhi - g.wl);
#pragma unroll
                for (int c = 0; c < 64; ++c) p[c] = ex2(fmaf(p[c], c2, -lse2));
                if (!full) {
                    // keys visible to this row: columns [vlo, vhi) of this half
                    int vlo = 0, vhi = min(64, tl.s.Lkv - k0);
                    if (g.wl >= 0) vlo = max(vlo, row - g.wl - k0);
                    if (g.wr >= 0) vhi = min(vhi, row + g.wr + 1 - k0);
                    if (row >= tl.s.Lq) vhi = vlo;
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (c < vlo || c >= vhi) p[c] = 0.f;
                }
                ok = __all_sync(0xffffffffu, mbar_wait(&bar.dp_full, gbk & 1, wd, 0xa1));
                if (!ok) break;
                tc_fence_after();
                uint32_t pk[32];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    uint32_t dr[32];
                    tmem_ld32(tP + 32 * h2, dr);
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int e = 32 * h2 + 2 * c;
                        pk[16 * h2 + c] = pack2<T>(p[e] * (__uint_as_float(dr[2 * c]) - dlt),
                                                   p[e + 1] * (__uint_as_float(dr[2 * c + 1]) - dlt));
                    }
                }
                tmem_st32(tP, pk);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bar.ds_full);
            }
            if (!ok) break;
            // dq of this item: read now (the next item reuses the TMEM), stored
            // once the next item's Q / dO are on their way
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.dq_done, tn & 1, wd, 0xa2));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc)
                tmem_ld32(tmem + C::kTmDQ + half * (D / 2) + cc * 32 + lane_off,
                          *reinterpret_cast<uint32_t(*)[32]>(&pend[cc * 32]));
            tc_fence_before();
            pend_dst = r < tl.nrows ? dst : nullptr;
            gb += tl.nb;
            ++tn;
        }
        if (pend_dst) {
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc)
                if (half * (D / 2) + cc * 32 < g.D)
                    store_row32<T>(pend_dst + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&pend[cc * 32]), g.scale);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <typename T, int D>
cudaError_t launch_typed(const BwdArgs &a, int max_lq, int max_lkv, int q_rows, cudaStream_t st) {
    const int dt = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;
    const Geometry &g = a.g;
    const uint64_t nb = g.thd ? 1 : (uint64_t)g.B;
    // inner extent: the real head dim (columns past it load as zeros)
    uint64_t dq[4] = {(uint64_t)g.D, (uint64_t)g.Sq, (uint64_t)g.Hq, nb};
    uint64_t dk[4] = {(uint64_t)g.D, (uint64_t)g.Skv, (uint64_t)g.Hkv, nb};
    auto strides = [&](const auto &v, const uint64_t dims[4], uint64_t out[3]) {
        tmap_strides(v.ss, v.sh, g.thd ? 0 : v.sb, dims, out);
    };
    uint64_t sq[3], sk[3], sv[3], sd[3];
    strides(a.q, dq, sq);
    strides(a.k, dk, sk);
    strides(a.v, dk, sv);
    strides(a.dout, dq, sd);
    CUtensorMap tq{}, tk{}, tv{}, tdo{};
    cudaError_t e;
    // every map and kernel attribute first: a refusal enqueues nothing
    const bool kv_pass = max_lkv > 0, q_pass = max_lq > 0;
    if (kv_pass || q_pass) {
        if (g.Sq > 0) {
            if ((e = make_tmap_16bit(&tq, a.q.ptr, dt, dq, sq, BLK)) != cudaSuccess) return e;
            if ((e = make_tmap_16bit(&tdo, a.dout.ptr, dt, dq, sd, BLK)) != cudaSuccess) return e;
        }
        if (g.Skv > 0) {
            if ((e = make_tmap_16bit(&tk, a.k.ptr, dt, dk, sk, BLK)) != cudaSuccess) return e;
            if ((e = make_tmap_16bit(&tv, a.v.ptr, dt, dk, sv, BLK)) != cudaSuccess) return e;
        }
    }
    auto kv_kern = tc_bwd_dkdv_kernel<T, D>;
    auto q_kern = tc_bwd_dq_kernel<T, D>;
    if (kv_pass && (e = cudaFuncSetAttribute(kv_kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             KVCfg<D>::kSmemBytes)) != cudaSuccess)
        return e;
    if (q_pass && (e = cudaFuncSetAttribute(q_kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            QCfg<D>::kSmemBytes)) != cudaSuccess)
        return e;
    const int n_ktiles = (max_lkv + BLK - 1) / BLK;
    const int64_t kv_grid = (int64_t)n_ktiles * g.Hkv * g.B * a.nsplit;
    const int n_mtiles = (max_lq + BLK - 1) / BLK;
    const int64_t n_work = (int64_t)n_mtiles * g.Hq * g.B;
    if (kv_grid > 0x7fffffff || n_work > 0x7fffffff) return cudaErrorInvalidConfiguration;
    if ((e = launch_bwd_preprocess(dt, a, q_rows, st)) != cudaSuccess) return e;
    if (kv_pass && kv_grid > 0) {
        prof_before(st, kProfBwdDkDv);
        kv_kern<<<(unsigned)kv_grid, kThreads, KVCfg<D>::kSmemBytes, st>>>(tq, tk, tv, tdo, a, n_ktiles);
        prof_after(st);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if (a.dkv_part && (e = launch_dkv_reduce(dt, a, st)) != cudaSuccess) return e;
    }
    if (q_pass && n_work > 0) {
        // one CTA per work item: the hardware dispatches them in work order as
        // SMs free up, which balances uneven (causal) items better than a
        // fixed assignment of items to resident CTAs
        prof_before(st, kProfBwdDq);
        q_kern<<<(int)n_work, kThreads, QCfg<D>::kSmemBytes, st>>>(tk, tv, a, n_mtiles);
        prof_after(st);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

bool uses_tc_bwd(int dtype, int D) {
    return (dtype == 0 || dtype == 1) && (D == 32 || D == 64 || D == 96 || D == 128);
}

cudaError_t launch_tc_bwd(int dtype, const BwdArgs &a, int max_lq, int max_lkv, int q_rows,
                          cudaStream_t st) {
    switch (dtype * 2 + (tc_dim(a.g.D) == 128)) {
        case 0: return launch_typed<__half, 64>(a, max_lq, max_lkv, q_rows, st);
        case 1: return launch_typed<__half, 128>(a, max_lq, max_lkv, q_rows, st);
        case 2: return launch_typed<__nv_bfloat16, 64>(a, max_lq, max_lkv, q_rows, st);
        case 3: return launch_typed<__nv_bfloat16, 128>(a, max_lq, max_lkv, q_rows, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gbattn
