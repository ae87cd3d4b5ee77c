// tc_bwd_fused64.cu -- single-pass tcgen05 backward attention, head dim 64.
//
// The same method as the head-dim-128 single pass (S and dP formed once per
// (query, key) pair, dV and dK owned by the CTA, each block's share of dQ
// added into an fp32 accumulator), laid out for D = 64, where TMEM has room
// for 128-query blocks and an untransposed dQ:
//   S^T  = K Q^T,  dP^T = V dO^T          (M = 128 keys, N = 128 queries;
//                                         K and V from TMEM)
//   P^T  = exp(scale S^T - LSE),  dS^T = P^T o (dP^T - delta)
//   dV  += P^T dO,  dK += dS^T Q          (P^T, dS^T from TMEM)
//   dQ   = dS K                           (M = 128 queries; dS from shared
//                                         memory as an MN-major A operand)
// so every product runs with M = 128 and the dQ drain holds query rows
// (thread = query row), which it writes as row-major boxes.
//
// One CTA per 128 keys of a (batch, key/value head); warps 0-7 copy K
// (warps 0-3) and V (warps 4-7) into TMEM, compute P and dS (thread = key
// row; warps 0-3 take query columns 0-63 of the block, warps 4-7 columns
// 64-127) and write dK / dV; warp 8 loads; warp 9 issues
// the MMAs (the whole warp runs the loop, an elected lane issues); warps
// 10-13 drain dQ (warp w: query rows [32 (w % 4), 32 (w % 4) + 32)).
//
// TMEM columns (512): dK 0-63, dV 64-127, S^T / P^T 128-255, dP^T / dS^T
// 256-383, dQ 384-447, K 448-479 and V 480-511 (bf16 pairs, the A operands
// of S^T and dP^T, which then take no shared-memory bandwidth).  MMA order per block t: dV_t, S^T_{t+1},
// dK_t, dQ_t, dP^T_{t+1}; dP^T_{t+1} overwrites dS^T_t after dK_t read it and
// is issued after dQ_t read dS_t from shared memory, so one dS^T buffer
// suffices (its next writer waits for dP^T_{t+1}).  Shared memory: K, V,
// three stages of Q and dO (16 KB each), dS^T (32 KB), eight 4 KB dQ staging
// boxes and the per-stage LSE / delta.
#include <type_traits>

#include "ptx.cuh"
#include "tc.h"
#include "tc_util.cuh"
#include "prof.h"
#include "tmap.h"

namespace gbattn {
namespace {

using namespace ptx;
using namespace tcu;

constexpr int D = 64;
constexpr int BK = 128;   // keys per CTA
constexpr int BQ = 128;   // query rows per block
constexpr int QS = 3;     // Q / dO stages
constexpr int kThreads = 448;
constexpr int kCompute = 256;
constexpr int kProdWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kDrainWarp0 = 10;
constexpr int kDrain = 128;
constexpr int kHeadBand = 4;

constexpr int kKVTile = BK * D * 2;   // 16 KB
constexpr int kQTile = BQ * D * 2;    // 16 KB
constexpr int kDSTile = BK * BQ * 2;  // 32 KB: two 64-query atoms
constexpr int kBox = 32 * 32 * 4;     // 4 KB: 32 query rows x 32 fp32
constexpr int kKOff = 0;
constexpr int kVOff = kKOff + kKVTile;
constexpr int kQOff = kVOff + kKVTile;
constexpr int kDOOff = kQOff + QS * kQTile;
constexpr int kDSOff = kDOOff + QS * kQTile;
constexpr int kStgOff = kDSOff + kDSTile;
constexpr int kStatOff = kStgOff + 8 * kBox;          // [QS][128] lse2, [QS][128] delta
constexpr int kBarOff = kStatOff + QS * BQ * 2 * 4;
constexpr int kSmemBytes = kBarOff + 256 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kTmDK = 0, kTmDV = 64, kTmS = 128, kTmDP = 256, kTmDQ = 384, kTmK = 448, kTmV = 480;

struct Bars {
    uint64_t kv_full;
    uint64_t q_full[QS], q_empty[QS];
    uint64_t kv_tmem, s_full, p_full, dp_full, ds_full;
    uint64_t dq_full, dq_free, acc_done;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// TMEM column of k-step kk (16 query columns) of packed P^T / dS^T: columns
// 0-63 of the block are packed into TMEM columns 0-31, 64-127 into 64-95.
__device__ __forceinline__ constexpr uint32_t pcol(int kk) { return (kk / 4) * 64 + (kk % 4) * 8; }

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd_fused64_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                          const __grid_constant__ CUtensorMap tm_acc, const __grid_constant__ CUtensorMap tm_dk,
                          const __grid_constant__ CUtensorMap tm_dv, BwdArgs a, int n_ktiles) {
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Bars &bar = *reinterpret_cast<Bars *>(smem + kBarOff);
    // Launched as a dependent of the preprocess: everything up to the first
    // read of its output (delta, the cleared dQ accumulator) overlaps its
    // tail; the dQ conversion may begin launching at once.
    griddep_launch();
    float *s_lse = reinterpret_cast<float *>(smem + kStatOff);  // log2 units
    float *s_delta = s_lse + QS * BQ;
    const Geometry &g = a.g;

    // (a split of the query heads of a group counts as a head of its own; the
    // splits of one key/value head are neighbours in the order)
    int bhs, kt;
    banded_order(blockIdx.x, n_ktiles, g.Hkv * g.B * a.nsplit, bhs, kt, kHeadBand);
    const int sp = bhs % a.nsplit, bh = bhs / a.nsplit;
    const int hk = bh % g.Hkv, b = bh / g.Hkv;
    const SeqInfo s = seq_info(g, b);
    const int n0 = kt * BK;
    if (kt == n_ktiles - 1 && sp == 0 && threadIdx.x == 0)
        report_uncovered(a.err, g, s.Lkv, n_ktiles * BK, kErrSeqlenKv);
    if (n0 >= s.Lkv) return;
    const int nkeys = min(BK, s.Lkv - n0);
    // query heads of this CTA: [h0, h0 + nh) of the group's G
    const int gs = (g.G + a.nsplit - 1) / a.nsplit;
    const int h0 = hk * g.G + sp * gs;
    const int nh = min(gs, g.G - sp * gs);

    int ilo, ihi;
    query_range(n0, n0 + nkeys, s.Lq, g.wl, g.wr, ilo, ihi);
    const int nqb = (ihi - ilo + BQ - 1) / BQ;
    const int n_it = nqb * nh;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        mbar_init(&bar.kv_full, 1);
        for (int i = 0; i < QS; ++i) {
            mbar_init(&bar.q_full[i], 32);
            mbar_init(&bar.q_empty[i], 1);
        }
        mbar_init(&bar.kv_tmem, kCompute);
        mbar_init(&bar.s_full, 1);
        mbar_init(&bar.p_full, kCompute);
        mbar_init(&bar.dp_full, 1);
        mbar_init(&bar.ds_full, kCompute);
        mbar_init(&bar.dq_full, 1);
        mbar_init(&bar.dq_free, kDrain);
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
        prefetch_tmap(&tm_acc);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem_base;
    const Watchdog wd{a.watchdog_ns, a.err, &bar.abort_flag};
    const int cb = g.thd ? 0 : b;

    if (warp == kProdWarp) {
        // ------------------------------------------------------------ loads
        if (n_it > 0) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&bar.kv_full, 2 * kKVTile);
                tma_load_4d(smem + kKOff, &tm_k, &bar.kv_full, 0, s.kv0 + n0, hk, cb);
                tma_load_4d(smem + kVOff, &tm_v, &bar.kv_full, 0, s.kv0 + n0, hk, cb);
            }
            griddep_wait();  // delta comes from the preprocess
            for (int t = 0; t < n_it; ++t) {
                const int st = t % QS;
                const uint32_t ph = (t / QS) & 1;
                const int h = h0 + t / nqb;
                const int i0 = ilo + (t % nqb) * BQ;
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
                if (!__all_sync(0xffffffffu, mbar_wait(&bar.q_empty[st], ph ^ 1, wd, 0xc8))) break;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    s_lse[st * BQ + lane + 32 * u] = lv[u];
                    s_delta[st * BQ + lane + 32 * u] = dv[u];
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bar.q_full[st], 2 * kQTile);
                    tma_load_4d(smem + kQOff + st * kQTile, &tm_q, &bar.q_full[st], 0, s.q0 + i0, h, cb);
                    tma_load_4d(smem + kDOOff + st * kQTile, &tm_do, &bar.q_full[st], 0, s.q0 + i0, h, cb);
                } else {
                    mbar_arrive(&bar.q_full[st]);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA
        if (n_it > 0) {
            constexpr uint32_t idSP = idesc_f16(BK, BQ, kBf16, 0, 0);  // S^T, dP^T
            constexpr uint32_t idKV = idesc_f16(BK, D, kBf16, 0, 1);   // dV, dK: B = dO / Q, MN-major
            constexpr uint32_t idQ = idesc_f16(BQ, D, kBf16, 1, 1);    // dQ: A = dS, B = K, MN-major
            const uint32_t sQ = smem_u32(smem + kQOff), sDO = smem_u32(smem + kDOOff);
            const uint64_t dKm = smem_desc_sw128(smem_u32(smem + kKOff), BK * 128, 1024);  // B of dQ
            const uint64_t dSm = smem_desc_sw128(smem_u32(smem + kDSOff), BK * 128, 1024); // A of dQ
            auto wait = [&](uint64_t *bb, uint32_t ph, unsigned code) {
                const bool r = __all_sync(0xffffffffu, mbar_wait(bb, ph, wd, code));
                if (r) tc_fence_after();
                return r;
            };
            auto issue_s = [&](int t) {
                const uint64_t db = smem_desc_sw128(sQ + (t % QS) * kQTile, 16, 1024);
                if (elect_one()) {
                    // k-step kk: head dims [16 kk, 16 kk + 16) = TMEM columns [8 kk, 8 kk + 8)
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ts(tmem + kTmS, tmem + kTmK + kk * 8, desc_add(db, kmaj_off(kk, BQ)), idSP, kk > 0);
                    mma_commit(&bar.s_full);
                }
                __syncwarp();
            };
            auto issue_dp = [&](int t) {
                const uint64_t db = smem_desc_sw128(sDO + (t % QS) * kQTile, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ts(tmem + kTmDP, tmem + kTmV + kk * 8, desc_add(db, kmaj_off(kk, BQ)), idSP, kk > 0);
                    mma_commit(&bar.dp_full);
                }
                __syncwarp();
            };
            bool ok = wait(&bar.kv_full, 0, 0xd8) && wait(&bar.kv_tmem, 0, 0xde) && wait(&bar.q_full[0], 0, 0xd9);
            if (ok) {
                issue_s(0);
                issue_dp(0);
            }
            for (int t = 0; ok && t < n_it; ++t) {
                const int st = t % QS;
                const bool next = t + 1 < n_it;
                // Q_t / dO_t as MN-major B operands (N = head dim, one 64-wide atom)
                const uint64_t dOm = smem_desc_sw128(sDO + st * kQTile, BQ * 128, 1024);
                const uint64_t dQm = smem_desc_sw128(sQ + st * kQTile, BQ * 128, 1024);
                const uint32_t acc0 = t > 0 ? 1u : 0u;
                if (!(ok = wait(&bar.p_full, t & 1, 0xda))) break;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BQ / 16; ++kk)
                        mma_ts(tmem + kTmDV, tmem + kTmS + pcol(kk), desc_add(dOm, kk * 16 * 128), idKV,
                               kk > 0 ? 1u : acc0);
                }
                __syncwarp();
                if (next) {
                    if (!(ok = wait(&bar.q_full[(t + 1) % QS], ((t + 1) / QS) & 1, 0xdb))) break;
                    issue_s(t + 1);
                }
                if (!(ok = wait(&bar.ds_full, t & 1, 0xdc))) break;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BQ / 16; ++kk)
                        mma_ts(tmem + kTmDK, tmem + kTmDP + pcol(kk), desc_add(dQm, kk * 16 * 128), idKV,
                               kk > 0 ? 1u : acc0);
                    mma_commit(&bar.q_empty[st]);
                }
                __syncwarp();
                if (t > 0 && !(ok = wait(&bar.dq_free, (t - 1) & 1, 0xdd))) break;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)  // K = keys: 16 key rows per step
                        mma_ss(tmem + kTmDQ, desc_add(dSm, kk * 16 * 128), desc_add(dKm, kk * 16 * 128), idQ, kk > 0);
                    mma_commit(&bar.dq_full);
                }
                __syncwarp();
                if (next) issue_dp(t + 1);
            }
            if (ok && elect_one()) mma_commit(&bar.acc_done);
            __syncwarp();
        }
    } else if (warp < kProdWarp) {
        // --------------------------------------- P, dS (thread = key row)
        const int half = warp / 4;             // query columns [64 half, 64 half + 64)
        const int c0 = half * 64;
        const int j = (warp % 4) * 32 + lane;
        const int key = n0 + j;
        const uint32_t lane_off = (uint32_t)((warp % 4) * 32) << 16;
        const uint32_t tS = tmem + kTmS + c0 + lane_off;
        const uint32_t tP = tmem + kTmDP + c0 + lane_off;
        // dS^T row j, query atom `half` (64 queries = 128 B per row)
        const uint32_t sDSrow = smem_u32(smem + kDSOff) + half * (BK * 128) + j * 128;
        const float c2 = g.scale_log2;
        bool ok = true;
        if (n_it > 0) {
            // row j of K (warps 0-3) or V (warps 4-7) into TMEM as bf16 pairs:
            // 16-byte chunk c of the swizzled row sits at c ^ (j % 8)
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.kv_full, 0, wd, 0xeb));
            if (ok) {
                const uint8_t *row = smem + (half == 0 ? kKOff : kVOff) + j * 128;
                uint32_t kr[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 x = *reinterpret_cast<const uint4 *>(row + ((c ^ (j & 7)) << 4));
                    kr[4 * c] = x.x;
                    kr[4 * c + 1] = x.y;
                    kr[4 * c + 2] = x.z;
                    kr[4 * c + 3] = x.w;
                }
                tmem_st32(tmem + (half == 0 ? kTmK : kTmV) + lane_off, kr);
                tmem_wait_st();
                tc_fence_before();
            }
            mbar_arrive(&bar.kv_tmem);
        }
        for (int t = 0; ok && t < n_it; ++t) {
            const int st = t % QS;
            const int i0 = ilo + (t % nqb) * BQ + c0;
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.s_full, t & 1, wd, 0xe8));
            if (!ok) break;
            tc_fence_after();
            const float *lse2 = s_lse + st * BQ + c0;
            const float *dlt = s_delta + st * BQ + c0;
            const bool full = (i0 + 63 < s.Lq) && (n0 + BK - 1 < s.Lkv) &&
                              (g.wr < 0 || n0 + BK - 1 <= i0 + g.wr) && (g.wl < 0 || n0 >= i0 + 63 - g.wl);
            float p[64];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t sr[32];
                tmem_ld32(tS + 32 * h2, sr);
                // 16-byte broadcast reads of the LSE (shared memory bandwidth
                // is shared with the MMA operand reads)
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
                int clo = 0, chi = min(64, s.Lq - i0);
                if (g.wr >= 0) clo = max(clo, key - g.wr - i0);
                if (g.wl >= 0) chi = min(chi, key + g.wl + 1 - i0);
                if (key >= s.Lkv) chi = clo;
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (c < clo || c >= chi) p[c] = 0.f;
            }
            {
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) pk[c] = pack2<T>(p[2 * c], p[2 * c + 1]);
                tmem_st32(tS, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bar.p_full);
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.dp_full, t & 1, wd, 0xe9));
            if (!ok) break;
            tc_fence_after();
            // dS^T_t: packed over dP^T_t in TMEM (A of dK) and into shared
            // memory (A of dQ); the shared copy was last read by dQ_{t-1},
            // issued before dP^T_t, whose completion we saw
            uint32_t pk[32];
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
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)  // 128B swizzle: 16-byte chunk cc of row j
                st_shared_v4(sDSrow + ((uint32_t)(cc ^ (j & 7)) << 4), pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2],
                             pk[4 * cc + 3]);
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar.ds_full);
        }
        // epilogue: dK (scaled) from warps 0-3, dV from warps 4-7, staged in
        // the idle K / V tile and written with TMA stores (THD tiles ending
        // inside the tensor are written row by row)
        if (ok && n_it > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bar.acc_done, 0, wd, 0xea));
        tc_fence_after();
        const float mul = half == 0 ? g.scale : 1.f;
        const uint32_t base = tmem + (half == 0 ? kTmDK : kTmDV) + lane_off;
        uint32_t v[64];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            if (n_it > 0) {
                tmem_ld32(base + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * cc]));
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[32 * cc + e] = 0u;
            }
        }
        if (a.dkv_part) {
            // split query heads: this split's fp32 partial row, summed by a
            // second kernel
            if (j < nkeys) {
                const int64_t krow = (g.thd ? 0 : (int64_t)b * g.Skv) + s.kv0 + key;
                const int64_t nrows = g.thd ? g.Skv : (int64_t)g.B * g.Skv;
                float *dst = a.dkv_part + (((int64_t)(sp * 2 + half) * nrows + krow) * g.Hkv + hk) * D;
                store_f32_row32(dst, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                store_f32_row32(dst + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            }
        } else if (!g.thd || nkeys == BK) {
            uint8_t *stage = smem + (half == 0 ? kKOff : kVOff);
            const uint32_t srow = smem_u32(stage) + j * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = pack2<T>(__uint_as_float(v[8 * q + 2 * e]) * mul, __uint_as_float(v[8 * q + 2 * e + 1]) * mul);
                st_shared_v4(srow + ((uint32_t)(q ^ (j & 7)) << 4), w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async_smem();
            named_bar_sync(1 + half, 128);
            if (warp % 4 == 0 && lane == 0) {
                tma_store_4d(half == 0 ? &tm_dk : &tm_dv, stage, 0, s.kv0 + n0, hk, cb);
                bulk_commit();
                bulk_wait_read0();  // the copy has read the staging before the CTA exits
            }
        } else if (j < nkeys) {
            const MutView &ov = half == 0 ? a.dk : a.dv;
            T *dstp = (T *)ov.ptr + (int64_t)b * ov.sb + (int64_t)(s.kv0 + key) * ov.ss + (int64_t)hk * ov.sh;
            store_row32<T>(dstp, *reinterpret_cast<uint32_t(*)[32]>(&v[0]), mul);
            if (g.D > 32) store_row32<T>(dstp + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]), mul);
        }
    } else if (warp >= kDrainWarp0) {
        // ------------------------------------- dQ drain (thread = query row)
        griddep_wait();  // the accumulator is cleared by the preprocess
        const int qd = warp % 4;  // TMEM lane quarter = query rows [32 qd, 32 qd + 32)
        const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
        const uint32_t box0 = smem_u32(smem + kStgOff) + qd * 2 * kBox;  // head dims 0-31, then 32-63
        const int zb = g.thd ? 0 : b * g.Hq;
        bool ok = true;
        for (int t = 0; t < n_it; ++t) {
            const int h = h0 + t / nqb;
            const int i0 = ilo + (t % nqb) * BQ;
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.dq_full, t & 1, wd, 0xf8));
            if (!ok) break;
            tc_fence_after();
            uint32_t v[64];
            tmem_ld32(tmem + kTmDQ + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld32(tmem + kTmDQ + 32 + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tc_fence_before();
            mbar_arrive(&bar.dq_free);
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
            // box row = lane (query i0 + 32 qd + lane), 128B swizzle
#pragma unroll
            for (int bx = 0; bx < 2; ++bx)
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_shared_v4(box0 + bx * kBox + lane * 128 + ((uint32_t)(c ^ (lane & 7)) << 4),
                                 v[32 * bx + 4 * c], v[32 * bx + 4 * c + 1], v[32 * bx + 4 * c + 2],
                                 v[32 * bx + 4 * c + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_reduce_add_3d(box0, &tm_acc, 0, s.q0 + i0 + 32 * qd, zb + h);
                tma_reduce_add_3d(box0 + kBox, &tm_acc, 32, s.q0 + i0 + 32 * qd, zb + h);
                bulk_commit();
            }
        }
        // the reductions must have read their boxes before the CTA's shared
        // memory goes away (their additions complete with the grid)
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <typename T>
cudaError_t launch_typed(const BwdArgs &a, int max_lkv, int q_rows, cudaStream_t st) {
    const int dt = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;
    const Geometry &g = a.g;
    const uint64_t nb = g.thd ? 1 : (uint64_t)g.B;
    // inner extent: the real head dim (columns past it load as zeros)
    uint64_t dq[4] = {(uint64_t)g.D, (uint64_t)g.Sq, (uint64_t)g.Hq, nb};
    uint64_t dk[4] = {(uint64_t)g.D, (uint64_t)g.Skv, (uint64_t)g.Hkv, nb};
    auto strides = [&](const auto &v, const uint64_t dims[4], uint64_t out[3]) {
        tmap_strides(v.ss, v.sh, g.thd ? 0 : v.sb, dims, out);
    };
    const uint64_t acc_rows = g.thd ? (uint64_t)g.Tq : (uint64_t)g.Sq;
    const uint64_t acc_heads = g.thd ? (uint64_t)g.Hq : (uint64_t)g.B * g.Hq;
    cudaError_t e;
    if (max_lkv > 0) {
        uint64_t sq[3], sk[3], sv[3], sd[3], sgk[3], sgv[3];
        strides(a.q, dq, sq);
        strides(a.k, dk, sk);
        strides(a.v, dk, sv);
        strides(a.dout, dq, sd);
        strides(a.dk, dk, sgk);
        strides(a.dv, dk, sgv);
        CUtensorMap tq, tk, tv, tdo, tacc, tgk, tgv;
        if ((e = make_tmap_16bit(&tq, a.q.ptr, dt, dq, sq, BQ)) != cudaSuccess) return e;
        if ((e = make_tmap_16bit(&tk, a.k.ptr, dt, dk, sk, BK)) != cudaSuccess) return e;
        if ((e = make_tmap_16bit(&tv, a.v.ptr, dt, dk, sv, BK)) != cudaSuccess) return e;
        if ((e = make_tmap_16bit(&tdo, a.dout.ptr, dt, dq, sd, BQ)) != cudaSuccess) return e;
        if ((e = make_tmap_f32_acc(&tacc, a.dq_acc, D, acc_rows, acc_heads, 32, 32)) != cudaSuccess) return e;
        if ((e = make_tmap_16bit(&tgk, a.dk.ptr, dt, dk, sgk, BK)) != cudaSuccess) return e;
        if ((e = make_tmap_16bit(&tgv, a.dv.ptr, dt, dk, sgv, BK)) != cudaSuccess) return e;
        auto kern = tc_bwd_fused64_kernel<T>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)) !=
            cudaSuccess)
            return e;
        if ((e = launch_bwd_preprocess(dt, a, q_rows, st)) != cudaSuccess) return e;
        const int n_ktiles = (max_lkv + BK - 1) / BK;
        const int64_t grid = (int64_t)n_ktiles * g.Hkv * g.B * a.nsplit;
        if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
        prof_before(st, kProfBwdFused);
        e = launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), kSmemBytes, st, tq, tk, tv, tdo, tacc, tgk, tgv, a,
                       n_ktiles);
        prof_after(st);
        if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) return e;
        if (a.dkv_part && (e = launch_dkv_reduce(dt, a, st)) != cudaSuccess) return e;
    } else if ((e = launch_bwd_preprocess(dt, a, q_rows, st)) != cudaSuccess) {
        return e;
    }
    return launch_dq_convert(dt, a, st);
}

}  // namespace

cudaError_t launch_tc_bwd_fused64(int dtype, const BwdArgs &a, int max_lkv, int q_rows, cudaStream_t st) {
    if (tc_dim(a.g.D) != D || !a.dq_acc) return cudaErrorInvalidValue;
    switch (dtype) {
        case 0: return launch_typed<__half>(a, max_lkv, q_rows, st);
        case 1: return launch_typed<__nv_bfloat16>(a, max_lkv, q_rows, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gbattn
