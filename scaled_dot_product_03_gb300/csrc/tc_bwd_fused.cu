// tc_bwd_fused.cu -- single-pass tcgen05 backward attention, head dim 128.
//
// One CTA per 128 keys of a (batch, key/value head).  K and V stay in shared
// memory while the CTA walks the 64-row query blocks of every query head of
// the group that sees its keys; per block (keys j, queries i):
//   S^T  = K Q^T                          (K from TMEM, Q from shared memory)
//   dP^T = V dO^T                         (both operands from shared memory)
//   P^T  = exp(scale S^T - LSE)           recomputed from the forward's LSE
//   dS^T = P^T o (dP^T - delta)           delta_i = <dO_i, O_i> (preprocess)
//   dV  += P^T dO                         (P^T from TMEM)
//   dK  += dS^T Q                         (dS^T from TMEM)
//   dQ^T = K^T dS^T                       this block's share of dQ (dS^T
//                                         from shared memory)
// S and dP are formed once per (query, key) pair, so the pass executes the
// five products of the method and nothing more.  dQ sums over every key
// tile, i.e. over CTAs: each block's share is staged in shared memory and
// added into an fp32 accumulator in global memory with TMA bulk
// reduce-adds (one instruction per 8 KB box; per-element red.global, as fast
// at the L2, costs the draining warps about 1 us of issue per block), and a
// small kernel scales and converts the sums at the end.  The order of those fp32 additions depends on scheduling, so
// dQ is reproducible only to rounding; dK and dV are owned by one CTA each.
//
// Warp roles (448 threads): warps 0-7 copy K into TMEM, compute P and dS
// (thread = key row; warps 0-3 take query columns 0-31 of the block, warps
// 4-7 columns 32-63) and write dK at the end; warp 8 issues TMA loads; warp
// 9 allocates TMEM and issues the MMAs; warps 10-13 drain dQ^T from TMEM
// (thread = head dim) into shared memory and issue the reductions, warp w
// owning head dims [32 (w % 4), 32 (w % 4) + 32), which is the TMEM lane
// quarter it may read, and one 64 x 32 fp32 staging box, and write dV at
// the end.  dK and dV leave in parallel, each warp staging 32-row boxes in
// the then idle K / V tiles for TMA stores.
//
// TMEM columns (512): dK 0-127, dV 128-255, S^T / P^T 256-319, dP^T / dS^T
// 320-383, dQ^T 384-447, and K 448-511 (bf16 pairs, written once by the
// compute warps) as the A operand of S^T: operands read from TMEM do not
// use the shared-memory port, which the five products' shared-memory
// operands and the warps' own traffic otherwise fill.  Shared memory: K, V
// (32 KB each), three stages of Q and dO (16 KB each), two dS^T buffers
// (16 KB each), the dQ staging boxes (32 KB) and the per-stage LSE / delta.
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

constexpr int D = 128;
constexpr int BK = 128;   // keys per CTA
constexpr int BQ = 64;    // query rows per block
constexpr int QS = 3;     // Q / dO stages
constexpr int kThreads = 448;
constexpr int kCompute = 256;
constexpr int kProdWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kDrainWarp0 = 10;
constexpr int kDrain = 128;
constexpr int kFusedHeadBand = 4;  // heads per band of the work order (see banded_order)

constexpr int kKVTile = BK * D * 2;   // 32 KB
constexpr int kQTile = BQ * D * 2;    // 16 KB
constexpr int kDSTile = BK * BQ * 2;  // 16 KB
constexpr int kBox = BQ * 32 * 4;     // 8 KB: 64 rows x 32 fp32
constexpr int kKOff = 0;
constexpr int kVOff = kKOff + kKVTile;
constexpr int kQOff = kVOff + kKVTile;
constexpr int kDOOff = kQOff + QS * kQTile;
constexpr int kDSOff = kDOOff + QS * kQTile;
constexpr int kStgOff = kDSOff + 2 * kDSTile;
constexpr int kStatOff = kStgOff + 4 * kBox;          // [QS][64] lse2, [QS][64] delta
constexpr int kBarOff = kStatOff + QS * BQ * 2 * 4;
constexpr int kSmemBytes = kBarOff + 256 + 1024;      // + barriers + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kTmDK = 0, kTmDV = 128, kTmS = 256, kTmDP = 320, kTmDQ = 384, kTmK = 448;

struct Bars {
    uint64_t kv_full;
    uint64_t q_full[QS], q_empty[QS];
    uint64_t k_tmem, s_full, p_full;
    uint64_t dp_full, ds_full;
    uint64_t dq_full, dq_free, acc_done;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// TMEM column of k-step kk (16 query columns) of packed P^T or dS^T: columns
// 0-31 of the block are packed into TMEM columns 0-15, 32-63 into 32-47.
__device__ __forceinline__ constexpr uint32_t pcol(int kk) { return (kk / 2) * 32 + (kk % 2) * 8; }
__device__ __forceinline__ void st_shared_f32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
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

    // banded work order; rank 0 = the first key tiles (seen by the most
    // queries when causal)
    // (a split of the query heads of a group counts as a head of its own; the
    // splits of one key/value head are neighbours in the order)
    int bhs, kt;
    banded_order(blockIdx.x, n_ktiles, g.Hkv * g.B * a.nsplit, bhs, kt, kFusedHeadBand);
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
    const int nqb = (ihi - ilo + BQ - 1) / BQ;  // query blocks per head
    const int n_it = nqb * nh;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cb = g.thd ? 0 : b;  // TMA batch coordinate
    // Block t's LSE (log2 units) and delta into stage t % QS, then its Q and
    // dO loads (the whole producer warp; lane 0 arms the stage).  With a
    // watchdog, the stage's previous block must have been consumed first;
    // the statistics are fetched before that wait.
    auto stage_block = [&](int t, const Watchdog *w) {
        const int st = t % QS;
        const uint32_t ph = (t / QS) & 1;
        const int h = h0 + t / nqb;
        const int i0 = ilo + (t % nqb) * BQ;
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
        if (w && !__all_sync(0xffffffffu, mbar_wait(&bar.q_empty[st], ph ^ 1, *w, 0xc0))) return false;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            s_lse[st * BQ + lane + 32 * u] = lv[u];
            s_delta[st * BQ + lane + 32 * u] = dv[u];
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive_expect_tx(&bar.q_full[st], 2 * kQTile);
            for (int c = 0; c < D / 64; ++c) {
                tma_load_4d(smem + kQOff + st * kQTile + c * BQ * 128, &tm_q, &bar.q_full[st], c * 64, s.q0 + i0, h,
                            cb);
                tma_load_4d(smem + kDOOff + st * kQTile + c * BQ * 128, &tm_do, &bar.q_full[st], c * 64, s.q0 + i0,
                            h, cb);
            }
        } else {
            mbar_arrive(&bar.q_full[st]);
        }
        return true;
    };
    if (warp == kProdWarp) {
        // The producer warp sets up the barriers and issues K, V and the first
        // block's loads at once, so they overlap the TMEM allocation and the
        // block-wide sync (stage 0 is free).
        if (lane == 0) {
            mbar_init(&bar.kv_full, 1);
            for (int i = 0; i < QS; ++i) {
                mbar_init(&bar.q_full[i], 32);
                mbar_init(&bar.q_empty[i], 1);
            }
            mbar_init(&bar.k_tmem, kCompute);
            mbar_init(&bar.s_full, 1);
            mbar_init(&bar.p_full, kCompute);
            mbar_init(&bar.dp_full, 1);
            mbar_init(&bar.ds_full, kCompute);
            mbar_init(&bar.dq_full, 1);
            mbar_init(&bar.dq_free, kDrain);
            mbar_init(&bar.acc_done, 1);
            bar.abort_flag = 0;
            fence_mbar_init();
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do);
            prefetch_tmap(&tm_acc);
        }
        __syncwarp();
        if (n_it > 0) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&bar.kv_full, 2 * kKVTile);
                for (int c = 0; c < D / 64; ++c) {
                    tma_load_4d(smem + kKOff + c * BK * 128, &tm_k, &bar.kv_full, c * 64, s.kv0 + n0, hk, cb);
                    tma_load_4d(smem + kVOff + c * BK * 128, &tm_v, &bar.kv_full, c * 64, s.kv0 + n0, hk, cb);
                }
            }
            griddep_wait();  // delta comes from the preprocess
            stage_block(0, nullptr);
        }
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bar.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem_base;
    const Watchdog wd{a.watchdog_ns, a.err, &bar.abort_flag};

    if (warp == kProdWarp) {
        // ------------------------------------------------------------ loads
        for (int t = 1; t < n_it; ++t)
            if (!stage_block(t, &wd)) break;
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA
        // Per block t: dV_t (once P_t is written), S^T_{t+1} (its TMEM held
        // P_t, read by dV_t just before: MMAs of one thread execute in issue
        // order), then, once dS_t is in TMEM and shared memory, dK_t,
        // dP^T_{t+1} (its TMEM held dS^T_t, read by dK_t just before) and
        // dQ^T_t.
        // The whole warp runs the loop (waits, operand descriptors) in step;
        // one elected lane issues each group of MMAs and its commit.
        if (n_it > 0) {
            constexpr uint32_t idSP = idesc_f16(BK, BQ, kBf16, 0, 0);  // S^T, dP^T
            constexpr uint32_t idKV = idesc_f16(BK, D, kBf16, 0, 1);   // dV, dK: B = dO / Q, MN-major
            constexpr uint32_t idQ = idesc_f16(D, BQ, kBf16, 1, 1);    // dQ^T: A = K, B = dS^T, MN-major
            const uint32_t sQ = smem_u32(smem + kQOff), sDO = smem_u32(smem + kDOOff);
            const uint32_t sDS = smem_u32(smem + kDSOff);
            const uint64_t dV = smem_desc_sw128(smem_u32(smem + kVOff), 16, 1024);
            // K as the MN-major A operand of dQ^T (M = head dim, two 64-wide atoms)
            const uint64_t dKm = smem_desc_sw128(smem_u32(smem + kKOff), BK * 128, 1024);
            auto wait = [&](uint64_t *b, uint32_t ph, unsigned code) {
                const bool r = __all_sync(0xffffffffu, mbar_wait(b, ph, wd, code));
                if (r) tc_fence_after();
                return r;
            };
            auto issue_s = [&](int t) {
                const uint64_t db = smem_desc_sw128(sQ + (t % QS) * kQTile, 16, 1024);
                if (elect_one()) {
                    // k-step kk of K: head dims [16 kk, 16 kk + 16) = TMEM columns [8 kk, 8 kk + 8)
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
                        mma_ss(tmem + kTmDP, desc_add(dV, kmaj_off(kk, BK)), desc_add(db, kmaj_off(kk, BQ)), idSP,
                               kk > 0);
                    mma_commit(&bar.dp_full);
                }
                __syncwarp();
            };
            bool ok = wait(&bar.kv_full, 0, 0xd0) && wait(&bar.k_tmem, 0, 0xd6) && wait(&bar.q_full[0], 0, 0xd1);
            if (ok) {
                issue_s(0);
                issue_dp(0);
            }
            for (int t = 0; ok && t < n_it; ++t) {
                const int st = t % QS;
                const bool next = t + 1 < n_it;
                // Q_t / dO_t as MN-major B operands (N = head dim, two 64-wide atoms)
                const uint64_t dOm = smem_desc_sw128(sDO + st * kQTile, BQ * 128, 1024);
                const uint64_t dQm = smem_desc_sw128(sQ + st * kQTile, BQ * 128, 1024);
                const uint32_t acc0 = t > 0 ? 1u : 0u;
                if (!(ok = wait(&bar.p_full, t & 1, 0xd2))) break;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BQ / 16; ++kk)
                        mma_ts(tmem + kTmDV, tmem + kTmS + pcol(kk), desc_add(dOm, kk * 16 * 128), idKV,
                               kk > 0 ? 1u : acc0);
                }
                __syncwarp();
                if (next) {
                    if (!(ok = wait(&bar.q_full[(t + 1) % QS], ((t + 1) / QS) & 1, 0xd3))) break;
                    issue_s(t + 1);
                }
                if (!(ok = wait(&bar.ds_full, t & 1, 0xd4))) break;
                // dS^T_t: A of dK from TMEM (packed over dP^T_t), MN-major B of
                // dQ^T from shared memory (N = queries)
                const uint64_t dSm = smem_desc_sw128(sDS + (t & 1) * kDSTile, BK * 128, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BQ / 16; ++kk)
                        mma_ts(tmem + kTmDK, tmem + kTmDP + pcol(kk), desc_add(dQm, kk * 16 * 128), idKV,
                               kk > 0 ? 1u : acc0);
                    mma_commit(&bar.q_empty[st]);
                }
                __syncwarp();
                if (next) issue_dp(t + 1);
                if (t > 0 && !(ok = wait(&bar.dq_free, (t - 1) & 1, 0xd5))) break;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_ss(tmem + kTmDQ, desc_add(dKm, kk * 16 * 128), desc_add(dSm, kk * 16 * 128), idQ, kk > 0);
                    mma_commit(&bar.dq_full);
                }
                __syncwarp();
            }
            if (ok && elect_one()) mma_commit(&bar.acc_done);
            __syncwarp();
        }
    } else if (warp < kProdWarp) {
        // --------------------------------------- P, dS (thread = key row)
        const int half = warp / 4;             // query columns [32 half, 32 half + 32)
        const int c0 = half * 32;
        const int j = (warp % 4) * 32 + lane;  // key within the tile
        const int key = n0 + j;
        const uint32_t lane_off = (uint32_t)((warp % 4) * 32) << 16;
        const uint32_t tS = tmem + kTmS + c0 + lane_off;
        const uint32_t sDSrow = smem_u32(smem + kDSOff) + j * 128;
        const float c2 = g.scale_log2;
        bool ok = true;
        if (n_it > 0) {
            // K row j into TMEM as bf16 pairs: this half's head dims [64 half,
            // 64 half + 64) are atom `half` of the swizzled tile (16-byte chunk
            // c of the row at c ^ (j % 8)), TMEM columns [32 half, 32 half + 32)
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.kv_full, 0, wd, 0xe3));
            if (ok) {
                const uint8_t *krow = smem + kKOff + half * (BK * 128) + j * 128;
                uint32_t kr[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 x = *reinterpret_cast<const uint4 *>(krow + ((c ^ (j & 7)) << 4));
                    kr[4 * c] = x.x;
                    kr[4 * c + 1] = x.y;
                    kr[4 * c + 2] = x.z;
                    kr[4 * c + 3] = x.w;
                }
                tmem_st32(tmem + kTmK + half * 32 + lane_off, kr);
                tmem_wait_st();
                tc_fence_before();
            }
            mbar_arrive(&bar.k_tmem);
        }
        for (int t = 0; ok && t < n_it; ++t) {
            const int st = t % QS;
            const int i0 = ilo + (t % nqb) * BQ + c0;  // first query row of this half
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.s_full, t & 1, wd, 0xe0));
            if (!ok) break;
            tc_fence_after();
            // (LSE / delta of stage st were written before q_full completed,
            // which S^T_t itself waited for)
            const float *lse2 = s_lse + st * BQ + c0;
            const float *dlt = s_delta + st * BQ + c0;
            const bool full = (i0 + 31 < s.Lq) && (n0 + BK - 1 < s.Lkv) &&
                              (g.wr < 0 || n0 + BK - 1 <= i0 + g.wr) && (g.wl < 0 || n0 >= i0 + 31 - g.wl);
            float p[32];
            {
                // LSE of the 32 columns as 16-byte broadcast reads (fewer
                // shared memory wavefronts)
                uint32_t sr[32];
                tmem_ld32(tS, sr);
                const float4 *l4 = reinterpret_cast<const float4 *>(lse2);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 l = l4[q];
                    p[4 * q] = ex2(fmaf(__uint_as_float(sr[4 * q]), c2, -l.x));
                    p[4 * q + 1] = ex2(fmaf(__uint_as_float(sr[4 * q + 1]), c2, -l.y));
                    p[4 * q + 2] = ex2(fmaf(__uint_as_float(sr[4 * q + 2]), c2, -l.z));
                    p[4 * q + 3] = ex2(fmaf(__uint_as_float(sr[4 * q + 3]), c2, -l.w));
                }
            }
            if (!full) {
                // queries that see this key: columns [clo, chi) of this half
                int clo = 0, chi = min(32, s.Lq - i0);
                if (g.wr >= 0) clo = max(clo, key - g.wr - i0);
                if (g.wl >= 0) chi = min(chi, key + g.wl + 1 - i0);
                if (key >= s.Lkv) chi = clo;
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if (c < clo || c >= chi) p[c] = 0.f;
            }
            {
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) pk[c] = pack2<T>(p[2 * c], p[2 * c + 1]);
                tmem_st16(tS, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bar.p_full);
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.dp_full, t & 1, wd, 0xe1));
            if (!ok) break;
            tc_fence_after();
            // dS^T_t packed over dP^T_t in TMEM (A of dK) and into shared memory
            // (B of dQ^T; the buffer was last read by dQ^T_{t-2}, issued
            // before dP^T_t, whose completion we saw)
            const uint32_t tDP = tmem + kTmDP + c0 + lane_off;
            uint32_t pk[16];
            {
                uint32_t dr[32];
                tmem_ld32(tDP, dr);
                const float4 *d4 = reinterpret_cast<const float4 *>(dlt);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 d = d4[q];
                    pk[2 * q] = pack2<T>(p[4 * q] * (__uint_as_float(dr[4 * q]) - d.x),
                                         p[4 * q + 1] * (__uint_as_float(dr[4 * q + 1]) - d.y));
                    pk[2 * q + 1] = pack2<T>(p[4 * q + 2] * (__uint_as_float(dr[4 * q + 2]) - d.z),
                                             p[4 * q + 3] * (__uint_as_float(dr[4 * q + 3]) - d.w));
                }
            }
            tmem_st16(tDP, pk);
            const uint32_t dst = sDSrow + (t & 1) * kDSTile;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)  // 128B swizzle: 16-byte chunk (half * 4 + cc) of row j
                st_shared_v4(dst + ((uint32_t)((half * 4 + cc) ^ (j & 7)) << 4), pk[4 * cc], pk[4 * cc + 1],
                             pk[4 * cc + 2], pk[4 * cc + 3]);
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar.ds_full);
        }
        // epilogue: dK (scaled), warp w taking rows [32 (w % 4), 32 (w % 4) +
        // 32) and head dims [64 half, 64 half + 64); the drain warps write dV
        // at the same time.  Once every MMA has completed the K tile is idle:
        // each warp stages its 32 x 64 box there (the tile's own 128B-swizzled
        // layout; the box starts at a 1 KB boundary, so row j's swizzle phase
        // is j % 8) and writes it with a TMA store, which drops rows past a
        // dense tensor's end.  A THD tile that ends inside the tensor would
        // spill into the next sequence, so it is written row by row instead.
        // With split query heads the row is this split's fp32 partial,
        // summed by a second kernel.
        if (ok && n_it > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bar.acc_done, 0, wd, 0xe2));
        tc_fence_after();
        const uint32_t base = tmem + kTmDK + half * 64 + lane_off;
        auto load_dk = [&](int cc, uint32_t (&v)[32]) {
            if (n_it > 0) {
                tmem_ld32(base + cc * 32, v);  // warp-wide: every lane loads
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0u;
            }
        };
        if (a.dkv_part) {
            const int64_t krow = (g.thd ? 0 : (int64_t)b * g.Skv) + s.kv0 + key;
            const int64_t nrows = g.thd ? g.Skv : (int64_t)g.B * g.Skv;
            float *dst = a.dkv_part + (((int64_t)(sp * 2) * nrows + krow) * g.Hkv + hk) * D + half * 64;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t v[32];
                load_dk(cc, v);
                if (j < nkeys) store_f32_row32(dst + cc * 32, v);
            }
        } else if (!g.thd || nkeys == BK) {
            uint8_t *boxp = smem + kKOff + half * (BK * 128) + (warp % 4) * 4096;
            const uint32_t srow = smem_u32(boxp) + lane * 128;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t v[32];
                load_dk(cc, v);
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[e] = pack2<T>(__uint_as_float(v[2 * e]) * g.scale, __uint_as_float(v[2 * e + 1]) * g.scale);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c16 = cc * 4 + q;  // 16-byte chunk of the box row
                    st_shared_v4(srow + ((uint32_t)(c16 ^ (lane & 7)) << 4), w[4 * q], w[4 * q + 1], w[4 * q + 2],
                                 w[4 * q + 3]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && (warp % 4) * 32 < nkeys) {
                tma_store_4d(&tm_dk, boxp, half * 64, s.kv0 + n0 + (warp % 4) * 32, hk, cb);
                bulk_commit();
                bulk_wait_read0();  // the copy has read the staging before the CTA exits
            }
            __syncwarp();
        } else {
            T *dstp = (T *)a.dk.ptr + (int64_t)b * a.dk.sb + (int64_t)(s.kv0 + key) * a.dk.ss + (int64_t)hk * a.dk.sh +
                      half * 64;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t v[32];
                load_dk(cc, v);
                if (j < nkeys && half * 64 + cc * 32 < g.D) store_row32<T>(dstp + cc * 32, v, g.scale);
            }
        }
    } else if (warp >= kDrainWarp0) {
        // ----------------------------------- dQ^T drain (thread = head dim)
        griddep_wait();  // the accumulator is cleared by the preprocess
        const int qd = warp % 4;  // TMEM lane quarter = head dims [32 qd, 32 qd + 32)
        const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
        const uint32_t box = smem_u32(smem + kStgOff) + qd * kBox;
        const int zb = g.thd ? 0 : b * g.Hq;
        bool ok = true;
        for (int t = 0; t < n_it; ++t) {
            const int h = h0 + t / nqb;
            const int i0 = ilo + (t % nqb) * BQ;
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.dq_full, t & 1, wd, 0xf0));
            if (!ok) break;
            tc_fence_after();
            uint32_t v[64];
            tmem_ld32(tmem + kTmDQ + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld32(tmem + kTmDQ + 32 + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tc_fence_before();
            mbar_arrive(&bar.dq_free);
            // the previous reduction must have read the box before it is rewritten
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
            // box row r = query i0 + r, 32 fp32 (this warp's head dims) per row,
            // 128B swizzle: 16-byte chunk (lane / 4) of row r at (lane / 4) ^ (r % 8)
#pragma unroll
            for (int r = 0; r < BQ; ++r)
                st_shared_f32(box + r * 128 + ((uint32_t)((lane >> 2) ^ (r & 7)) << 4) + (lane & 3) * 4, v[r]);
            fence_proxy_async_smem();
            __syncwarp();
            // rows past the tensor's end are dropped by the copy; rows past a
            // THD sequence add the 0s of their masked dS to the next sequence
            if (lane == 0) {
                tma_reduce_add_3d(box, &tm_acc, qd * 32, s.q0 + i0, zb + h);
                bulk_commit();
            }
        }
        // dV rows [32 qd, 32 qd + 32), all head dims, once every MMA has
        // completed: staged as two 32 x 64 boxes in the then idle V tile
        // (swizzle phase lane % 8, as for dK) and written with TMA stores; THD
        // tiles ending inside the tensor row by row; with split query heads
        // this split's fp32 partial.
        if (ok && n_it > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bar.acc_done, 0, wd, 0xf2));
        tc_fence_after();
        {
            const int j = qd * 32 + lane;  // key within the tile
            const uint32_t base = tmem + kTmDV + lane_off;
            auto load_dv = [&](int cc, uint32_t (&v)[32]) {
                if (n_it > 0) {
                    tmem_ld32(base + cc * 32, v);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0u;
                }
            };
            if (a.dkv_part) {
                const int64_t krow = (g.thd ? 0 : (int64_t)b * g.Skv) + s.kv0 + n0 + j;
                const int64_t nrows = g.thd ? g.Skv : (int64_t)g.B * g.Skv;
                float *dst = a.dkv_part + (((int64_t)(sp * 2 + 1) * nrows + krow) * g.Hkv + hk) * D;
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t v[32];
                    load_dv(cc, v);
                    if (j < nkeys) store_f32_row32(dst + cc * 32, v);
                }
            } else if (!g.thd || nkeys == BK) {
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t v[32];
                    load_dv(cc, v);
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) w[e] = pack2<T>(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int c16 = cc * 4 + q;  // 16-byte chunk of the row: atom c16 / 8
                        st_shared_v4(smem_u32(smem + kVOff) + (c16 / 8) * (BK * 128) + qd * 4096 + lane * 128 +
                                         ((uint32_t)((c16 % 8) ^ (lane & 7)) << 4),
                                     w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && qd * 32 < nkeys) {
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        tma_store_4d(&tm_dv, smem + kVOff + c * (BK * 128) + qd * 4096, c * 64, s.kv0 + n0 + qd * 32, hk,
                                     cb);
                    bulk_commit();
                }
                __syncwarp();
            } else {
                T *dstp = (T *)a.dv.ptr + (int64_t)b * a.dv.sb + (int64_t)(s.kv0 + n0 + j) * a.dv.ss + (int64_t)hk * a.dv.sh;
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t v[32];
                    load_dv(cc, v);
                    if (j < nkeys && cc * 32 < g.D) store_row32<T>(dstp + cc * 32, v, 1.f);
                }
            }
        }
        // the copies must have read their boxes before the CTA's shared
        // memory goes away (the reductions' additions complete with the grid)
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

// dq = scale * acc in the element type, acc laid out like LSE with DD
// columns per row.  A row is covered by DD / 8 lanes, each reading 8 floats
// (two 16-byte loads) and writing 8 elements (one 16-byte store); every warp
// keeps U rows per lane group in flight.  32-bit index arithmetic (the
// launcher guarantees fewer than 2^31 rows).
template <typename T, int DD, int U>
__global__ void __launch_bounds__(256)
    dq_convert_kernel(MutView dq, const float *__restrict__ acc, Geometry g, FastDiv fRows, FastDiv fHq) {
    griddep_wait();  // the accumulator is complete once the single pass has finished
    constexpr int LPR = DD / 8;
    constexpr int RPW = 32 / LPR;
    const unsigned rows = g.thd ? (unsigned)g.Hq * (unsigned)g.Tq : (unsigned)g.B * (unsigned)g.Hq * (unsigned)g.Sq;
    const int lane = threadIdx.x & 31, sub = lane / LPR, c = lane % LPR;
    const unsigned nwarps = gridDim.x * (blockDim.x / 32);
    for (unsigned base = (blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * (RPW * U); base < rows;
         base += nwarps * (RPW * U)) {
        float4 x0[U], x1[U];
        T *dst[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const unsigned r = base + u * RPW + sub;
            dst[u] = nullptr;
            if (r >= rows || c * 8 >= g.D) continue;  // (columns past the head dim are padding)
            unsigned b = 0, h, srow;
            // fRows divides by the rows of one head (Tq for THD, Sq dense)
            if (g.thd) {
                h = fRows.div(r);
                srow = r - h * (unsigned)g.Tq;
                // token rows outside every sequence (the tail, or the gaps of a
                // padded buffer) are not written
                if (!thd_row_in_sequence(g.cu_q, g.pad_q, g.B, (int)srow)) continue;
            } else {
                const unsigned bh = fRows.div(r);
                srow = r - bh * (unsigned)g.Sq;
                b = fHq.div(bh);
                h = bh - b * (unsigned)g.Hq;
            }
            const float4 *src = reinterpret_cast<const float4 *>(acc + (size_t)r * DD + c * 8);
            x0[u] = __ldg(src);
            x1[u] = __ldg(src + 1);
            dst[u] = (T *)dq.ptr + (int64_t)b * dq.sb + (int64_t)srow * dq.ss + (int64_t)h * dq.sh + c * 8;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (!dst[u]) continue;
            uint4 y;
            y.x = pack2<T>(x0[u].x * g.scale, x0[u].y * g.scale);
            y.y = pack2<T>(x0[u].z * g.scale, x0[u].w * g.scale);
            y.z = pack2<T>(x1[u].x * g.scale, x1[u].y * g.scale);
            y.w = pack2<T>(x1[u].z * g.scale, x1[u].w * g.scale);
            *reinterpret_cast<uint4 *>(dst[u]) = y;
        }
    }
}

// Split query heads: dk = scale * (sum of the splits' partial dK) and
// dv = sum of their partial dV, added in split order (so the result does not
// depend on scheduling) and written in the element type and strides of dk,
// dv.  Partials: [nsplit][2][rows][Hkv][DD] fp32.  A (row, head) is covered
// by DD / 8 lanes of 8 head dims each; 32-bit index arithmetic.
template <typename T, int DD>
__global__ void __launch_bounds__(256)
    dkv_reduce_kernel(MutView dk, MutView dv, const float *__restrict__ part, int nsplit, Geometry g) {
    griddep_wait();  // the partials are complete once the single pass has finished
    constexpr int LPR = DD / 8;
    constexpr int RPW = 32 / LPR;
    const unsigned nrows = g.thd ? (unsigned)g.Skv : (unsigned)g.B * (unsigned)g.Skv;
    const unsigned pairs = nrows * (unsigned)g.Hkv;
    const size_t slice = (size_t)pairs * DD;  // floats of one (split, dK or dV)
    const int lane = threadIdx.x & 31, sub = lane / LPR, c = lane % LPR;
    const unsigned nwarps = gridDim.x * (blockDim.x / 32);
    for (unsigned rh = (blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * RPW + sub; rh < pairs;
         rh += nwarps * RPW) {
        if (c * 8 >= g.D) continue;  // (columns past the head dim are padding)
        const unsigned r = rh / (unsigned)g.Hkv, hk = rh - r * (unsigned)g.Hkv;
        unsigned b = 0, key = r;
        if (g.thd) {
            if (!thd_row_in_sequence(g.cu_kv, g.pad_kv, g.B, (int)key)) continue;
        } else {
            b = r / (unsigned)g.Skv;
            key = r - b * (unsigned)g.Skv;
        }
        float sk[8], sv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) sk[e] = sv[e] = 0.f;
        const float *src = part + (size_t)rh * DD + c * 8;
        for (int sp = 0; sp < nsplit; ++sp) {
            const float4 *pk = reinterpret_cast<const float4 *>(src + (size_t)(2 * sp) * slice);
            const float4 *pv = reinterpret_cast<const float4 *>(src + (size_t)(2 * sp + 1) * slice);
            const float4 k0 = __ldg(pk), k1 = __ldg(pk + 1), v0 = __ldg(pv), v1 = __ldg(pv + 1);
            sk[0] += k0.x; sk[1] += k0.y; sk[2] += k0.z; sk[3] += k0.w;
            sk[4] += k1.x; sk[5] += k1.y; sk[6] += k1.z; sk[7] += k1.w;
            sv[0] += v0.x; sv[1] += v0.y; sv[2] += v0.z; sv[3] += v0.w;
            sv[4] += v1.x; sv[5] += v1.y; sv[6] += v1.z; sv[7] += v1.w;
        }
        uint4 yk, yv;
        yk.x = pack2<T>(sk[0] * g.scale, sk[1] * g.scale);
        yk.y = pack2<T>(sk[2] * g.scale, sk[3] * g.scale);
        yk.z = pack2<T>(sk[4] * g.scale, sk[5] * g.scale);
        yk.w = pack2<T>(sk[6] * g.scale, sk[7] * g.scale);
        yv.x = pack2<T>(sv[0], sv[1]);
        yv.y = pack2<T>(sv[2], sv[3]);
        yv.z = pack2<T>(sv[4], sv[5]);
        yv.w = pack2<T>(sv[6], sv[7]);
        const int64_t ok = (int64_t)b * dk.sb + (int64_t)key * dk.ss + (int64_t)hk * dk.sh + c * 8;
        const int64_t ov = (int64_t)b * dv.sb + (int64_t)key * dv.ss + (int64_t)hk * dv.sh + c * 8;
        *reinterpret_cast<uint4 *>((T *)dk.ptr + ok) = yk;
        *reinterpret_cast<uint4 *>((T *)dv.ptr + ov) = yv;
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
    if (max_lkv > 0) {  // (no key at all: dk, dv are empty and dq = 0)
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
        if ((e = make_tmap_f32_acc(&tacc, a.dq_acc, D, acc_rows, acc_heads, 32, BQ)) != cudaSuccess) return e;
        // dK / dV leave in 32-row boxes, one per TMEM lane quarter
        if ((e = make_tmap_16bit(&tgk, a.dk.ptr, dt, dk, sgk, 32)) != cudaSuccess) return e;
        if ((e = make_tmap_16bit(&tgv, a.dv.ptr, dt, dk, sgv, 32)) != cudaSuccess) return e;
        auto kern = tc_bwd_fused_kernel<T>;
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

template <typename T, int DD>
cudaError_t dkv_reduce_typed(const BwdArgs &a, cudaStream_t st) {
    const Geometry &g = a.g;
    const int64_t pairs = (g.thd ? (int64_t)g.Skv : (int64_t)g.B * g.Skv) * g.Hkv;
    if (pairs <= 0) return cudaSuccess;
    if (pairs >= ((int64_t)1 << 31)) return cudaErrorInvalidConfiguration;
    int sms = 0;
    cudaError_t e = device_sm_count(&sms);
    if (e != cudaSuccess) return e;
    const int64_t warps = (pairs + (256 / DD) - 1) / (256 / DD);
    int64_t blocks = (warps + 7) / 8;
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    prof_before(st, kProfBwdDkvReduce);
    cudaError_t le = launch_pdl(dkv_reduce_kernel<T, DD>, dim3((unsigned)blocks), dim3(256), 0, st, a.dk, a.dv,
                                a.dkv_part, a.nsplit, g);
    prof_after(st);
    return le != cudaSuccess ? le : cudaGetLastError();
}

template <typename T, int DD>
cudaError_t dq_convert_typed(const BwdArgs &a, cudaStream_t st) {
    constexpr int U = 4;
    const Geometry &g = a.g;
    const int64_t rows = g.thd ? (int64_t)g.Hq * g.Tq : (int64_t)g.B * g.Hq * g.Sq;
    if (rows <= 0) return cudaSuccess;
    if (rows >= ((int64_t)1 << 31)) return cudaErrorInvalidConfiguration;
    int sms = 0;
    cudaError_t e = device_sm_count(&sms);
    if (e != cudaSuccess) return e;
    const int64_t per_warp = (32 / (DD / 8)) * U;
    const int64_t warps = (rows + per_warp - 1) / per_warp;
    int64_t blocks = (warps + 7) / 8;
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    prof_before(st, kProfBwdDqConvert);
    const int per_head = g.thd ? g.Tq : g.Sq;
    cudaError_t le = launch_pdl(dq_convert_kernel<T, DD, U>, dim3((unsigned)blocks), dim3(256), 0, st, a.dq, a.dq_acc, g,
                                FastDiv(per_head > 0 ? per_head : 1), FastDiv(g.Hq));
    prof_after(st);
    return le != cudaSuccess ? le : cudaGetLastError();
}

}  // namespace

cudaError_t launch_dq_convert(int dtype, const BwdArgs &a, cudaStream_t st) {
    switch (dtype * 2 + (tc_dim(a.g.D) == 128)) {
        case 0: return dq_convert_typed<__half, 64>(a, st);
        case 1: return dq_convert_typed<__half, 128>(a, st);
        case 2: return dq_convert_typed<__nv_bfloat16, 64>(a, st);
        case 3: return dq_convert_typed<__nv_bfloat16, 128>(a, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_dkv_reduce(int dtype, const BwdArgs &a, cudaStream_t st) {
    switch (dtype * 2 + (tc_dim(a.g.D) == 128)) {
        case 0: return dkv_reduce_typed<__half, 64>(a, st);
        case 1: return dkv_reduce_typed<__half, 128>(a, st);
        case 2: return dkv_reduce_typed<__nv_bfloat16, 64>(a, st);
        case 3: return dkv_reduce_typed<__nv_bfloat16, 128>(a, st);
    }
    return cudaErrorInvalidValue;
}

bool uses_tc_bwd_fused(int dtype, int D_) {
    return (dtype == 0 || dtype == 1) && (D_ == 32 || D_ == 64 || D_ == 96 || D_ == 128);
}

cudaError_t launch_tc_bwd_fused(int dtype, const BwdArgs &a, int max_lkv, int q_rows, cudaStream_t st) {
    // callers route problems without query rows to the two-kernel backward
    if (!a.dq_acc || (a.g.thd ? a.g.Tq : a.g.Sq) <= 0) return cudaErrorInvalidValue;
    if (tc_dim(a.g.D) == 64) return launch_tc_bwd_fused64(dtype, a, max_lkv, q_rows, st);
    if (tc_dim(a.g.D) != D) return cudaErrorInvalidValue;
    switch (dtype) {
        case 0: return launch_typed<__half>(a, max_lkv, q_rows, st);
        case 1: return launch_typed<__nv_bfloat16>(a, max_lkv, q_rows, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gbattn
