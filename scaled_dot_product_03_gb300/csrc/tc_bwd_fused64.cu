// tc_bwd_fused64.cu -- single-pass tcgen05 backward attention, head dim 64.
//
// The same method as the head-dim-128 single pass (S and dP formed once per
// (query, key) pair, dV and dK owned by the CTA, each block's share of dQ
// added into an fp32 accumulator), laid out for D = 64, where TMEM has room
// for 128-query blocks and an untransposed dQ:
//   S^T  = K Q^T,  dP^T = V dO^T          (M = 128 keys, N = 128 queries;
//                                         K and V from shared memory)
//   P^T  = exp(scale S^T - LSE),  dS^T = P^T o (dP^T - delta)
//   dV  += P^T dO,  dK += dS^T Q          (P^T, dS^T from TMEM)
//   dQ   = dS K                           (M = 128 queries; dS from shared
//                                         memory as an MN-major A operand)
// so every product runs with M = 128 and the dQ drain holds query rows
// (thread = query row), which it writes as row-major boxes.  dS^T is the
// 16-bit product of the 16-bit P^T that dV reads with dP^T - delta (formed
// in fp32 and rounded): P stays packed between the two steps.
//
// Work item: the 128 keys of key tile kt of a (batch, key/value head, split
// of its query heads).  The grid is persistent: one CTA per SM starts with
// the item of its block index and then takes items, heaviest first, from a
// counter in the workspace until none are left.  Per CTA the items follow
// one another without a gap: the next item's K is loaded (K has two buffers)
// and its first S^T product issued while the current item finishes, its V
// as soon as the current item's last dP^T product is done with the single V
// buffer, and the current item's dK / dV leave TMEM while the next item's
// first products run.
//
// Warps 0-7 compute P and dS (thread = key row; warps 0-3 take query columns
// 0-63 of the block, warps 4-7 columns 64-127) and write dK (warps 0-3) and
// dV (warps 4-7); warp 8 takes items and loads; warp 9 issues the MMAs (the
// whole warp runs the loop, an elected lane issues); warps 10-13 drain dQ
// (warp w: query rows [32 (w % 4), 32 (w % 4) + 32)).
//
// TMEM columns (448 of 512): dK 0-63, dV 64-127, S^T / P^T 128-255, dP^T /
// dS^T 256-383, dQ 384-447.  MMA order per block t: dV_t, S^T_{t+1}, dK_t,
// dQ_t, dP^T_{t+1} (block t + 1 may be the next item's first); dP^T_{t+1}
// overwrites dS^T_t after dK_t read it and is issued after dQ_t read dS_t
// from shared memory, so one dS^T buffer suffices (its next writer waits for
// dP^T_{t+1}).  Shared memory: two K buffers, V, three stages of Q and dO
// (16 KB each), dS^T (32 KB, also the staging of the dK / dV stores), eight
// 4 KB dQ staging boxes and the per-stage LSE / delta.
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
constexpr int BK = 128;   // keys per item
constexpr int BQ = 128;   // query rows per block
constexpr int QS = 3;     // Q / dO stages
constexpr int kThreads = 448;
constexpr int kCompute = 256;
constexpr int kProdWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kDrainWarp0 = 10;
constexpr int kDrain = 128;
constexpr int kHeadBand = 4;
// warps reading the item ring: the MMA warp, the 8 compute and 4 drain warps
constexpr int kItemReaders = 13;

constexpr int kKVTile = BK * D * 2;   // 16 KB
constexpr int kQTile = BQ * D * 2;    // 16 KB
constexpr int kDSTile = BK * BQ * 2;  // 32 KB: two 64-query atoms
constexpr int kBox = 32 * 32 * 4;     // 4 KB: 32 query rows x 32 fp32
constexpr int kKOff = 0;                        // two K buffers (items alternate)
constexpr int kVOff = kKOff + 2 * kKVTile;
constexpr int kQOff = kVOff + kKVTile;
constexpr int kDOOff = kQOff + QS * kQTile;
constexpr int kDSOff = kDOOff + QS * kQTile;
constexpr int kStgOff = kDSOff + kDSTile;
constexpr int kStatOff = kStgOff + 8 * kBox;          // [QS][128] lse2, [QS][128] delta
constexpr int kBarOff = kStatOff + QS * BQ * 2 * 4;
constexpr int kSmemBytes = kBarOff + 256 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kTmDK = 0, kTmDV = 64, kTmS = 128, kTmDP = 256, kTmDQ = 384;

struct Bars {
    uint64_t k_full[2], k_empty[2], v_full, v_empty;
    uint64_t q_full[QS], q_empty[QS];
    uint64_t item_full[2], item_empty[2];
    uint64_t s_full, p_full, dp_full, ds_full;
    uint64_t dq_full, dq_free, acc_done, acc_empty;
    int item[2];
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
                          const __grid_constant__ CUtensorMap tm_dv, BwdArgs a, int n_ktiles, int n_items) {
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Bars &bar = *reinterpret_cast<Bars *>(smem + kBarOff);
    // Launched as a dependent of the preprocess: everything up to the first
    // read of its output (delta, the cleared dQ accumulator, the work
    // counter) overlaps its tail; the dQ conversion may begin launching at once.
    griddep_launch();
    float *s_lse = reinterpret_cast<float *>(smem + kStatOff);  // log2 units
    float *s_delta = s_lse + QS * BQ;
    const Geometry &g = a.g;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    auto item_of = [&](int w) { return bwd_item(w, g, a.nsplit, n_ktiles, BK, BQ, kHeadBand); };
    // K of the kn-th item with blocks into buffer kn % 2 (lane 0 of the
    // loading warp; the buffer is free)
    auto load_k = [&](const BwdItem &it, int kn) {
        const int kb = kn & 1;
        mbar_arrive_expect_tx(&bar.k_full[kb], kKVTile);
        tma_load_4d(smem + kKOff + kb * kKVTile, &tm_k, &bar.k_full[kb], 0, it.s.kv0 + it.n0, it.hk,
                    g.thd ? 0 : it.b);
    };
    auto load_v = [&](const BwdItem &it) {
        mbar_arrive_expect_tx(&bar.v_full, kKVTile);
        tma_load_4d(smem + kVOff, &tm_v, &bar.v_full, 0, it.s.kv0 + it.n0, it.hk, g.thd ? 0 : it.b);
    };

    if (warp == kProdWarp && lane == 0) {
        // The loading lane sets up the barriers, posts this CTA's first item
        // (its block index) and issues that item's K and V loads at once, so
        // that they overlap the TMEM allocation and the block-wide sync.
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar.k_full[i], 1);
            mbar_init(&bar.k_empty[i], 1);
            mbar_init(&bar.item_full[i], 1);
            mbar_init(&bar.item_empty[i], kItemReaders);
        }
        mbar_init(&bar.v_full, 1);
        mbar_init(&bar.v_empty, 1);
        for (int i = 0; i < QS; ++i) {
            mbar_init(&bar.q_full[i], 32);
            mbar_init(&bar.q_empty[i], 1);
        }
        mbar_init(&bar.s_full, 1);
        mbar_init(&bar.p_full, kCompute);
        mbar_init(&bar.dp_full, 1);
        mbar_init(&bar.ds_full, kCompute);
        mbar_init(&bar.dq_full, 1);
        mbar_init(&bar.dq_free, kDrain);
        mbar_init(&bar.acc_done, 1);
        mbar_init(&bar.acc_empty, kCompute);
        bar.abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
        prefetch_tmap(&tm_acc);
        bar.item[0] = (int)blockIdx.x;
        mbar_arrive(&bar.item_full[0]);
        const BwdItem it = item_of((int)blockIdx.x);
        if (it.n_it > 0) {
            load_k(it, 0);
            load_v(it);
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

    // Ring item n of this CTA (slot n % 2).  Every warp but the loader reads
    // every item in order; its lane 0 frees the slot once the warp has it.
    auto read_item = [&](int n, int &w, unsigned code) {
        const int slot = n & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&bar.item_full[slot], (n >> 1) & 1, wd, code))) return false;
        w = *reinterpret_cast<volatile int *>(&bar.item[slot]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.item_empty[slot]);
        return true;
    };

    if (warp == kProdWarp) {
        // ------------------------------------------------------------ loads
        // Per item: K once the item is posted (its buffer was freed by the
        // item before last), the blocks' LSE, delta, Q and dO as stages free
        // up, and V after the first block, once the previous item's last
        // dP^T product is done with the V buffer.  The next item is taken
        // after the last block's loads and posted in the ring.
        griddep_wait();  // delta and the work counter come from the preprocess
        bool ok = true;
        int gt = 0, kn = 0, w = (int)blockIdx.x;  // blocks and items with blocks so far
        for (int n = 0; ok; ++n) {
            const BwdItem it = item_of(w);
            if (lane == 0 && it.kt == n_ktiles - 1 && it.sp == 0)
                report_uncovered(a.err, g, it.s.Lkv, n_ktiles * BK, kErrSeqlenKv);
            const int cb = g.thd ? 0 : it.b;
            const bool pre = n == 0;  // the first item's K and V were issued before the sync
            if (it.n_it > 0 && !pre) {
                if (!(ok = __all_sync(0xffffffffu,
                                      mbar_wait(&bar.k_empty[kn & 1], ((kn >> 1) & 1) ^ 1, wd, 0xc9))))
                    break;
                if (lane == 0) {
                    load_k(it, kn);
                    tma_prefetch_l2_4d(&tm_v, 0, it.s.kv0 + it.n0, it.hk, cb);
                }
            }
            for (int t = 0; t <= it.n_it; ++t) {
                if (t == 1 && !pre) {
                    if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.v_empty, (kn & 1) ^ 1, wd, 0xca)))) break;
                    if (lane == 0) load_v(it);
                }
                if (t == it.n_it) break;
                const int gb = gt + t;
                const int st = gb % QS;
                const uint32_t ph = (gb / QS) & 1;
                const int h = it.h0 + t / it.nqb;
                const int i0 = it.ilo + (t % it.nqb) * BQ;
                // LSE (log2 units) and delta of the block's rows, fetched
                // while the stage is still in use
                float lv[4], dv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + lane + 32 * u;
                    lv[u] = dv[u] = 0.f;
                    if (i < it.s.Lq) {
                        const int64_t li = lse_index(g, it.s, it.b, h, i);
                        lv[u] = a.lse[li] * kLog2e;
                        dv[u] = a.delta[li];
                    }
                }
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.q_empty[st], ph ^ 1, wd, 0xc8)))) break;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    s_lse[st * BQ + lane + 32 * u] = lv[u];
                    s_delta[st * BQ + lane + 32 * u] = dv[u];
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bar.q_full[st], 2 * kQTile);
                    tma_load_4d(smem + kQOff + st * kQTile, &tm_q, &bar.q_full[st], 0, it.s.q0 + i0, h, cb);
                    tma_load_4d(smem + kDOOff + st * kQTile, &tm_do, &bar.q_full[st], 0, it.s.q0 + i0, h, cb);
                } else {
                    mbar_arrive(&bar.q_full[st]);
                }
            }
            if (!ok) break;
            // the next item, posted in ring slot (n + 1) % 2 once every reader
            // has taken item n - 1 from it (an index past the last item ends
            // every role's loop)
            int wn = 0;
            if (lane == 0) wn = (int)gridDim.x + (int)atomicAdd(a.work_ctr, 1u);
            wn = __shfl_sync(0xffffffffu, wn, 0);
            const int slot = (n + 1) & 1;
            if (!(ok = __all_sync(0xffffffffu,
                                  mbar_wait(&bar.item_empty[slot], (((n + 1) >> 1) & 1) ^ 1, wd, 0xc1))))
                break;
            if (lane == 0) {
                bar.item[slot] = wn;
                mbar_arrive(&bar.item_full[slot]);
            }
            __syncwarp();
            gt += it.n_it;
            if (it.n_it > 0) ++kn;
            if (wn >= n_items) break;
            w = wn;
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA
        // At an item's last block the next ring item is read ahead: if it has
        // blocks, its first S^T takes the place of S^T_{t+1} and its first
        // dP^T follows the item's last dQ.  (Only one item is read ahead: the
        // other roles free a ring slot only when they reach its item.)
        constexpr uint32_t idSP = idesc_f16(BK, BQ, kBf16, 0, 0);  // S^T, dP^T
        constexpr uint32_t idKV = idesc_f16(BK, D, kBf16, 0, 1);   // dV, dK: B = dO / Q, MN-major
        constexpr uint32_t idQ = idesc_f16(BQ, D, kBf16, 1, 1);    // dQ: A = dS, B = K, MN-major
        const uint32_t sQ = smem_u32(smem + kQOff), sDO = smem_u32(smem + kDOOff), sK = smem_u32(smem + kKOff);
        const uint64_t dVa = smem_desc_sw128(smem_u32(smem + kVOff), 16, 1024);          // A of dP^T
        const uint64_t dSm = smem_desc_sw128(smem_u32(smem + kDSOff), BK * 128, 1024);  // A of dQ
        auto wait = [&](uint64_t *bb, uint32_t ph, unsigned code) {
            const bool r = __all_sync(0xffffffffu, mbar_wait(bb, ph, wd, code));
            if (r) tc_fence_after();
            return r;
        };
        auto issue_s = [&](int gb, int kb) {
            const uint64_t da = smem_desc_sw128(sK + kb * kKVTile, 16, 1024);
            const uint64_t db = smem_desc_sw128(sQ + (gb % QS) * kQTile, 16, 1024);
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + kTmS, desc_add(da, kmaj_off(kk, BK)), desc_add(db, kmaj_off(kk, BQ)), idSP, kk > 0);
                mma_commit(&bar.s_full);
            }
            __syncwarp();
        };
        // dP^T of block gb; after the item's last one the V buffer is free
        auto issue_dp = [&](int gb, bool last) {
            const uint64_t db = smem_desc_sw128(sDO + (gb % QS) * kQTile, 16, 1024);
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + kTmDP, desc_add(dVa, kmaj_off(kk, BK)), desc_add(db, kmaj_off(kk, BQ)), idSP,
                           kk > 0);
                mma_commit(&bar.dp_full);
                if (last) mma_commit(&bar.v_empty);
            }
            __syncwarp();
        };
        bool ok = true, done = false, ahead = false;
        int n = 0, gt = 0, kn = 0;  // ring items read, blocks and items with blocks so far
        int cur = 0, nxt = 0;       // blocks of the current item, of the one read ahead
        while (ok && !done) {
            if (ahead) {
                cur = nxt;  // its first S^T and dP^T are issued
                ahead = false;
            } else {
                // the next item with blocks; its first S^T and dP^T
                for (;;) {
                    int w = 0;
                    if (!(ok = read_item(n++, w, 0xd7))) break;
                    if (w >= n_items) {
                        done = true;
                        break;
                    }
                    cur = item_of(w).n_it;
                    if (cur > 0) break;
                }
                if (!ok || done) break;
                if (!(ok = wait(&bar.k_full[kn & 1], (kn >> 1) & 1, 0xd8) &&
                           wait(&bar.q_full[gt % QS], (gt / QS) & 1, 0xd9)))
                    break;
                issue_s(gt, kn & 1);
                if (!(ok = wait(&bar.v_full, kn & 1, 0xd0))) break;
                issue_dp(gt, cur == 1);
            }
            const int kb = kn & 1;
            const uint64_t dKm = smem_desc_sw128(sK + kb * kKVTile, BK * 128, 1024);  // B of dQ
            for (int t = 0; t < cur; ++t) {
                const int gb = gt + t;
                const int st = gb % QS;
                const bool last = t + 1 == cur;
                // Q_t / dO_t as MN-major B operands (N = head dim, one 64-wide atom)
                const uint64_t dOm = smem_desc_sw128(sDO + st * kQTile, BQ * 128, 1024);
                const uint64_t dQm = smem_desc_sw128(sQ + st * kQTile, BQ * 128, 1024);
                const uint32_t acc0 = t > 0 ? 1u : 0u;
                if (!(ok = wait(&bar.p_full, gb & 1, 0xda))) break;
                // the previous item's dK and dV have left TMEM
                if (t == 0 && kn > 0 && !(ok = wait(&bar.acc_empty, (kn - 1) & 1, 0xde))) break;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BQ / 16; ++kk)
                        mma_ts(tmem + kTmDV, tmem + kTmS + pcol(kk), desc_add(dOm, kk * 16 * 128), idKV,
                               kk > 0 ? 1u : acc0);
                }
                __syncwarp();
                if (!last) {
                    if (!(ok = wait(&bar.q_full[(gb + 1) % QS], ((gb + 1) / QS) & 1, 0xdb))) break;
                    issue_s(gb + 1, kb);
                } else {
                    int w = 0;
                    if (!(ok = read_item(n++, w, 0xd7))) break;
                    if (w >= n_items) {
                        done = true;
                    } else {
                        nxt = item_of(w).n_it;
                        if (nxt > 0) {
                            if (!(ok = wait(&bar.k_full[kb ^ 1], ((kn + 1) >> 1) & 1, 0xdf) &&
                                       wait(&bar.q_full[(gb + 1) % QS], ((gb + 1) / QS) & 1, 0xdb)))
                                break;
                            issue_s(gb + 1, kb ^ 1);
                            ahead = true;
                        }
                    }
                }
                if (!(ok = wait(&bar.ds_full, gb & 1, 0xdc))) break;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BQ / 16; ++kk)
                        mma_ts(tmem + kTmDK, tmem + kTmDP + pcol(kk), desc_add(dQm, kk * 16 * 128), idKV,
                               kk > 0 ? 1u : acc0);
                    mma_commit(&bar.q_empty[st]);
                }
                __syncwarp();
                if (gb > 0 && !(ok = wait(&bar.dq_free, (gb - 1) & 1, 0xdd))) break;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)  // K = keys: 16 key rows per step
                        mma_ss(tmem + kTmDQ, desc_add(dSm, kk * 16 * 128), desc_add(dKm, kk * 16 * 128), idQ, kk > 0);
                    mma_commit(&bar.dq_full);
                }
                __syncwarp();
                if (!last) issue_dp(gb + 1, t + 2 == cur);
            }
            if (!ok) break;
            // the item's products are done with TMEM's dK / dV and with its K buffer
            if (elect_one()) {
                mma_commit(&bar.acc_done);
                mma_commit(&bar.k_empty[kb]);
            }
            __syncwarp();
            gt += cur;
            ++kn;
            if (ahead) {
                if (!(ok = wait(&bar.v_full, kn & 1, 0xd0))) break;
                issue_dp(gt, nxt == 1);
            }
        }
    } else if (warp < kProdWarp) {
        // --------------------------------------- P, dS (thread = key row)
        const int half = warp / 4;  // query columns [64 half, 64 half + 64)
        const int c0 = half * 64;
        const int j = (warp % 4) * 32 + lane;
        const uint32_t lane_off = (uint32_t)((warp % 4) * 32) << 16;
        const uint32_t tS = tmem + kTmS + c0 + lane_off;
        const uint32_t tP = tmem + kTmDP + c0 + lane_off;
        // dS^T row j, query atom `half` (64 queries = 128 B per row); the
        // warp's 32 rows (4 KB) also stage its share of dK / dV
        uint8_t *const box = smem + kDSOff + half * (BK * 128) + (warp % 4) * 4096;
        const uint32_t sDSrow = smem_u32(box) + lane * 128;
        const float c2 = g.scale_log2;
        bool ok = true;
        int gt = 0, kn = 0;  // blocks and items with blocks so far
        for (int n = 0; ok; ++n) {
            int w = 0;
            if (!(ok = read_item(n, w, 0xe4))) break;
            if (w >= n_items) break;
            const BwdItem bi = item_of(w);
            if (bi.nkeys <= 0) continue;  // past the sequence: no rows
            const int n_it = bi.n_it;
            for (int t = 0; t < n_it; ++t) {
                const int n0 = bi.n0;
                const int key = n0 + j;
                const SeqInfo &s = bi.s;
                const int gb = gt + t;
                const int st = gb % QS;
                const int i0 = bi.ilo + (t % bi.nqb) * BQ + c0;
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.s_full, gb & 1, wd, 0xe8)))) break;
                tc_fence_after();
                const float *lse2 = s_lse + st * BQ + c0;
                const float *dlt = s_delta + st * BQ + c0;
                const bool full = (i0 + 63 < s.Lq) && (n0 + BK - 1 < s.Lkv) &&
                                  (g.wr < 0 || n0 + BK - 1 <= i0 + g.wr) && (g.wl < 0 || n0 >= i0 + 63 - g.wl);
                // P kept packed (the 16-bit values the dV product reads): dS
                // below is the packed product of the same P with dP - delta
                // (formed in fp32, then rounded), and 32 registers fewer are
                // live across the wait for dP^T
                uint32_t pp[32];
                {
                    // query columns [clo, chi) of this half see the key
                    int clo = 0, chi = 64;
                    if (!full) {
                        chi = min(64, s.Lq - i0);
                        if (g.wr >= 0) clo = max(clo, key - g.wr - i0);
                        if (g.wl >= 0) chi = min(chi, key + g.wl + 1 - i0);
                        if (key >= s.Lkv) chi = clo;
                    }
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        // 32 columns at a time: exp2, mask, pack
                        uint32_t sr[32];
                        tmem_ld32(tS + 32 * h2, sr);
                        // 16-byte broadcast reads of the LSE (shared memory
                        // bandwidth is shared with the MMA operand reads)
                        const float4 *l4 = reinterpret_cast<const float4 *>(lse2 + 32 * h2);
                        float p[32];
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 l = l4[q];
                            p[4 * q] = ex2(fmaf(__uint_as_float(sr[4 * q]), c2, -l.x));
                            p[4 * q + 1] = ex2(fmaf(__uint_as_float(sr[4 * q + 1]), c2, -l.y));
                            p[4 * q + 2] = ex2(fmaf(__uint_as_float(sr[4 * q + 2]), c2, -l.z));
                            p[4 * q + 3] = ex2(fmaf(__uint_as_float(sr[4 * q + 3]), c2, -l.w));
                        }
                        if (!full) {
#pragma unroll
                            for (int c = 0; c < 32; ++c)
                                if (32 * h2 + c < clo || 32 * h2 + c >= chi) p[c] = 0.f;
                        }
#pragma unroll
                        for (int c = 0; c < 16; ++c) pp[16 * h2 + c] = pack2<T>(p[2 * c], p[2 * c + 1]);
                    }
                }
                tmem_st32(tS, pp);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bar.p_full);
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.dp_full, gb & 1, wd, 0xe9)))) break;
                tc_fence_after();
                // dS^T_t: packed over dP^T_t in TMEM (A of dK) and into shared
                // memory (A of dQ); the shared copy was last read by dQ_{t-1},
                // issued before dP^T_t, whose completion we saw, and, at an
                // item's first block, by the store of the previous item's
                // dK / dV, which the issuing lane waits for
                uint32_t pk[32];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    uint32_t dr[32];
                    tmem_ld32(tP + 32 * h2, dr);
                    const float4 *d4 = reinterpret_cast<const float4 *>(dlt + 32 * h2);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 d = d4[q];
                        pk[16 * h2 + 2 * q] =
                            mul2<T>(pp[16 * h2 + 2 * q], pack2<T>(__uint_as_float(dr[4 * q]) - d.x,
                                                                  __uint_as_float(dr[4 * q + 1]) - d.y));
                        pk[16 * h2 + 2 * q + 1] =
                            mul2<T>(pp[16 * h2 + 2 * q + 1], pack2<T>(__uint_as_float(dr[4 * q + 2]) - d.z,
                                                                      __uint_as_float(dr[4 * q + 3]) - d.w));
                    }
                }
                tmem_st32(tP, pk);
                if (t == 0) {
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
                }
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)  // 128B swizzle: 16-byte chunk cc of row j
                    st_shared_v4(sDSrow + ((uint32_t)(cc ^ (j & 7)) << 4), pk[4 * cc], pk[4 * cc + 1],
                                 pk[4 * cc + 2], pk[4 * cc + 3]);
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bar.ds_full);
            }
            if (!ok) break;
            // (the item decoded again: fewer values live across the loop)
            asm volatile("" : "+r"(w));
            const BwdItem it = item_of(w);
            const int n0 = it.n0;
            const int key = n0 + j;
            const SeqInfo &s = it.s;
            // dK (scaled; warps 0-3) or dV (warps 4-7) of the warp's 32 key
            // rows: read out of TMEM once the item's products are done (the
            // MMA warp starts the next item's dV / dK once every warp has
            // them); a tile that no query sees has zeros
            uint32_t v[64];
            if (it.n_it > 0) {
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.acc_done, kn & 1, wd, 0xea)))) break;
                tc_fence_after();
                const uint32_t base = tmem + (half == 0 ? kTmDK : kTmDV) + lane_off;
                tmem_ld32(base, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                tmem_ld32(base + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                tc_fence_before();
                mbar_arrive(&bar.acc_empty);
            } else {
#pragma unroll
                for (int e = 0; e < 64; ++e) v[e] = 0u;
            }
            const float mul = half == 0 ? g.scale : 1.f;
            if (a.dkv_part) {
                // split query heads: this split's fp32 partial row, summed by
                // a second kernel
                if (j < it.nkeys) {
                    const int64_t krow = (g.thd ? 0 : (int64_t)it.b * g.Skv) + s.kv0 + key;
                    const int64_t nrows = g.thd ? g.Skv : (int64_t)g.B * g.Skv;
                    float *dst = a.dkv_part + (((int64_t)(it.sp * 2 + half) * nrows + krow) * g.Hkv + it.hk) * D;
                    store_f32_row32(dst, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                    store_f32_row32(dst + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                }
            } else if (!g.thd || it.nkeys == BK) {
                // one 32-row box in the warp's share of the dS^T buffer
                // (128B-swizzled like the loads; the box sits at a 1 KB
                // boundary, so row lane's swizzle phase is lane % 8), written
                // with a TMA store, which drops rows past a dense tensor's
                // end.  (A THD tile that ends inside the tensor would spill
                // into the next sequence: it is written row by row below.)
                if (lane == 0) bulk_wait_read0();
                __syncwarp();
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    uint32_t wv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        wv[e] = pack2<T>(__uint_as_float(v[8 * q + 2 * e]) * mul,
                                         __uint_as_float(v[8 * q + 2 * e + 1]) * mul);
                    st_shared_v4(sDSrow + ((uint32_t)(q ^ (lane & 7)) << 4), wv[0], wv[1], wv[2], wv[3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && (warp % 4) * 32 < it.nkeys) {
                    tma_store_4d(half == 0 ? &tm_dk : &tm_dv, box, 0, s.kv0 + n0 + (warp % 4) * 32, it.hk,
                                 g.thd ? 0 : it.b);
                    bulk_commit();
                }
            } else if (j < it.nkeys) {
                const MutView &ov = half == 0 ? a.dk : a.dv;
                T *dstp = (T *)ov.ptr + (int64_t)it.b * ov.sb + (int64_t)(s.kv0 + key) * ov.ss + (int64_t)it.hk * ov.sh;
                store_row32<T>(dstp, *reinterpret_cast<uint32_t(*)[32]>(&v[0]), mul);
                if (g.D > 32) store_row32<T>(dstp + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]), mul);
            }
            gt += it.n_it;
            if (it.n_it > 0) ++kn;
        }
        // the stores have read their boxes before the CTA's shared memory
        // goes away
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
    } else if (warp >= kDrainWarp0) {
        // ------------------------------------- dQ drain (thread = query row)
        griddep_wait();  // the accumulator is cleared by the preprocess
        const int qd = warp % 4;  // TMEM lane quarter = query rows [32 qd, 32 qd + 32)
        const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
        const uint32_t box0 = smem_u32(smem + kStgOff) + qd * 2 * kBox;  // head dims 0-31, then 32-63
        bool ok = true;
        int gt = 0;
        for (int n = 0; ok; ++n) {
            int w = 0;
            if (!(ok = read_item(n, w, 0xf1))) break;
            if (w >= n_items) break;
            const BwdItem it = item_of(w);
            const int zb = g.thd ? 0 : it.b * g.Hq;
            for (int t = 0; t < it.n_it; ++t) {
                const int gb = gt + t;
                const int h = it.h0 + t / it.nqb;
                const int i0 = it.ilo + (t % it.nqb) * BQ;
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.dq_full, gb & 1, wd, 0xf8)))) break;
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
                    tma_reduce_add_3d(box0, &tm_acc, 0, it.s.q0 + i0 + 32 * qd, zb + h);
                    tma_reduce_add_3d(box0 + kBox, &tm_acc, 32, it.s.q0 + i0 + 32 * qd, zb + h);
                    bulk_commit();
                }
            }
            gt += it.n_it;
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
        // dK / dV: one 32-row box per compute warp
        if ((e = make_tmap_16bit(&tgk, a.dk.ptr, dt, dk, sgk, 32)) != cudaSuccess) return e;
        if ((e = make_tmap_16bit(&tgv, a.dv.ptr, dt, dk, sgv, 32)) != cudaSuccess) return e;
        auto kern = tc_bwd_fused64_kernel<T>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)) !=
            cudaSuccess)
            return e;
        int sms = 0;
        if ((e = device_sm_count(&sms)) != cudaSuccess) return e;
        const int n_ktiles = (max_lkv + BK - 1) / BK;
        const int64_t n_items = (int64_t)n_ktiles * g.Hkv * g.B * a.nsplit;
        // (item indices stay below 2^31 with the grid's extra fetches)
        if (n_items > 0x7fffffff - 65536) return cudaErrorInvalidConfiguration;
        if ((e = launch_bwd_preprocess(dt, a, q_rows, st)) != cudaSuccess) return e;
        // persistent: one CTA per SM, taking items from the counter
        const int grid = (int)(n_items < sms ? n_items : sms);
        prof_before(st, kProfBwdFused);
        e = launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), kSmemBytes, st, tq, tk, tv, tdo, tacc, tgk, tgv, a,
                       n_ktiles, (int)n_items);
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
    if (tc_dim(a.g.D) != D || !a.dq_acc || !a.work_ctr) return cudaErrorInvalidValue;
    switch (dtype) {
        case 0: return launch_typed<__half>(a, max_lkv, q_rows, st);
        case 1: return launch_typed<__nv_bfloat16>(a, max_lkv, q_rows, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gbattn
