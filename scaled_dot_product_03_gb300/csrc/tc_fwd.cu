// tc_fwd.cu -- tcgen05 forward attention for fp16 / bf16 (head dims 32 to 256).
//
// One CTA owns two 128-row query tiles of one (batch, query head) and walks
// the key/value blocks of 128 rows that any of its rows can see (causal and
// window masks are resolved per block: blocks nobody sees are never loaded,
// blocks everybody sees are never masked).  Per block and tile:
//
//   S = Q K^T           tcgen05.mma, Q and K from shared memory (TMA, 128B
//                       swizzle), fp32 accumulator in tensor memory (TMEM)
//   online softmax      one thread per row: row max, exp2, row sum, P rounded
//                       to the input type and written back over S in TMEM;
//                       O is rescaled only when the running max grows by more
//                       than 2^8 (exact: the same reference max is used for P,
//                       l and O, and the final O / l cancels it)
//   O += P V            tcgen05.mma with P read from TMEM, V from shared memory
//
// Warp roles (320 threads): warps 0-3 softmax + epilogue of tile 0, warps 4-7
// the same for tile 1, warp 8 issues TMA loads, warp 9 allocates TMEM and
// issues the MMAs.  Tiles are handed between roles with mbarriers; every wait
// is bounded by the watchdog.  At head dim 256 a CTA owns one query tile
// (192 threads: warps 0-3 softmax, 4 loads, 5 MMAs), since TMEM holds the
// S and O of one tile only.
//
// TMEM columns (512 allocated): S/P of tile 0 at 0, of tile 1 at 128; O of
// tile 0 at 256, of tile 1 at 256 + D (one tile: S at 0, O at 128).
#include <type_traits>

#include "ptx.cuh"
#include "tc.h"
#include "prof.h"
#include "tmap.h"

namespace gbattn {
namespace {

using namespace ptx;

constexpr int BM = 128;          // query rows per tile
constexpr int BN = 128;          // keys per block
constexpr int kMaxNQ = 2;        // query tiles per CTA (one at D = 256)
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct FwdCfg {
    // Two query tiles per CTA ping-pong on the tensor pipe; at D = 256 the
    // TMEM holds S (128 columns) and O (256) of one tile only, and shared
    // memory one 64 KB K and V stage.
    static constexpr int NQ = D == 256 ? 1 : 2;
    static constexpr int kProdWarp = 4 * NQ;               // after the softmax warps
    static constexpr int kMmaWarp = 4 * NQ + 1;
    static constexpr int kThreads = 32 * (4 * NQ + 2);
    static constexpr int kChunks = D / 64;                 // 64-element swizzle atoms per row
    static constexpr int kTileBytes = BM * D * 2;          // one 128 x D tile
    static constexpr int kStages = D == 256 ? 1 : D == 128 ? 2 : 3;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + NQ * kTileBytes;
    static constexpr int kVOff = kKOff + kStages * kTileBytes;
    static constexpr int kBarOff = kVOff + kStages * kTileBytes;
    static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // + barriers + alignment slack
};

struct Bars {
    uint64_t q_full[kMaxNQ];  // one per query tile: tile 0 starts before tile 1's Q lands
    uint64_t k_full[3], k_empty[3], v_full[3], v_empty[3];
    uint64_t s_full[kMaxNQ], p_full[kMaxNQ], pv_done[kMaxNQ];
    uint32_t tmem_base;
    int abort_flag;
};

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

// Key-block range of one query tile, in blocks relative to the CTA's first key.
struct TileRange {
    int row0;     // first query row of the tile
    int nrows;    // valid rows (0 if the tile lies past the sequence)
    int blo, bhi; // blocks [blo, bhi)
};

template <typename T, int D>
__global__ void __launch_bounds__(FwdCfg<D>::kThreads, 1)
    tc_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, FwdArgs a,
                  int n_mtiles) {
    using C = FwdCfg<D>;
    constexpr int KS = C::kStages;
    constexpr int NQ = C::NQ;
    constexpr int kProdWarp = C::kProdWarp;
    constexpr int kMmaWarp = C::kMmaWarp;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Bars &bar = *reinterpret_cast<Bars *>(smem + C::kBarOff);
    const Geometry &g = a.g;

    // banded work order; rank 0 = the last query tiles (most keys when causal)
    int bh, rank;
    banded_order(blockIdx.x, n_mtiles, g.Hq * g.B, bh, rank);
    const int mt = n_mtiles - 1 - rank;
    const int h = bh % g.Hq, b = bh / g.Hq;
    const int hk = h / g.G;
    const SeqInfo s = seq_info(g, b);
    const int m0 = mt * (BM * NQ);
    if (rank == 0 && threadIdx.x == 0) report_uncovered(a.err, g, s.Lq, n_mtiles * BM * NQ, kErrSeqlenQ);
    if (m0 >= s.Lq) return;

    // key range of the CTA and of each tile
    int jlo, jhi;
    key_range(m0, min(m0 + BM * NQ, s.Lq), s.Lkv, g.wl, g.wr, jlo, jhi);
    const int nb = (jhi - jlo + BN - 1) / BN;
    TileRange tr[NQ];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        tr[i].row0 = m0 + i * BM;
        tr[i].nrows = max(0, min(BM, s.Lq - tr[i].row0));
        tr[i].blo = tr[i].bhi = 0;
        if (tr[i].nrows > 0) {
            int lo, hi;
            key_range(tr[i].row0, tr[i].row0 + tr[i].nrows, s.Lkv, g.wl, g.wr, lo, hi);
            if (hi > lo) {
                tr[i].blo = (lo - jlo) / BN;
                tr[i].bhi = (hi - jlo + BN - 1) / BN;
            }
        }
    }

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // TMA coordinates: (d, row, head, batch); THD views have one "batch"
    const int qb = g.thd ? 0 : b, q_row = s.q0 + m0;
    const int kv_row = s.kv0 + jlo;
    auto load_q = [&](int i) {
        mbar_arrive_expect_tx(&bar.q_full[i], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
            tma_load_4d(smem + C::kQOff + i * C::kTileBytes + c * BM * 128, &tm_q, &bar.q_full[i], c * 64,
                        q_row + i * BM, h, qb);
    };
    auto load_k = [&](int jb) {
        const int st = jb % KS;
        mbar_arrive_expect_tx(&bar.k_full[st], C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
            tma_load_4d(smem + C::kKOff + st * C::kTileBytes + c * BN * 128, &tm_k, &bar.k_full[st], c * 64,
                        kv_row + jb * BN, hk, qb);
    };
    if (warp == kProdWarp && lane == 0) {
        // The loading lane sets up the barriers and issues tile 0's Q and the
        // first K block at once, so those loads overlap the TMEM allocation
        // and the block-wide sync (tile 0's first S product needs only them).
        for (int i = 0; i < kMaxNQ; ++i) mbar_init(&bar.q_full[i], 1);
        for (int i = 0; i < KS; ++i) {
            mbar_init(&bar.k_full[i], 1);
            mbar_init(&bar.k_empty[i], 1);
            mbar_init(&bar.v_full[i], 1);
            mbar_init(&bar.v_empty[i], 1);
        }
        for (int i = 0; i < NQ; ++i) {
            mbar_init(&bar.s_full[i], 1);
            mbar_init(&bar.p_full[i], BM);
            mbar_init(&bar.pv_done[i], 1);
        }
        bar.abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        if (nb > 0) {
            load_q(0);
            load_k(0);
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

    const uint32_t sQ = smem_u32(smem + C::kQOff);
    const uint32_t sK = smem_u32(smem + C::kKOff);
    const uint32_t sV = smem_u32(smem + C::kVOff);

    if (warp == kProdWarp) {
        // ------------------------------------------------------------ TMA
        // (tile 0's Q and K block 0 were issued before the sync; the other
        // tiles' Q follow K block 0)
        if (lane == 0 && nb > 0) {
            for (int jb = 0; jb < nb; ++jb) {
                const int st = jb % KS;
                const uint32_t ph = (jb / KS) & 1;
                if (jb > 0) {
                    if (!mbar_wait(&bar.k_empty[st], ph ^ 1, wd, 0x10)) break;
                    load_k(jb);
                } else {
                    for (int i = 1; i < NQ; ++i) load_q(i);
                }
                if (!mbar_wait(&bar.v_empty[st], ph ^ 1, wd, 0x11)) break;
                mbar_arrive_expect_tx(&bar.v_full[st], C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_4d(smem + C::kVOff + st * C::kTileBytes + c * BN * 128, &tm_v,
                                &bar.v_full[st], c * 64, kv_row + jb * BN, hk, qb);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA
        // Per tile the chain is S -> softmax -> PV; the tiles alternate so one
        // tile's MMAs run while the other tile's softmax does.  Issue order per
        // block jb: PV_0(jb), S_0(jb+1), PV_1(jb), S_1(jb+1).  S_i(jb+1) reuses
        // the TMEM that P_i(jb) occupies; MMAs issued by one thread execute in
        // issue order, so it is written only after PV_i(jb) has read P.
        // Descriptors are formed once; each MMA adds a compile-time offset.
        // The whole warp runs the loop in step (waits, descriptors) and one
        // elected lane issues each group of MMAs with its commit.
        if (nb > 0) {
            constexpr uint32_t idS = idesc_f16(BM, BN, kBf16, 0, 0);
            constexpr uint32_t idPV = idesc_f16(BM, D, kBf16, 0, 1);
            const uint64_t dQ = smem_desc_sw128(sQ, 16, 1024);
            auto wait = [&](uint64_t *b, uint32_t ph, unsigned code) {
                const bool r = __all_sync(0xffffffffu, mbar_wait(b, ph, wd, code));
                if (r) tc_fence_after();
                return r;
            };
            auto issue_s = [&](int i, int jb) {  // S_i = Q_i K_jb^T
                const int st = jb % KS;
                const uint64_t da = desc_add(dQ, i * C::kTileBytes);
                const uint64_t db = smem_desc_sw128(sK + st * C::kTileBytes, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        constexpr int kRow = BM * 128;
                        const uint32_t off = (kk / 4) * kRow + (kk % 4) * 32;
                        mma_ss(tmem + i * BN, desc_add(da, off), desc_add(db, off), idS, kk > 0);
                    }
                    mma_commit(&bar.s_full[i]);
                }
                __syncwarp();
            };
            auto commit = [&](uint64_t *b) {
                if (elect_one()) mma_commit(b);
                __syncwarp();
            };
            auto in_range = [&](int i, int jb) { return jb >= tr[i].blo && jb < tr[i].bhi; };
            bool ok = wait(&bar.k_full[0], 0, 0x21);
            if (ok) {
#pragma unroll
                for (int i = 0; i < NQ; ++i) {
                    if (!(ok = wait(&bar.q_full[i], 0, 0x20))) break;
                    if (in_range(i, 0)) issue_s(i, 0);
                }
                if (ok) commit(&bar.k_empty[0]);
            }
            for (int jb = 0; ok && jb < nb; ++jb) {
                const int st = jb % KS;
                const uint32_t ph = (jb / KS) & 1;
                const bool has_next = jb + 1 < nb;
                if (!(ok = wait(&bar.v_full[st], ph, 0x23))) break;
                if (has_next && !(ok = wait(&bar.k_full[(jb + 1) % KS], ((jb + 1) / KS) & 1, 0x22))) break;
                const uint64_t dv = smem_desc_sw128(sV + st * C::kTileBytes, BN * 128, 1024);
#pragma unroll
                for (int i = 0; i < NQ; ++i) {
                    if (in_range(i, jb)) {
                        const int t = jb - tr[i].blo;
                        if (!(ok = wait(&bar.p_full[i], t & 1, 0x24))) break;
                        const uint32_t acc0 = t > 0 ? 1u : 0u;
                        if (elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < BN / 16; ++kk)
                                mma_ts(tmem + NQ * BN + i * D, tmem + i * BN + kk * 8, desc_add(dv, kk * 16 * 128),
                                       idPV, kk > 0 ? 1u : acc0);
                            mma_commit(&bar.pv_done[i]);
                        }
                        __syncwarp();
                    }
                    if (has_next && in_range(i, jb + 1)) issue_s(i, jb + 1);
                }
                if (!ok) break;
                commit(&bar.v_empty[st]);
                if (has_next) commit(&bar.k_empty[(jb + 1) % KS]);
            }
        }
    } else {
        // ------------------------------------------------- softmax + epilogue
        const int i = warp / 4;          // tile
        const int wq = warp % 4;         // TMEM lane quarter
        const int r = wq * 32 + lane;    // row within the tile
        const int row = tr[i].row0 + r;  // row within the sequence
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + i * BN + lane_off;
        const uint32_t tO = tmem + NQ * BN + i * D + lane_off;
        const int n_i = tr[i].bhi - tr[i].blo;
        const float c2 = g.scale_log2;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int t = 0; t < n_i; ++t) {
            const int jb = tr[i].blo + t;
            const int n0 = jlo + jb * BN;  // first key of the block
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.s_full[i], t & 1, wd, 0x30));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[BN];
            tmem_ld128(tS, sr);
            // mask only blocks that some row of the tile sees only in part
            const int rlo = tr[i].row0, rhi = tr[i].row0 + tr[i].nrows - 1;
            const bool full = (n0 + BN - 1 < s.Lkv) && (g.wr < 0 || n0 + BN - 1 <= rlo + g.wr) &&
                              (g.wl < 0 || n0 >= rhi - g.wl);
            if (!full) {
                // keys visible to this row: columns [vlo, vhi) of the block
                int vlo = 0, vhi = min(BN, s.Lkv - n0);
                if (g.wl >= 0) vlo = max(vlo, row - g.wl - n0);
                if (g.wr >= 0) vhi = min(vhi, row + g.wr + 1 - n0);
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (c < vlo || c >= vhi) sr[c] = __float_as_uint(-INFINITY);
            }
            // four independent chains of three-input maxima
            float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN; c += 8) {
                m0 = max3f(m0, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
                m1 = max3f(m1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
                m2 = max3f(m2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
                m3 = max3f(m3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
            }
            const float mx = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
            const float xm = mx * c2;  // scale > 0, so the max commutes with scaling
            float alpha = 1.f;
            bool resc = false;
            if (xm > m + kRescaleThreshold) {  // also the first visible block (m = -inf)
                alpha = ex2(m - xm);
                m = xm;
                resc = true;
            }
            const float mref = m == -INFINITY ? 0.f : m;
            // scale and subtract two columns per instruction; the row sum in
            // two packed accumulators (four partial sums)
            const uint64_t c2x2 = f2pack(c2, c2), mr2 = f2pack(-mref, -mref);
            uint64_t rsa = 0ull, rsb = 0ull;
#pragma unroll
            for (int c = 0; c < BN / 2; ++c) {
                float x0, x1;
                f2unpack(fma2(f2pack(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), c2x2, mr2), x0,
                         x1);
                const float p0 = ex2(x0), p1 = ex2(x1);
                if (c & 1)
                    rsb = add2(rsb, f2pack(p0, p1));
                else
                    rsa = add2(rsa, f2pack(p0, p1));
                sr[c] = pack2<T>(p0, p1);
            }
            float ra0, ra1;
            f2unpack(add2(rsa, rsb), ra0, ra1);
            const float rs = ra0 + ra1;
            l = l * alpha + rs;
            tmem_st32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
            tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
            // O holds the blocks before this one (their PV completed before
            // this block's S was issued); rescale it when some row's max moved.
            if (t > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t ov[32];
                    tmem_ld32(tO + cc * 32, ov);
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                    tmem_st32(tO + cc * 32, ov);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bar.p_full[i]);
        }
        // epilogue: O / l -> global, LSE
        if (ok && n_i > 0)
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.pv_done[i], (n_i - 1) & 1, wd, 0x31));
        tc_fence_after();
        const bool valid = r < tr[i].nrows;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        if (!g.thd || tr[i].nrows == BM) {
            // Stage O_i in its Q tile (idle once the tile's last S MMA has
            // completed, and its load has landed: a tile without keys may
            // still have it in flight) in the load's 128B-swizzled layout and
            // write it with TMA stores, which drop rows past a dense tensor's
            // end.  A THD tile ending inside the tensor is written row by row.
            if (nb > 0 && !__all_sync(0xffffffffu, mbar_wait(&bar.q_full[i], 0, wd, 0x32))) ok = false;
            uint8_t *stage = smem + C::kQOff + i * C::kTileBytes;
            const uint32_t srow = smem_u32(stage) + r * 128;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t ov[32];
                if (n_i > 0) {
                    tmem_ld32(tO + cc * 32, ov);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = 0u;
                }
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[e] = pack2<T>(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c16 = cc * 4 + q;  // 16-byte chunk of the row: atom c16 / 8
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                     srow + (c16 / 8) * (BM * 128) + ((uint32_t)((c16 % 8) ^ (r & 7)) << 4)),
                                 "r"(w[4 * q]), "r"(w[4 * q + 1]), "r"(w[4 * q + 2]), "r"(w[4 * q + 3])
                                 : "memory");
                }
            }
            fence_proxy_async_smem();
            named_bar_sync(1 + i, 128);
            if (wq == 0 && lane == 0) {
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c)
                    tma_store_4d(&tm_o, stage + c * BM * 128, c * 64, q_row + i * BM, h, qb);
                bulk_commit();
                bulk_wait_read0();  // the copy has read the staging before the CTA exits
            }
        } else {
            T *orow = (T *)a.o.ptr + (int64_t)b * a.o.sb + (int64_t)(s.q0 + row) * a.o.ss +
                      (int64_t)h * a.o.sh;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t ov[32];
                if (n_i > 0) {
                    tmem_ld32(tO + cc * 32, ov);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = 0u;
                }
                if (valid && cc * 32 < g.D) {
                    uint4 pk[4];
                    uint32_t *pw = reinterpret_cast<uint32_t *>(pk);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pw[e] = pack2<T>(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e) dst[e] = pk[e];
                }
            }
        }
        if (valid)
            a.lse[lse_index(g, s, b, h, row)] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
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
cudaError_t launch_typed(const FwdArgs &a, int max_lq, int max_lkv, cudaStream_t st) {
    const int dt = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;
    const Geometry &g = a.g;
    CUtensorMap tq, tk, tv, to;
    // dims (d, rows, heads, batch); THD: rows = all tokens, one batch
    const uint64_t nb = g.thd ? 1 : (uint64_t)g.B;
    // inner extent: the real head dim (columns past it load as zeros)
    uint64_t dq[4] = {(uint64_t)g.D, (uint64_t)g.Sq, (uint64_t)g.Hq, nb};
    uint64_t dk[4] = {(uint64_t)g.D, (uint64_t)g.Skv, (uint64_t)g.Hkv, nb};
    auto strides = [&](const auto &v, const uint64_t dims[4], uint64_t out[3]) {
        tmap_strides(v.ss, v.sh, g.thd ? 0 : v.sb, dims, out);
    };
    uint64_t sq[3], sk[3], sv[3], so[3];
    strides(a.q, dq, sq);
    strides(a.k, dk, sk);
    strides(a.v, dk, sv);
    strides(a.o, dq, so);
    cudaError_t e;
    if ((e = make_tmap_16bit(&tq, a.q.ptr, dt, dq, sq, BM)) != cudaSuccess) return e;
    if ((e = make_tmap_16bit(&tk, a.k.ptr, dt, dk, sk, BN)) != cudaSuccess) return e;
    if ((e = make_tmap_16bit(&tv, a.v.ptr, dt, dk, sv, BN)) != cudaSuccess) return e;
    if ((e = make_tmap_16bit(&to, a.o.ptr, dt, dq, so, BM)) != cudaSuccess) return e;
    const int smem = FwdCfg<D>::kSmemBytes;
    auto kern = tc_fwd_kernel<T, D>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
        cudaSuccess)
        return e;
    constexpr int NQ = FwdCfg<D>::NQ;
    const int n_mtiles = (max_lq + BM * NQ - 1) / (BM * NQ);
    const int64_t grid = (int64_t)n_mtiles * g.Hq * g.B;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
    prof_before(st, kProfFwd);
    kern<<<(unsigned)grid, FwdCfg<D>::kThreads, smem, st>>>(tq, tk, tv, to, a, n_mtiles);
    prof_after(st);
    return cudaGetLastError();
}

}  // namespace

bool uses_tc_fwd(int dtype, int D) {
    return (dtype == 0 || dtype == 1) && (D == 32 || D == 64 || D == 96 || D == 128 || D == 256);
}

cudaError_t launch_tc_fwd(int dtype, const FwdArgs &a, int max_lq, int max_lkv, cudaStream_t st) {
    if (a.g.D == 256) {
        if (dtype == 0) return launch_typed<__half, 256>(a, max_lq, max_lkv, st);
        if (dtype == 1) return launch_typed<__nv_bfloat16, 256>(a, max_lq, max_lkv, st);
        return cudaErrorInvalidValue;
    }
    switch (dtype * 2 + (tc_dim(a.g.D) == 128)) {
        case 0: return launch_typed<__half, 64>(a, max_lq, max_lkv, st);
        case 1: return launch_typed<__half, 128>(a, max_lq, max_lkv, st);
        case 2: return launch_typed<__nv_bfloat16, 64>(a, max_lq, max_lkv, st);
        case 3: return launch_typed<__nv_bfloat16, 128>(a, max_lq, max_lkv, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gbattn
