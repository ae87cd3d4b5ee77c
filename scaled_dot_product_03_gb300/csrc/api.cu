// api.cu -- the C ABI (include/gbattn.h): argument validation, workspace
// layout, kernel selection by element type, and the device error word.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "gbattn.h"
#include "launch.h"
#include "prof.h"
#include "tc.h"
#include "tmap.h"
#include <vector>

namespace gbattn {
namespace {

thread_local std::string t_error;

attn_status fail(attn_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_error = buf;
    return st;
}

attn_status cuda_fail(cudaError_t e, const char *what) {
    if (e == kTmapRefused)  // a view the tensor-memory accelerator cannot address
        return fail(ATTN_ERR_UNSUPPORTED, "%s: tensor map refused: %s", what, tmap_refusal());
    return fail(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device error word set by bounded device-side waits that gave up.
__device__ unsigned int g_device_error;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned *g_err_ptr[kMaxDevices];
uint64_t g_watchdog_ns = 2000000000ull;

attn_status device_error_word(unsigned **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_CUDA, "device index %d too large", dev);
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_error);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(device error word)");
        g_err_ptr[dev] = (unsigned *)p;
    }
    *out = g_err_ptr[dev];
    return ATTN_OK;
}

uint64_t watchdog_ns() {
    std::lock_guard<std::mutex> lock(g_mu);
    return g_watchdog_ns;
}

size_t elt_size(attn_dtype dt) { return dt == ATTN_F32 ? 4 : 2; }

bool dtype_ok(int dt) { return dt == ATTN_F16 || dt == ATTN_BF16 || dt == ATTN_F32; }

// Validates the shared problem description.
attn_status check_params(const attn_params *p) {
    if (!p) return fail(ATTN_ERR_INVALID_ARG, "params is NULL");
    if (!dtype_ok(p->dtype)) return fail(ATTN_ERR_INVALID_ARG, "unknown dtype %d", (int)p->dtype);
    if (p->layout != ATTN_LAYOUT_DENSE4D && p->layout != ATTN_LAYOUT_THD)
        return fail(ATTN_ERR_INVALID_ARG, "unknown layout %d", (int)p->layout);
    if (p->B < 0 || p->Sq < 0 || p->Skv < 0)
        return fail(ATTN_ERR_INVALID_ARG, "negative size (B=%d Sq=%d Skv=%d)", p->B, p->Sq, p->Skv);
    if (p->Hq < 1 || p->Hkv < 1 || p->Hq % p->Hkv != 0)
        return fail(ATTN_ERR_INVALID_ARG, "Hq=%d must be a positive multiple of Hkv=%d", p->Hq, p->Hkv);
    if (p->D != 32 && p->D != 64 && p->D != 96 && p->D != 128 && p->D != 256)
        return fail(ATTN_ERR_UNSUPPORTED, "head dim %d not supported (32, 64, 96, 128; 256 forward only)", p->D);
    if (p->deterministic != 0 && p->deterministic != 1)
        return fail(ATTN_ERR_INVALID_ARG, "deterministic must be 0 or 1");
    if (p->window_left < -1 || p->window_right < -1)
        return fail(ATTN_ERR_INVALID_ARG, "window (%d, %d): each bound must be >= -1",
                    p->window_left, p->window_right);
    if (!std::isfinite(p->scale) || !(p->scale > 0.f))
        return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and positive");
    if (p->layout == ATTN_LAYOUT_THD) {
        if (p->B > 0 && (!p->cu_seqlens_q || !p->cu_seqlens_kv))
            return fail(ATTN_ERR_INVALID_ARG, "THD layout needs cu_seqlens_q and cu_seqlens_kv");
        if (p->max_seqlen_q < 0 || p->max_seqlen_kv < 0)
            return fail(ATTN_ERR_INVALID_ARG, "negative max_seqlen");
        if (p->max_seqlen_q > p->Sq || p->max_seqlen_kv > p->Skv)
            return fail(ATTN_ERR_INVALID_ARG, "max_seqlen exceeds the total token rows");
    } else if (p->cu_seqlens_q_padded || p->cu_seqlens_kv_padded) {
        return fail(ATTN_ERR_INVALID_ARG, "padded cu_seqlens need the THD layout");
    }
    return ATTN_OK;
}

// Largest byte stride a tensor map can step (the tensor-memory accelerator
// holds strides in 40 bits).
constexpr int64_t kMaxTmaStride = (int64_t)1 << 40;

// Checks a view.  rows / heads: extents of its sequence and head dims (the
// batch dim has B); a dim of extent 1 is never stepped, so its stride is
// not checked against the accelerator's limits.
attn_status check_tensor(const attn_params *p, const attn_tensor &t, const char *name, int rows, int heads) {
    if (!t.ptr) return fail(ATTN_ERR_INVALID_ARG, "%s: NULL pointer", name);
    if (t.stride[3] != 1)
        return fail(ATTN_ERR_UNSUPPORTED, "%s: innermost (d) stride %lld must be 1", name,
                    (long long)t.stride[3]);
    const int first = p->layout == ATTN_LAYOUT_THD ? 1 : 0;
    for (int i = first; i < 3; ++i)
        if (t.stride[i] < 0) return fail(ATTN_ERR_UNSUPPORTED, "%s: negative stride", name);
    if (p->dtype != ATTN_F32) {
        const size_t es = elt_size(p->dtype);
        if ((uintptr_t)t.ptr % 16)
            return fail(ATTN_ERR_UNSUPPORTED, "%s: base pointer not 16-byte aligned", name);
        const int extent[3] = {p->B, rows, heads};
        for (int i = first; i < 3; ++i) {
            if (extent[i] <= 1) continue;
            if ((t.stride[i] * (int64_t)es) % 16)
                return fail(ATTN_ERR_UNSUPPORTED,
                            "%s: stride[%d]=%lld elements is not a multiple of 16 bytes", name, i,
                            (long long)t.stride[i]);
            if (t.stride[i] >= kMaxTmaStride / (int64_t)es)
                return fail(ATTN_ERR_UNSUPPORTED,
                            "%s: stride[%d]=%lld elements is 2^40 bytes or more, beyond what a "
                            "tensor map can step", name, i, (long long)t.stride[i]);
        }
    } else if ((uintptr_t)t.ptr % 4) {
        return fail(ATTN_ERR_UNSUPPORTED, "%s: base pointer not 4-byte aligned", name);
    }
    return ATTN_OK;
}

View view_of(const attn_params *p, const attn_tensor &t) {
    View v;
    v.ptr = t.ptr;
    v.sb = p->layout == ATTN_LAYOUT_THD ? 0 : t.stride[0];
    v.ss = t.stride[1];
    v.sh = t.stride[2];
    return v;
}

MutView mview_of(const attn_params *p, const attn_tensor &t) {
    MutView v;
    v.ptr = t.ptr;
    v.sb = p->layout == ATTN_LAYOUT_THD ? 0 : t.stride[0];
    v.ss = t.stride[1];
    v.sh = t.stride[2];
    return v;
}

Geometry geometry_of(const attn_params *p) {
    Geometry g;
    g.B = p->B;
    g.Sq = p->Sq;
    g.Skv = p->Skv;
    g.Hq = p->Hq;
    g.Hkv = p->Hkv;
    g.D = p->D;
    g.G = p->Hq / p->Hkv;
    g.thd = p->layout == ATTN_LAYOUT_THD;
    g.Tq = p->Sq;
    g.cu_q = p->cu_seqlens_q;
    g.cu_kv = p->cu_seqlens_kv;
    g.pad_q = p->cu_seqlens_q_padded;
    g.pad_kv = p->cu_seqlens_kv_padded;
    g.wl = p->window_left;
    g.wr = p->window_right;
    g.scale = p->scale;
    g.scale_log2 = p->scale * kLog2e;
    return g;
}

int max_lq(const attn_params *p) { return p->layout == ATTN_LAYOUT_THD ? p->max_seqlen_q : p->Sq; }
int max_lkv(const attn_params *p) { return p->layout == ATTN_LAYOUT_THD ? p->max_seqlen_kv : p->Skv; }
int64_t q_rows(const attn_params *p) {
    return p->layout == ATTN_LAYOUT_THD ? (int64_t)p->Sq : (int64_t)p->B * p->Sq;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Single-pass backward: not asked to be deterministic, covered by the
// kernel, and at least one query row (the fp32 accumulator is not empty).
bool fused_bwd(const attn_params *p) {
    return !p->deterministic && uses_tc_bwd_fused(p->dtype, p->D) && max_lq(p) > 0;
}

// CTAs below which the single-pass backward splits the query heads of a
// key/value group over several CTAs per key tile: twice the SM count of a
// GB300 (152).  A constant rather than the device's count, so that the
// workspace size and the order of the partial sums depend on the problem
// alone.
constexpr int64_t kSplitTargetCtas = 2 * 152;

// Query-head splits per key tile of the tensor-core dK / dV kernels (the
// single pass and the deterministic two-kernel form): 1 unless the grid of
// (key tile, key/value head, sequence) units is small and the groups have
// several query heads (multi- and grouped-query attention with few
// key/value heads), in which case enough splits to reach the target, with
// every split non-empty.  The partial dK, dV of the splits are summed in
// split order, so both forms keep dK and dV reproducible.
int fused_split(const attn_params *p) {
    const int G = p->Hq / p->Hkv;
    if (G == 1 || !uses_tc_bwd(p->dtype, p->D) || max_lq(p) == 0) return 1;
    const int64_t units = (int64_t)((max_lkv(p) + 127) / 128) * p->Hkv * p->B;
    if (units <= 0 || units >= kSplitTargetCtas) return 1;
    const int64_t want = std::min<int64_t>(G, (kSplitTargetCtas + units - 1) / units);
    const int gs = (int)((G + want - 1) / want);  // query heads per split
    return (G + gs - 1) / gs;
}

int64_t kv_rows(const attn_params *p) {
    return p->layout == ATTN_LAYOUT_THD ? (int64_t)p->Skv : (int64_t)p->B * p->Skv;
}

struct WsLayout {
    size_t delta_off, acc_off, part_off, ctr_off, total;
    bool fused;
    int nsplit;
};

// Workspace: the fp32 row terms delta_i = <dO_i, O_i>, laid out like LSE,
// then (single-pass backward only) the fp32 dq accumulator, D floats per
// LSE entry, then (split query heads only) the fp32 partial dK and dV of
// every split, then (single pass) the work counter of its persistent CTAs.
WsLayout ws_layout(const attn_params *p) {
    WsLayout w;
    const size_t rows = (size_t)q_rows(p) * p->Hq;
    w.fused = fused_bwd(p);
    w.nsplit = fused_split(p);
    w.delta_off = 0;
    w.acc_off = round_up(sizeof(float) * rows, 256);
    // (the tensor-core kernels lay out dq sums and partials tc_dim(D) wide)
    const size_t dc = (size_t)tc_dim(p->D);
    w.part_off = w.fused ? w.acc_off + round_up(sizeof(float) * rows * dc, 256) : w.acc_off;
    w.total = w.part_off;
    if (w.nsplit > 1)
        w.total += round_up(sizeof(float) * (size_t)w.nsplit * 2 * kv_rows(p) * p->Hkv * dc, 256);
    w.ctr_off = w.total;
    if (w.fused) w.total += 256;
    return w;
}

}  // namespace

cudaError_t device_sm_count(int *out) {
    static std::mutex mu;
    static int counts[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!counts[dev]) {
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        counts[dev] = n > 0 ? n : 1;
    }
    *out = counts[dev];
    return cudaSuccess;
}

// ----------------------------------------------------------------- timing
// Per-thread launch timing: while enabled, each kernel launch is bracketed
// by two events recorded on its stream.
struct ProfState {
    bool on = false;
    int cap = 0, n = 0;
    std::vector<cudaEvent_t> ev;  // 2 per launch
    std::vector<int> kind;
};
thread_local ProfState t_prof;

void prof_before(cudaStream_t st, int kind) {
    ProfState &p = t_prof;
    if (!p.on || p.n >= p.cap) return;
    cudaEventRecord(p.ev[2 * p.n], st);
    p.kind[p.n] = kind;
}

void prof_after(cudaStream_t st) {
    ProfState &p = t_prof;
    if (!p.on || p.n >= p.cap) return;
    cudaEventRecord(p.ev[2 * p.n + 1], st);
    ++p.n;
}

attn_status record_error(attn_status st, const char *msg) {
    t_error = msg;
    return st;
}

}  // namespace gbattn

using namespace gbattn;

extern "C" {

const char *attn_last_error_string(void) { return t_error.c_str(); }

uint64_t attn_set_watchdog_ns(uint64_t ns) {
    std::lock_guard<std::mutex> lock(g_mu);
    const uint64_t old = g_watchdog_ns;
    g_watchdog_ns = ns;
    return old;
}

attn_status attn_check_device_error(attn_stream_t stream) {
    unsigned *word = nullptr;
    attn_status st = device_error_word(&word);
    if (st != ATTN_OK) return st;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned v = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof v);
    if (e != cudaSuccess) return cuda_fail(e, "read device error word");
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
        if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
        if (v & (kErrSeqlenQ | kErrSeqlenKv))
            return fail(ATTN_ERR_INVALID_ARG,
                        "a THD sequence is longer than max_seqlen_%s: rows past that length were not "
                        "computed (code 0x%x)", (v & kErrSeqlenQ) ? "q" : "kv", v);
        return fail(ATTN_ERR_TIMEOUT, "a device-side wait gave up (code 0x%x)", v);
    }
    return ATTN_OK;
}

attn_status attn_fwd(const attn_params *p, attn_tensor q, attn_tensor k, attn_tensor v,
                     attn_tensor o, float *lse, attn_stream_t stream) {
    t_error.clear();
    attn_status st = check_params(p);
    if (st != ATTN_OK) return st;
    if (p->D == 256 && p->dtype == ATTN_F32)
        return fail(ATTN_ERR_UNSUPPORTED, "head dim 256 runs on the fp16 / bf16 tensor-core forward only");
    if (p->B == 0 || max_lq(p) == 0) return ATTN_OK;  // no query row: nothing to write
    const int rq = p->Sq, rkv = p->Skv;
    if ((st = check_tensor(p, q, "q", rq, p->Hq)) || (st = check_tensor(p, k, "k", rkv, p->Hkv)) ||
        (st = check_tensor(p, v, "v", rkv, p->Hkv)) || (st = check_tensor(p, o, "o", rq, p->Hq)))
        return st;
    if (!lse) return fail(ATTN_ERR_INVALID_ARG, "lse: NULL pointer");
    FwdArgs a;
    a.g = geometry_of(p);
    a.q = view_of(p, q);
    a.k = view_of(p, k);
    a.v = view_of(p, v);
    a.o = mview_of(p, o);
    a.lse = lse;
    a.watchdog_ns = watchdog_ns();
    if ((st = device_error_word(&a.err))) return st;
    cudaError_t e;
    if (uses_tc_fwd(p->dtype, p->D))
        e = launch_tc_fwd(p->dtype, a, max_lq(p), max_lkv(p), (cudaStream_t)stream);
    else
        e = launch_simt_fwd(p->dtype, a, max_lq(p), (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "attn_fwd launch");
    return ATTN_OK;
}

size_t attn_bwd_workspace_size(const attn_params *p) {
    if (check_params(p) != ATTN_OK || p->D == 256) return 0;
    return ws_layout(p).total;
}

}  // extern "C"

namespace gbattn {
namespace {

attn_status bwd_impl(const attn_params *p, attn_tensor q, attn_tensor k, attn_tensor v, attn_tensor o,
                     attn_tensor dout, const float *lse, const float *dlse, attn_tensor dq, attn_tensor dk,
                     attn_tensor dv, void *workspace, size_t workspace_bytes, attn_stream_t stream) {
    t_error.clear();
    attn_status st = check_params(p);
    if (st != ATTN_OK) return st;
    if (p->D == 256)  // 256-column dK and dV accumulators do not fit the tensor memory
        return fail(ATTN_ERR_UNSUPPORTED, "head dim 256: forward only");
    // Nothing to write when there is neither a query row (dq) nor a key row (dk, dv).
    if (p->B == 0 || (max_lq(p) == 0 && max_lkv(p) == 0)) return ATTN_OK;
    const int rq = p->Sq, rkv = p->Skv;
    if ((st = check_tensor(p, q, "q", rq, p->Hq)) || (st = check_tensor(p, k, "k", rkv, p->Hkv)) ||
        (st = check_tensor(p, v, "v", rkv, p->Hkv)) || (st = check_tensor(p, o, "o", rq, p->Hq)) ||
        (st = check_tensor(p, dout, "dout", rq, p->Hq)) || (st = check_tensor(p, dq, "dq", rq, p->Hq)) ||
        (st = check_tensor(p, dk, "dk", rkv, p->Hkv)) || (st = check_tensor(p, dv, "dv", rkv, p->Hkv)))
        return st;
    if (!lse) return fail(ATTN_ERR_INVALID_ARG, "lse: NULL pointer");
    const WsLayout w = ws_layout(p);
    if (!workspace && w.total) return fail(ATTN_ERR_INVALID_ARG, "workspace: NULL pointer");
    if ((uintptr_t)workspace % 256) return fail(ATTN_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    if (workspace_bytes < w.total)
        return fail(ATTN_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", workspace_bytes,
                    w.total);
    BwdArgs a;
    a.g = geometry_of(p);
    a.q = view_of(p, q);
    a.k = view_of(p, k);
    a.v = view_of(p, v);
    a.o = view_of(p, o);
    a.dout = view_of(p, dout);
    a.lse = lse;
    a.dlse = dlse;
    a.dq = mview_of(p, dq);
    a.dk = mview_of(p, dk);
    a.dv = mview_of(p, dv);
    a.delta = (float *)((char *)workspace + w.delta_off);
    a.dq_acc = w.fused ? (float *)((char *)workspace + w.acc_off) : nullptr;
    a.nsplit = w.nsplit;
    a.acc_d = tc_dim(p->D);
    a.dkv_part = w.nsplit > 1 ? (float *)((char *)workspace + w.part_off) : nullptr;
    a.work_ctr = w.fused ? (unsigned *)((char *)workspace + w.ctr_off) : nullptr;
    a.watchdog_ns = watchdog_ns();
    if ((st = device_error_word(&a.err))) return st;
    const cudaStream_t s = (cudaStream_t)stream;
    // each launcher encodes its tensor maps before its first launch (the
    // row-term preprocess), so a refused view enqueues nothing
    cudaError_t e;
    if (w.fused)
        e = launch_tc_bwd_fused(p->dtype, a, max_lkv(p), (int)q_rows(p), s);
    else if (uses_tc_bwd(p->dtype, p->D))
        e = launch_tc_bwd(p->dtype, a, max_lq(p), max_lkv(p), (int)q_rows(p), s);
    else
        e = launch_simt_bwd(p->dtype, a, max_lq(p), max_lkv(p), (int)q_rows(p), s);
    if (e != cudaSuccess) return cuda_fail(e, "attn_bwd launch");
    return ATTN_OK;
}

}  // namespace
}  // namespace gbattn

extern "C" {

attn_status attn_bwd(const attn_params *p, attn_tensor q, attn_tensor k, attn_tensor v,
                     attn_tensor o, attn_tensor dout, const float *lse, attn_tensor dq,
                     attn_tensor dk, attn_tensor dv, void *workspace, size_t workspace_bytes,
                     attn_stream_t stream) {
    return bwd_impl(p, q, k, v, o, dout, lse, nullptr, dq, dk, dv, workspace, workspace_bytes, stream);
}

attn_status attn_bwd_dlse(const attn_params *p, attn_tensor q, attn_tensor k, attn_tensor v,
                          attn_tensor o, attn_tensor dout, const float *lse, const float *dlse,
                          attn_tensor dq, attn_tensor dk, attn_tensor dv, void *workspace,
                          size_t workspace_bytes, attn_stream_t stream) {
    return bwd_impl(p, q, k, v, o, dout, lse, dlse, dq, dk, dv, workspace, workspace_bytes, stream);
}

attn_status attn_merge_lse(attn_dtype dtype, int B, int S, int H, int D, attn_tensor o1,
                           const float *lse1, attn_tensor o2, const float *lse2,
                           attn_tensor o_out, float *lse_out, attn_stream_t stream) {
    t_error.clear();
    if (!dtype_ok(dtype)) return fail(ATTN_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (B < 0 || S < 0 || H < 0) return fail(ATTN_ERR_INVALID_ARG, "negative size");
    if (D < 1 || D > 256) return fail(ATTN_ERR_UNSUPPORTED, "head dim %d not in 1..256", D);
    if ((int64_t)B * S * H == 0) return ATTN_OK;
    const attn_tensor *ts[3] = {&o1, &o2, &o_out};
    const char *names[3] = {"o1", "o2", "o_out"};
    for (int i = 0; i < 3; ++i) {
        if (!ts[i]->ptr) return fail(ATTN_ERR_INVALID_ARG, "%s: NULL pointer", names[i]);
        if (ts[i]->stride[3] != 1)
            return fail(ATTN_ERR_UNSUPPORTED, "%s: innermost stride must be 1", names[i]);
        if ((uintptr_t)ts[i]->ptr % elt_size(dtype))
            return fail(ATTN_ERR_UNSUPPORTED, "%s: misaligned pointer", names[i]);
    }
    if (!lse1 || !lse2 || !lse_out) return fail(ATTN_ERR_INVALID_ARG, "lse: NULL pointer");
    MergeArgs a;
    a.B = B;
    a.S = S;
    a.H = H;
    a.D = D;
    a.o1 = View{o1.ptr, o1.stride[0], o1.stride[1], o1.stride[2]};
    a.o2 = View{o2.ptr, o2.stride[0], o2.stride[1], o2.stride[2]};
    a.out = MutView{o_out.ptr, o_out.stride[0], o_out.stride[1], o_out.stride[2]};
    a.lse1 = lse1;
    a.lse2 = lse2;
    a.lse_out = lse_out;
    cudaError_t e = launch_merge(dtype, a, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "attn_merge_lse launch");
    return ATTN_OK;
}

attn_status attn_merge_lse_bwd(attn_dtype dtype, int B, int S, int H, int D, attn_tensor o1,
                               const float *lse1, attn_tensor o2, const float *lse2, attn_tensor dout,
                               const float *dlse, attn_tensor do1, float *dlse1, attn_tensor do2,
                               float *dlse2, attn_stream_t stream) {
    t_error.clear();
    if (!dtype_ok(dtype)) return fail(ATTN_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (B < 0 || S < 0 || H < 0) return fail(ATTN_ERR_INVALID_ARG, "negative size");
    if (D < 1 || D > 256) return fail(ATTN_ERR_UNSUPPORTED, "head dim %d not in 1..256", D);
    if ((int64_t)B * S * H == 0) return ATTN_OK;
    const attn_tensor *ts[5] = {&o1, &o2, &dout, &do1, &do2};
    const char *names[5] = {"o1", "o2", "dout", "do1", "do2"};
    for (int i = 0; i < 5; ++i) {
        if (!ts[i]->ptr) return fail(ATTN_ERR_INVALID_ARG, "%s: NULL pointer", names[i]);
        if (ts[i]->stride[3] != 1)
            return fail(ATTN_ERR_UNSUPPORTED, "%s: innermost stride must be 1", names[i]);
        if ((uintptr_t)ts[i]->ptr % elt_size(dtype))
            return fail(ATTN_ERR_UNSUPPORTED, "%s: misaligned pointer", names[i]);
    }
    if (!lse1 || !lse2 || !dlse1 || !dlse2) return fail(ATTN_ERR_INVALID_ARG, "lse: NULL pointer");
    MergeBwdArgs a;
    a.B = B;
    a.S = S;
    a.H = H;
    a.D = D;
    a.o1 = View{o1.ptr, o1.stride[0], o1.stride[1], o1.stride[2]};
    a.o2 = View{o2.ptr, o2.stride[0], o2.stride[1], o2.stride[2]};
    a.dout = View{dout.ptr, dout.stride[0], dout.stride[1], dout.stride[2]};
    a.do1 = MutView{do1.ptr, do1.stride[0], do1.stride[1], do1.stride[2]};
    a.do2 = MutView{do2.ptr, do2.stride[0], do2.stride[1], do2.stride[2]};
    a.lse1 = lse1;
    a.lse2 = lse2;
    a.dlse = dlse;
    a.dlse1 = dlse1;
    a.dlse2 = dlse2;
    cudaError_t e = launch_merge_bwd(dtype, a, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "attn_merge_lse_bwd launch");
    return ATTN_OK;
}

attn_status attn_thd_partitioned_indices(const int32_t *cu_seqlens_padded, int B, int total_tokens,
                                         int world_size, int rank, int32_t *indices,
                                         attn_stream_t stream) {
    t_error.clear();
    if (world_size < 1 || rank < 0 || rank >= world_size)
        return fail(ATTN_ERR_INVALID_ARG, "rank %d of world size %d", rank, world_size);
    if (B < 0 || total_tokens < 0) return fail(ATTN_ERR_INVALID_ARG, "negative size");
    if (total_tokens % (2 * world_size))
        return fail(ATTN_ERR_INVALID_ARG, "total_tokens %d is not a multiple of 2 x world size %d",
                    total_tokens, world_size);
    if (total_tokens == 0) return ATTN_OK;
    if (B < 1 || !cu_seqlens_padded || !indices)
        return fail(ATTN_ERR_INVALID_ARG, "need B >= 1 and non-NULL cu_seqlens_padded, indices");
    cudaError_t e = launch_partitioned_indices(cu_seqlens_padded, B, world_size, rank,
                                               total_tokens / world_size, indices, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "attn_thd_partitioned_indices launch");
    return ATTN_OK;
}

namespace {

attn_status thd_rows(const char *name, attn_dtype dtype, int T, int H, int D, attn_tensor v, float *acc,
                     const int32_t *cu, const int32_t *pad, int B, int mode, attn_stream_t stream) {
    t_error.clear();
    if (dtype != ATTN_F16 && dtype != ATTN_BF16 && dtype != ATTN_F32)
        return fail(ATTN_ERR_INVALID_ARG, "%s: unknown dtype %d", name, (int)dtype);
    if (T < 0 || H < 0 || B < 0) return fail(ATTN_ERR_INVALID_ARG, "%s: negative size", name);
    if (D < 8 || D > 256 || D % 8) return fail(ATTN_ERR_INVALID_ARG, "%s: D = %d is not a multiple of 8 in [8, 256]", name, D);
    if ((int64_t)T * H == 0) return ATTN_OK;
    if (B < 1 || !cu || !v.ptr || !acc) return fail(ATTN_ERR_INVALID_ARG, "%s: need B >= 1 and non-NULL pointers", name);
    const int64_t elt = dtype == ATTN_F32 ? 4 : 2;
    if (v.stride[3] != 1) return fail(ATTN_ERR_INVALID_ARG, "%s: the d stride must be 1", name);
    if ((uintptr_t)v.ptr % 16 || (uintptr_t)acc % 16 || (v.stride[1] * elt) % 16 || (v.stride[2] * elt) % 16)
        return fail(ATTN_ERR_INVALID_ARG, "%s: pointers and strides must be 16-byte aligned", name);
    MutView mv;
    mv.ptr = v.ptr;
    mv.sb = 0;
    mv.ss = v.stride[1];
    mv.sh = v.stride[2];
    cudaError_t e = launch_thd_rows((int)dtype, mode, T, H, D, mv, acc, cu, pad, B, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, name);
    return ATTN_OK;
}

}  // namespace

attn_status attn_thd_accumulate(attn_dtype dtype, int T, int H, int D, attn_tensor src, float *acc, int accumulate,
                                const int32_t *cu_seqlens, const int32_t *cu_seqlens_padded, int B,
                                attn_stream_t stream) {
    return thd_rows("attn_thd_accumulate", dtype, T, H, D, src, acc, cu_seqlens, cu_seqlens_padded, B,
                    accumulate ? 0 : 2, stream);
}

attn_status attn_thd_store(attn_dtype dtype, int T, int H, int D, const float *acc, attn_tensor dst,
                           const int32_t *cu_seqlens, const int32_t *cu_seqlens_padded, int B,
                           attn_stream_t stream) {
    return thd_rows("attn_thd_store", dtype, T, H, D, dst, const_cast<float *>(acc), cu_seqlens, cu_seqlens_padded,
                    B, 1, stream);
}

attn_status attn_profile_begin(int max_launches) {
    t_error.clear();
    if (max_launches < 1) return fail(ATTN_ERR_INVALID_ARG, "max_launches must be positive");
    ProfState &p = t_prof;
    if ((int)p.ev.size() < 2 * max_launches) {
        const size_t old = p.ev.size();
        p.ev.resize(2 * (size_t)max_launches);
        for (size_t i = old; i < p.ev.size(); ++i) {
            cudaError_t e = cudaEventCreate(&p.ev[i]);
            if (e != cudaSuccess) {
                p.ev.resize(i);
                return cuda_fail(e, "cudaEventCreate");
            }
        }
    }
    p.kind.assign(max_launches, -1);
    p.cap = max_launches;
    p.n = 0;
    p.on = true;
    return ATTN_OK;
}

int attn_profile_read(float *ms, int *kind, int capacity) {
    ProfState &p = t_prof;
    if (!p.on) return 0;
    p.on = false;
    const int n = p.n < capacity ? p.n : capacity;
    for (int i = 0; i < n; ++i) {
        if (cudaEventSynchronize(p.ev[2 * i + 1]) != cudaSuccess) return -1;
        float t = 0.f;
        if (cudaEventElapsedTime(&t, p.ev[2 * i], p.ev[2 * i + 1]) != cudaSuccess) return -1;
        if (ms) ms[i] = t;
        if (kind) kind[i] = p.kind[i];
    }
    return n;
}

attn_status attn_watchdog_selftest(attn_stream_t stream) {
    t_error.clear();
    unsigned *word = nullptr;
    attn_status st = device_error_word(&word);
    if (st != ATTN_OK) return st;
    cudaError_t e = launch_watchdog_selftest(word, watchdog_ns(), (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "watchdog self-test launch");
    return ATTN_OK;
}

}  // extern "C"
