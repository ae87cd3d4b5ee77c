/*
 * gbattn.h -- C ABI of a fused scaled-dot-product attention library for
 * NVIDIA GB300 (sm_103a).
 *
 * Operation.  For every query row i of every query head h
 *
 *     O_i   = sum_j softmax_j(scale * <q_i, k_j>) v_j     over visible keys j
 *     LSE_i = log sum_j exp(scale * <q_i, k_j>)           (natural log)
 *
 * which is the operation behind every attention API the source pages call:
 * torch.nn.functional.scaled_dot_product_attention and FlashAttention
 * ("Add torch scaled dot product attention (FlashAttention)", title and
 * benchmark), flex_attention with return_lse=True ("Significant Accuracy
 * Difference between Compiled and Eager Flex Attention", repro and the
 * merge_attn example), and TransformerEngine's FlashAttention /
 * FusedAttention modules ("[PyTorch] fused CUDNN attention kernel not
 * properly handling strides", repro).
 *
 * Visibility.  Key j is visible to query i iff
 *     (window_left  < 0 or j >= i - window_left) and
 *     (window_right < 0 or j <= i + window_right) and 0 <= j < L_kv,
 * with i and j both counted from 0 inside their own sequence (top-left
 * alignment).  window = (-1, 0) is causal, as in the TransformerEngine
 * repro's window_size=(-1, 0); (band, 0) is the sliding-window-causal mask
 * (q_idx >= kv_idx) & (q_idx - kv_idx <= band) of the flex-attention repro.
 * A query row with no visible key gets O = 0 and LSE = -inf.
 *
 * Grouped heads.  Hq must be a multiple of Hkv; query head h reads key/value
 * head h / (Hq / Hkv) (the repro's q_heads=16, kv_heads=1, num_gqa_groups).
 *
 * Layouts.  No layout is ever guessed and no input is ever copied: each
 * tensor is described by a pointer and explicit element strides, so views
 * such as the packed sb(h+2h_g)d split of the TransformerEngine strides
 * issue (strides (1152, 1152, 64, 1)) are read where they lie.
 *   ATTN_LAYOUT_DENSE4D: element (b, s, h, d) lives at
 *       ptr + b*stride[0] + s*stride[1] + h*stride[2] + d*stride[3]
 *     This covers bshd, sbhd, bhsd and split packed layouts alike.
 *   ATTN_LAYOUT_THD: packed variable-length batch ("[PyTorch] Add support
 *     for cuDNN FusedAttention + THD + CP", the thd branch): element
 *     (t, h, d) lives at ptr + t*stride[1] + h*stride[2] + d*stride[3]
 *     (stride[0] is ignored); sequence b owns token rows
 *     [cu_seqlens[b], cu_seqlens[b+1]).  With cu_seqlens_*_padded (the
 *     thread's cu_seqlens_q_padded / cu_seqlens_kv_padded, used where each
 *     sequence is padded, e.g. to a multiple of 2 x the context-parallel
 *     size) sequence b instead owns rows [padded[b], padded[b] + L_b) with
 *     L_b = cu_seqlens[b+1] - cu_seqlens[b] (padded[b] + L_b <= padded[b+1]
 *     is the caller's to ensure); rows in the gaps are never written and
 *     the LSE keeps the buffer's row numbering.  Gap rows must hold finite
 *     values: a tile that runs past a sequence multiplies them by exact
 *     zero weights.
 * The innermost stride (d) must be 1.  For 16-bit types every other stride
 * and the base pointer must be 16-byte aligned (a tensor-memory-accelerator
 * requirement); otherwise the call fails with ATTN_ERR_UNSUPPORTED rather
 * than copying.  So does a stride of 2^40 bytes or more on a dim of extent
 * above 1 (beyond what a tensor map can step).
 *
 * LSE layout: fp32, contiguous, [B, Hq, Sq] for DENSE4D and [Hq, Tq] for THD.
 *
 * Ownership and threading.  Every pointer is caller-owned device memory,
 * except the attn_params struct itself (host).  The library allocates
 * nothing, copies no input, and never synchronises the host: each call only
 * enqueues kernels on the given stream (NULL = legacy default stream) and
 * returns.  The stream must belong to the calling thread's current device
 * (cudaSetDevice), on which the library launches.  Inputs must stay valid
 * until that work has run.  Calls are thread-safe; the error string is per
 * host thread.
 *
 * Errors.  Every entry point returns an attn_status.  On ATTN_ERR_INVALID_ARG
 * and ATTN_ERR_UNSUPPORTED nothing has been enqueued.  ATTN_ERR_CUDA reports
 * a launch error.  Device-side waits are bounded: a kernel whose pipeline
 * stalls past the watchdog limit sets a device error word and returns; the
 * host reads it with attn_check_device_error().  attn_last_error_string()
 * explains the last failure of the calling thread.
 */
#ifndef GBATTN_H_
#define GBATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GBATTN_API __attribute__((visibility("default")))
#else
#define GBATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so that the header needs no CUDA
 * include. */
typedef struct CUstream_st *attn_stream_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1, /* inconsistent sizes, null pointers, bad window */
    ATTN_ERR_UNSUPPORTED = 2, /* valid request the kernels do not cover (D, alignment) */
    ATTN_ERR_CUDA = 3,        /* a CUDA call or launch failed */
    ATTN_ERR_TIMEOUT = 4      /* a device-side wait ran past the watchdog limit */
} attn_status;

typedef enum { ATTN_F16 = 0, ATTN_BF16 = 1, ATTN_F32 = 2 } attn_dtype;

typedef enum { ATTN_LAYOUT_DENSE4D = 0, ATTN_LAYOUT_THD = 1 } attn_layout;

/* A tensor view: device pointer plus element strides (see Layouts). */
typedef struct {
    void *ptr;
    int64_t stride[4];
} attn_tensor;

typedef struct {
    attn_dtype dtype;    /* element type of q, k, v, o, dO, dq, dk, dv */
    attn_layout layout;
    int B;               /* batch size (DENSE4D) or number of sequences (THD) */
    int Sq, Skv;         /* DENSE4D: sequence lengths.  THD: total token rows
                            Tq and Tkv of the packed q and k/v tensors */
    int Hq, Hkv;         /* query heads, key/value heads (Hq % Hkv == 0) */
    int D;               /* head dimension: 32, 64, 96 or 128 (tensor cores for
                            fp16 / bf16, 32 and 96 on the 64- and 128-wide
                            kernels with zero padding; FFMA kernels for fp32),
                            or 256 (fp16 / bf16 forward only) */
    const int32_t *cu_seqlens_q;  /* THD only: device, B + 1 non-decreasing */
    const int32_t *cu_seqlens_kv; /* offsets starting at 0 (NULL for DENSE4D) */
    int max_seqlen_q;    /* THD only: upper bound of the sequence lengths;
                            grids are sized from it, so a longer sequence is
                            left partly unwritten and reported by
                            attn_check_device_error as ATTN_ERR_INVALID_ARG */
    int max_seqlen_kv;
    float scale;         /* softmax scale, finite and > 0, e.g. 1/sqrt(D) */
    int window_left;     /* -1 = unbounded */
    int window_right;    /* -1 = unbounded; (-1, 0) = causal */
    int deterministic;   /* backward only (see attn_bwd): 0 = single pass with
                            an fp32 dq accumulator, 1 = bitwise reproducible */
    const int32_t *cu_seqlens_q_padded;  /* THD only, optional (NULL: none): */
    const int32_t *cu_seqlens_kv_padded; /* device, B + 1 first rows of the
                            sequences in a padded buffer (see Layouts) */
} attn_params;

/*
 * Forward: O and LSE from q, k, v.
 * q, o: [B, Sq, Hq, D] (or [Tq, Hq, D]); k, v: [B, Skv, Hkv, D] (or
 * [Tkv, Hkv, D]); lse: fp32 as described under "LSE layout".  o and lse
 * are written for every query row (rows with no visible key: 0 and -inf).
 */
GBATTN_API attn_status attn_fwd(const attn_params *p, attn_tensor q, attn_tensor k,
                     attn_tensor v, attn_tensor o, float *lse,
                     attn_stream_t stream);

/*
 * Bytes of device scratch memory attn_bwd needs for these parameters: the
 * fp32 row terms delta_i = <dO_i, O_i> (one per query row and head) and,
 * when the single-pass backward applies (deterministic == 0, fp16 / bf16,
 * at least one query row), an fp32 dq accumulator of D' floats per query row
 * and head, D' = 64 for D <= 64 and 128 otherwise (the head dim the
 * tensor-core kernels compute with).  With grouped heads on a small grid
 * (fewer than 304 units of 128 keys x key/value head x sequence, fp16 /
 * bf16) the query heads of each group are split over several CTAs, and the
 * workspace also holds every split's fp32 partial dK and dV (2 D' floats per
 * key row and key/value head per split), summed in split order, so dK and dV
 * stay reproducible.  Every single-pass workspace also keeps a 256-byte
 * block for the work counter that the persistent CTAs of the D' = 64 single
 * pass take their key tiles from (cleared on the stream by each call).
 * Returns 0 for invalid parameters.
 */
GBATTN_API size_t attn_bwd_workspace_size(const attn_params *p);

/*
 * Backward of the forward above for a loss with gradient dout = dL/dO
 * (the flex-attention repro's out.sum().backward() is dout = ones):
 *   dq = scale * sum_j dS_ij k_j,  dk_j = scale * sum_i dS_ij q_i,
 *   dv_j = sum_i P_ij dO_i,        dS_ij = P_ij (<dO_i, v_j> - <dO_i, O_i>),
 * with P recomputed from q, k and the forward's lse (no saved P); dk and dv
 * sum over the Hq / Hkv query heads that share a key/value head.
 * o and lse must be the forward's outputs for the same inputs.  dq has q's
 * shape, dk and dv k's shape, each with its own strides (they may be views
 * of one packed gradient buffer).
 * Determinism.  With p->deterministic = 0 and fp16 / bf16 inputs, one pass
 * over the (key block, query block) pairs forms S and dP
 * once and adds each pair's share of dq into an fp32 accumulator in the
 * workspace; those fp32 additions happen in an order set by the GPU's
 * scheduling, so dq may differ between runs in its last bits (dk and dv do
 * not).  In every other case (p->deterministic = 1, or fp32) every
 * output element is written by exactly one thread of one kernel and the
 * results do not depend on scheduling.  workspace: device memory of at least
 * attn_bwd_workspace_size(p) bytes, 256-byte aligned, whose contents on
 * entry do not matter; it must not be shared with a call that may run at
 * the same time.
 */
GBATTN_API attn_status attn_bwd(const attn_params *p, attn_tensor q, attn_tensor k,
                     attn_tensor v, attn_tensor o, attn_tensor dout,
                     const float *lse, attn_tensor dq, attn_tensor dk,
                     attn_tensor dv, void *workspace, size_t workspace_bytes,
                     attn_stream_t stream);

/*
 * attn_bwd for a loss that also depends on the forward's LSE output
 * ("Significant Accuracy Difference between Compiled and Eager Flex
 * Attention": flex_attention returns the LSE and merge_attn combines two
 * partial attentions through it, so training that split sends a gradient
 * into each part's LSE).  dlse: gradient of the loss with respect to lse,
 * fp32 in the LSE layout (NULL: zero, which is attn_bwd).  Since
 * d LSE_i / d s_ij = P_ij, it adds P_ij dLSE_i to dS_ij:
 *   dS_ij = P_ij (<dO_i, v_j> - <dO_i, O_i> + dLSE_i).
 * Everything else (arguments, workspace, determinism) is as for attn_bwd.
 */
GBATTN_API attn_status attn_bwd_dlse(const attn_params *p, attn_tensor q, attn_tensor k,
                          attn_tensor v, attn_tensor o, attn_tensor dout,
                          const float *lse, const float *dlse, attn_tensor dq,
                          attn_tensor dk, attn_tensor dv, void *workspace,
                          size_t workspace_bytes, attn_stream_t stream);

/*
 * Merge two partial attentions of the same queries over disjoint key sets
 * (merge_attn in "Significant Accuracy Difference between Compiled and Eager
 * Flex Attention"):
 *   m = max(lse1, lse2); e1 = exp(lse1 - m); e2 = exp(lse2 - m)
 *   o = (o1 e1 + o2 e2) / (e1 + e2);  lse = m + log(e1 + e2)
 * computed in fp32.  A side whose lse is -inf contributes nothing; when both
 * are -inf the row becomes o = 0, lse = -inf.
 * o1, o2, o_out: DENSE4D views [B, S, H, D] of element type dtype (a THD
 * tensor [T, H, D] is passed as B = 1, S = T with stride[0] = 0);
 * lse1, lse2, lse_out: fp32 contiguous [B, H, S].  o_out may alias o1 or
 * o2 exactly and lse_out may alias lse1 or lse2 (in-place merge); other
 * overlaps are undefined.  D: 1..256, D*elt a multiple of 16 bytes for
 * 16-bit types.
 */
GBATTN_API attn_status attn_merge_lse(attn_dtype dtype, int B, int S, int H, int D,
                           attn_tensor o1, const float *lse1, attn_tensor o2,
                           const float *lse2, attn_tensor o_out,
                           float *lse_out, attn_stream_t stream);

/*
 * Backward of attn_merge_lse: given the partial results (o1, lse1), (o2,
 * lse2) that were merged and the gradients dout of the merged o and dlse of
 * the merged lse (NULL: zero), writes
 *   do_k   = w_k dout,
 *   dlse_k = w_k (<dout, o_k - o> + dlse),   w_k = exp(lse_k - lse),
 * the derivative of the merge formula (o = w1 o1 + w2 o2 recomputed in
 * fp32).  A side whose lse is -inf gets zeros.  Layouts and limits as for
 * attn_merge_lse; dout, do1, do2 are views of element type dtype, dlse1 and
 * dlse2 fp32 [B, H, S].  No output may overlap an input or another output;
 * o1 and o2 must be finite.
 */
GBATTN_API attn_status attn_merge_lse_bwd(attn_dtype dtype, int B, int S, int H, int D,
                               attn_tensor o1, const float *lse1, attn_tensor o2,
                               const float *lse2, attn_tensor dout, const float *dlse,
                               attn_tensor do1, float *dlse1, attn_tensor do2,
                               float *dlse2, attn_stream_t stream);

/*
 * Token rows of a padded THD buffer that rank `rank` of `world_size` holds
 * under the load-balanced context-parallel split of "[PyTorch] Add support
 * for cuDNN FusedAttention + THD + CP" (its thd_get_partitioned_indices):
 * every sequence b, padded to cu_seqlens_padded[b+1] - cu_seqlens_padded[b]
 * rows (a multiple of 2 x world_size), is cut into 2 x world_size equal
 * chunks and the rank holds chunk `rank` and chunk 2 x world_size - 1 -
 * rank.  indices (device, int32, total_tokens / world_size entries)
 * receives, sequence by sequence, the rows of the first chunk then of the
 * second.  cu_seqlens_padded: device, B + 1 entries from 0 to total_tokens;
 * the per-sequence multiples are the caller's to ensure.
 */
GBATTN_API attn_status attn_thd_partitioned_indices(const int32_t *cu_seqlens_padded, int B,
                                         int total_tokens, int world_size, int rank,
                                         int32_t *indices, attn_stream_t stream);

/*
 * Gradient sums of the context-parallel ring ("[PyTorch] Add support for
 * cuDNN FusedAttention + THD + CP", which runs THD + CP through the fused
 * attention kernels).  The pages do not spell out the ring's backward; the
 * library takes its plainest reading, the derivative of the merged result:
 * each ring step's attention backward, called with the merged O and LSE,
 * gives the step's share of dQ (rows of the rank's query chunk) and of dK,
 * dV (rows of the key/value chunk it holds), and each gradient is the sum
 * of its shares.
 * These two calls add the shares in fp32 and write the sums out.
 *
 * attn_thd_accumulate: acc[t, h, :] += src[t, h, :] (accumulate = 1) or
 * acc[t, h, :] = src[t, h, :] (accumulate = 0, for a first share) for every
 * head h < H and every token row t inside a sequence (rows
 * cu_seqlens_padded[b] + i, i < cu_seqlens[b+1] - cu_seqlens[b];
 * cu_seqlens_padded NULL: rows cu_seqlens[b] + i).  Other rows of acc are
 * left as they are.
 * attn_thd_store: dst[t, h, :] = acc[t, h, :] in the element type for rows
 * inside a sequence, and 0 for every other row t < T.
 * src / dst: THD views [T, H, D] of element type dtype (fp16, bf16 or fp32;
 * element (t, h, d) at ptr + t*stride[1] + h*stride[2] + d, stride[3] = 1).
 * acc: fp32 [T, H, D], contiguous.  D: a multiple of 8 up to 256.  Pointers
 * (device) and strides must be 16-byte aligned; cu_seqlens (and
 * cu_seqlens_padded) are device int32 with B + 1 entries.  T = 0 or H = 0
 * does nothing.  Returns INVALID_ARG (nothing enqueued) on bad sizes, NULL
 * pointers or misalignment.
 */
GBATTN_API attn_status attn_thd_accumulate(attn_dtype dtype, int T, int H, int D, attn_tensor src,
                                           float *acc, int accumulate, const int32_t *cu_seqlens,
                                           const int32_t *cu_seqlens_padded, int B,
                                           attn_stream_t stream);
GBATTN_API attn_status attn_thd_store(attn_dtype dtype, int T, int H, int D, const float *acc,
                                      attn_tensor dst, const int32_t *cu_seqlens,
                                      const int32_t *cu_seqlens_padded, int B, attn_stream_t stream);

/*
 * Per-launch timing, for benchmarks and profilers.  After
 * attn_profile_begin(n) the calling thread's next (at most n) kernel
 * launches by this library are each bracketed by two CUDA events recorded
 * on the launch stream.  attn_profile_read() waits for those events, writes
 * each launch's duration in milliseconds to ms[i] and its kind (below) to
 * kind[i] for i < capacity (either array may be NULL), ends the timing and
 * returns the number of launches recorded (-1 on a CUDA error).  Recording
 * events adds no work on the GPU beyond the events themselves.
 */
enum {
    ATTN_KERNEL_FWD = 0,            /* tensor-core forward */
    ATTN_KERNEL_BWD_PREPROCESS = 1, /* row terms delta_i = <dO_i, O_i> */
    ATTN_KERNEL_BWD_DKDV = 2,       /* tensor-core dK, dV */
    ATTN_KERNEL_BWD_DQ = 3,         /* tensor-core dQ */
    ATTN_KERNEL_MERGE = 4,          /* LSE merge */
    ATTN_KERNEL_SIMT_FWD = 5,       /* fp32 forward */
    ATTN_KERNEL_SIMT_BWD_DQ = 6,    /* fp32 dQ */
    ATTN_KERNEL_SIMT_BWD_DKDV = 7,  /* fp32 dK, dV */
    ATTN_KERNEL_BWD_FUSED = 8,      /* tensor-core single-pass dK, dV, dQ share */
    ATTN_KERNEL_BWD_DQ_CONVERT = 9, /* fp32 dq accumulator -> dq */
    ATTN_KERNEL_MERGE_BWD = 10,     /* backward of the LSE merge */
    ATTN_KERNEL_BWD_DKV_REDUCE = 11, /* dK, dV summed over split query heads */
    ATTN_KERNEL_THD_ROWS = 12        /* THD gradient sums of the context-parallel ring */
};
GBATTN_API attn_status attn_profile_begin(int max_launches);
GBATTN_API int attn_profile_read(float *ms, int *kind, int capacity);

/*
 * attn_bwd without a caller-provided workspace.  (The source pages have no
 * counterpart: this entry point exists for callers of the library, not for
 * the method.)
 *
 * Some callers cannot allocate device memory at the point where they run the
 * backward pass: code that owns no allocator (a plugin or foreign-language
 * host handed only tensor pointers), or code that must not allocate once its
 * set-up is over.  This variant takes the same arguments as attn_bwd minus
 * the workspace and uses a fixed scratch array that the library itself holds
 * in device memory: GBATTN_NOALLOC_SCRATCH_BYTES bytes, reserved on every GPU
 * that loads this part of the library and held until the process exits.  It
 * never calls cudaMalloc, cudaFree or any allocating routine.
 *
 * Limits and behaviour:
 *   - Problems whose attn_bwd_workspace_size exceeds the scratch size are
 *     rejected with ATTN_ERR_UNSUPPORTED before anything is enqueued.
 *   - The first call on each device looks up the device address of the
 *     scratch (with that device current); make that first call before any
 *     stream capture begins.  When CUDA loads modules lazily, that first
 *     call is also when the scratch is reserved on the device, so a caller
 *     that must not allocate after its set-up should make one accepted
 *     call during set-up.
 *   - Every call, on every stream, shares the one scratch array, which keeps
 *     the previous call's contents (each call clears what it needs cleared).
 *     Calls whose work may overlap on the GPU (different streams without
 *     ordering between them) race on the scratch and give wrong gradients;
 *     serialise them.
 */
#define GBATTN_NOALLOC_SCRATCH_BYTES (64u << 20)
GBATTN_API attn_status attn_bwd_noalloc(const attn_params *p, attn_tensor q,
                                        attn_tensor k, attn_tensor v,
                                        attn_tensor o, attn_tensor dout,
                                        const float *lse, attn_tensor dq,
                                        attn_tensor dk, attn_tensor dv,
                                        attn_stream_t stream);

/* Description of the calling thread's last failure ("" if none). */
GBATTN_API const char *attn_last_error_string(void);

/*
 * Reads and clears the device error word set by kernels on the current
 * device.  Synchronises the given stream first.  Returns ATTN_OK,
 * ATTN_ERR_TIMEOUT (a kernel watchdog gave up), ATTN_ERR_INVALID_ARG (a THD
 * sequence was longer than the call's max_seqlen_q / max_seqlen_kv; the
 * rows past it were not computed), or ATTN_ERR_CUDA if the read itself
 * failed.
 */
GBATTN_API attn_status attn_check_device_error(attn_stream_t stream);

/*
 * Watchdog limit of every bounded device-side wait, in nanoseconds
 * (default 2e9).  Affects launches enqueued after the call.  Returns the
 * previous value.
 */
GBATTN_API uint64_t attn_set_watchdog_ns(uint64_t ns);

/*
 * Self-test of the watchdog: enqueues one kernel that waits on a barrier
 * nothing ever arrives on, with the current watchdog limit; the kernel gives
 * up, records ATTN_ERR_TIMEOUT in the device error word and returns.  No
 * fault, trap or hang is involved.
 */
GBATTN_API attn_status attn_watchdog_selftest(attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_H_ */
