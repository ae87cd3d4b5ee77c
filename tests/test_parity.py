"""GPU parity of the CUDA library against the float64 oracle, through the C
ABI (via the ctypes binding), on the pages' workloads and on edge cases."""
import math

import numpy as np
import pytest
import torch

import scaled_dot_product_03_gb300 as gb
from scaled_dot_product_03_gb300 import inputs
from gpu_helpers import (GRAD_FLOOR, check_bwd, check_fwd, kw, lse_rows, rows_of, run_bwd,
                         run_fwd, sample_keys, sample_rows)
from helpers import oracle_fwd, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dev(prob):
    return prob.to(DEV)


def _sync_ok():
    torch.cuda.synchronize()
    gb.check_device_error()


# ---------------------------------------------------------------- workloads

def test_pr1_fp16_mqa_causal():
    prob = inputs.pr1()
    o, lse = run_fwd(_dev(prob))
    _sync_ok()
    check_fwd(prob, o, lse)


@pytest.mark.parametrize("scale", [1.0, 0.1])
def test_page1_packed_views_equal_contiguous_and_oracle(scale):
    prob = inputs.page1(scale=scale)
    d = _dev(prob)
    assert d.q.stride() == (1152, 1152, 64, 1)
    o, lse = run_fwd(d)
    qc, kc, vc = (t.contiguous() for t in (d.q, d.k, d.v))
    oc, lsec = gb.attn_fwd(qc, kc, vc, **kw(d))
    _sync_ok()
    # same kernel, same tiles, same arithmetic: bitwise equal
    assert torch.equal(o, oc) and torch.equal(lse, lsec)
    check_fwd(prob, o, lse)


@pytest.mark.parametrize("scale,det", [(1.0, False), (0.1, False), (0.1, True)])
def test_page1_mqa_backward_full_size_sampled(scale, det):
    """The page-1 workload (fp16, S=2048, 16 query heads over one KV head,
    packed strided views) through the backward at full size: the single pass
    splits the 16 query heads of the group over CTAs and sums their fp32
    dK / dV partials.  Sampled rows (dq) and keys (dk, dv, which sum over all
    16 heads) against the oracle."""
    prob = inputs.page1(scale=scale, dout_seed=5)
    d = _dev(prob)
    o, lse = run_fwd(d)
    dq, dk, dv = run_bwd(d, o, lse, deterministic=det)
    _sync_ok()
    rows = sample_rows(prob, 48, seed=7)
    check_fwd(prob, o, lse, row_sel=rows)
    keys = sample_keys(prob, [(0, 0)], 64, seed=7)
    check_bwd(prob, dq, dk, dv, row_sel=rows, key_sel=keys)


def test_mqa_d128_backward_sampled():
    """Multi-query attention at head dim 128 (16 query heads over one KV
    head, B=2, S=4096): the query-head split of the single pass at D=128."""
    prob = inputs.dense(2, 4096, 16, 128, Hkv=1, seed=13, dout_seed=14)
    d = _dev(prob)
    o, lse = run_fwd(d)
    dq, dk, dv = run_bwd(d, o, lse)
    _sync_ok()
    rows = sample_rows(prob, 24, seed=13)
    check_fwd(prob, o, lse, row_sel=rows)
    keys = sample_keys(prob, [(0, 0), (1, 0)], 24, seed=13)
    check_bwd(prob, dq, dk, dv, row_sel=rows, key_sel=keys)


def test_split_and_unsplit_backward_agree_bitwise_on_dkdv():
    """dK and dV of the split single pass are sums of per-split partials in a
    fixed order, so repeated runs give bitwise equal dK and dV."""
    prob = inputs.dense(1, 1000, 8, 64, Hkv=1, seed=17, dout_seed=18)
    d = _dev(prob)
    o, lse = run_fwd(d)
    a = run_bwd(d, o, lse)
    b = run_bwd(d, o, lse)
    _sync_ok()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    check_bwd(prob, *a)


def test_page3_fp32_forward_backward():
    prob = inputs.page3()
    d = _dev(prob)
    o, lse = run_fwd(d)
    dq, dk, dv = run_bwd(d, o, lse)
    _sync_ok()
    check_fwd(prob, o, lse)
    check_bwd(prob, dq, dk, dv)


def test_page3_local_global_merge_equals_causal():
    """Sliding-window-causal (band 64) over all rows, causal over the query
    rows shifted by 65 (keys with q - kv > 64), merged by LSE on the shifted
    rows: equals full causal attention (GPU vs GPU and vs oracle)."""
    prob = inputs.page3()
    d = _dev(prob)
    band = 64
    o_loc, l_loc = gb.attn_fwd(d.q, d.k, d.v, scale=d.scale, window=(band, 0))
    qg = d.q[:, band + 1:]
    o_glb, l_glb = gb.attn_fwd(qg, d.k, d.v, scale=d.scale, window=(-1, 0))
    o_m, l_m = gb.attn_merge_lse(o_loc[:, band + 1:], l_loc[:, :, band + 1:].contiguous(),
                                 o_glb, l_glb)
    o = torch.cat([o_loc[:, :band + 1], o_m], dim=1)
    lse = torch.cat([l_loc[:, :, :band + 1], l_m], dim=2)
    o_full, l_full = gb.attn_fwd(d.q, d.k, d.v, scale=d.scale, window=(-1, 0))
    _sync_ok()
    causal = inputs.page3()
    causal.window = (-1, 0)
    check_fwd(causal, o, lse)
    check_fwd(causal, o_full, l_full)
    assert float((o - o_full).abs().max()) <= 1e-4


def test_dense_bf16_s1024_d64_fwd_bwd():
    prob = inputs.dense(8, 1024, 16, 64)
    d = _dev(prob)
    o, lse = run_fwd(d)
    dq, dk, dv = run_bwd(d, o, lse)
    _sync_ok()
    check_fwd(prob, o, lse)
    check_bwd(prob, dq, dk, dv)


@pytest.mark.parametrize("S,det", [(1024, False), (2048, False), (4096, False), (8192, False),
                                   (16384, False), (4096, True)])
def test_dense_bf16_sweep_d128_sampled(S, det):
    """16384 tokens per batch at head dim 128, the bench's launch shapes;
    compared on sampled rows (O, LSE, dq) and on the keys of two (batch, kv
    head) units (dk, dv).  det: the bitwise-reproducible backward."""
    prob = inputs.dense(16384 // S, S, 16, 128)
    d = _dev(prob)
    o, lse = run_fwd(d)
    dq, dk, dv = run_bwd(d, o, lse, deterministic=det)
    _sync_ok()
    rows = sample_rows(prob, 48, seed=S)
    check_fwd(prob, o, lse, row_sel=rows)
    units = [(0, 0), (prob.B - 1, prob.Hkv - 1)]
    keys = sample_keys(prob, units, 24, seed=S)
    check_bwd(prob, dq, dk, dv, row_sel=rows, key_sel=keys)


@pytest.mark.parametrize("window,det", [((1023, 0), False), ((1023, 0), True), ((255, 255), False)])
def test_sliding_window_s16384_sampled(window, det):
    """A local band over a long sequence (B1 S16384 H16 D128, the bench's
    sliding-window workload, and a two-sided band): most key blocks of a
    query tile are skipped, the band's edges are masked inside blocks.
    Sampled rows and keys include the first and last of the sequence."""
    prob = inputs.dense(1, 16384, 16, 128, window=window, seed=3, dout_seed=4)
    d = _dev(prob)
    o, lse = run_fwd(d)
    dq, dk, dv = run_bwd(d, o, lse, deterministic=det)
    _sync_ok()
    rows = sample_rows(prob, 48, seed=11)
    check_fwd(prob, o, lse, row_sel=rows)
    keys = sample_keys(prob, [(0, 0), (0, prob.Hkv - 1)], 24, seed=11)
    check_bwd(prob, dq, dk, dv, row_sel=rows, key_sel=keys)


@pytest.mark.parametrize("det", [False, True])
def test_varlen_thd_gqa_fwd_bwd_sampled(det):
    prob = inputs.varlen()
    d = _dev(prob)
    o, lse = run_fwd(d)
    dq, dk, dv = run_bwd(d, o, lse, deterministic=det)
    _sync_ok()
    rows = sample_rows(prob, 64)
    check_fwd(prob, o, lse, row_sel=rows)
    keys = sample_keys(prob, [(0, 0), (7, 3), (15, 7)], 24)
    check_bwd(prob, dq, dk, dv, row_sel=rows, key_sel=keys)


@pytest.mark.parametrize("window,dtype", [((-1, 0), torch.bfloat16), ((-1, -1), torch.float16),
                                          ((63, 0), torch.bfloat16)])
def test_d64_many_short_items_sampled(window, dtype):
    """Head dim 64 at S=256 over 32 sequences and 16 heads: 1024 key tiles of
    one or two query blocks each, several per CTA of the persistent single
    pass (the next tile's loads and first products overlap the current
    one's last), causal, full and a narrow band."""
    prob = inputs.dense(32, 256, 16, 64, dtype=dtype, window=window, seed=11, dout_seed=12)
    d = _dev(prob)
    o, lse = run_fwd(d)
    dq, dk, dv = run_bwd(d, o, lse)
    _sync_ok()
    rows = sample_rows(prob, 16, seed=5)
    check_fwd(prob, o, lse, row_sel=rows)
    keys = sample_keys(prob, [(0, 0), (13, 7), (31, 15)], 32, seed=6)
    check_bwd(prob, dq, dk, dv, row_sel=rows, key_sel=keys)


def test_d64_thd_mixed_lengths_sampled():
    """Packed THD at head dim 64, 40 sequences of 1 to 700 tokens (GQA 4:1):
    the key tiles past a short sequence's end are items without rows, those
    that no query sees have zero gradients, and the others vary from one to
    six blocks per query head."""
    prob = inputs.varlen(nseq=40, min_len=1, max_len=700, Hq=8, Hkv=2, D=64, len_seed=7, seed=8,
                         dout_seed=9)
    d = _dev(prob)
    o, lse = run_fwd(d)
    dq, dk, dv = run_bwd(d, o, lse)
    _sync_ok()
    rows = sample_rows(prob, 48, seed=3)
    check_fwd(prob, o, lse, row_sel=rows)
    keys = sample_keys(prob, [(0, 0), (17, 1), (39, 1)], 24, seed=4)
    check_bwd(prob, dq, dk, dv, row_sel=rows, key_sel=keys)


# ---------------------------------------------------------------- edge cases

# (dtype, D, deterministic): the 16-bit backward at D=64 and 128 has a
# single-pass and a two-kernel (bitwise reproducible) form; fp32 has one.
_EDGE_KINDS = [(torch.float16, 64, False), (torch.bfloat16, 64, False), (torch.float32, 64, False),
               (torch.bfloat16, 64, True),
               (torch.float16, 128, False), (torch.bfloat16, 128, False),
               (torch.float32, 128, False), (torch.float16, 128, True),
               (torch.bfloat16, 128, True)]


@pytest.mark.parametrize("dtype,D,det", _EDGE_KINDS)
@pytest.mark.parametrize("case", [
    dict(B=2, Sq=1, Skv=1, Hq=2, Hkv=1, window=(-1, 0)),
    dict(B=1, Sq=17, Skv=17, Hq=3, Hkv=3, window=(-1, -1)),
    dict(B=2, Sq=129, Skv=129, Hq=4, Hkv=2, window=(-1, 0)),
    dict(B=1, Sq=200, Skv=77, Hq=2, Hkv=1, window=(-1, 0)),     # Sq > Skv, top-left
    dict(B=1, Sq=70, Skv=300, Hq=2, Hkv=2, window=(-1, 0)),     # Sq < Skv
    dict(B=1, Sq=300, Skv=300, Hq=4, Hkv=1, window=(40, 0)),    # sliding window
    dict(B=1, Sq=260, Skv=260, Hq=2, Hkv=1, window=(5, 37)),    # two-sided window
    dict(B=1, Sq=150, Skv=90, Hq=2, Hkv=1, window=(0, 0)),      # rows >= 90 see nothing
])
def test_edge_shapes_fwd_bwd(dtype, D, det, case):
    prob = inputs.dense(case["B"], case["Sq"], case["Hq"], D, dtype=dtype,
                        window=case["window"], Hkv=case["Hkv"], Skv=case["Skv"],
                        seed=case["Sq"] + D)
    d = _dev(prob)
    o, lse = run_fwd(d)
    dq, dk, dv = run_bwd(d, o, lse, deterministic=det)
    _sync_ok()
    check_fwd(prob, o, lse)
    check_bwd(prob, dq, dk, dv)


@pytest.mark.parametrize("order", ["sbhd", "bhsd"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_layouts_equal_bshd(order, dtype):
    """The same values stored as sbhd or bhsd give bitwise the same results
    as bshd (strides are resolved by the kernels, never by copies)."""
    a = inputs.random_case(5, B=2, Sq=192, Hq=4, Hkv=2, D=64, dtype=dtype, order="bshd")
    b = inputs.random_case(5, B=2, Sq=192, Hq=4, Hkv=2, D=64, dtype=dtype, order=order)
    da, db = _dev(a), _dev(b)
    assert torch.equal(da.q, db.q) and da.q.stride() != db.q.stride()
    oa, la = run_fwd(da)
    ob, lb = run_fwd(db)
    ga = run_bwd(da, oa, la)
    gbb = run_bwd(db, ob, lb)
    _sync_ok()
    assert torch.equal(oa, ob) and torch.equal(la, lb)
    for x, y in zip(ga, gbb):
        assert torch.allclose(x.float(), y.float(), atol=0, rtol=0) or \
            float((x.float() - y.float()).abs().max()) <= 2e-2 * float(x.float().abs().max())
    check_fwd(a, oa, la)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_thd_with_empty_and_single_token_sequences(dtype):
    prob = inputs.varlen(lengths=[1, 0, 129, 64, 300, 7], Hq=4, Hkv=2, D=64, dtype=dtype)
    d = _dev(prob)
    o, lse = run_fwd(d)
    dq, dk, dv = run_bwd(d, o, lse)
    _sync_ok()
    check_fwd(prob, o, lse)
    check_bwd(prob, dq, dk, dv)


def test_thd_equals_dense_per_sequence():
    """A THD pack gives, per sequence, exactly what the dense path gives for
    that sequence alone (batch independence)."""
    prob = inputs.varlen(lengths=[130, 257, 64], Hq=4, Hkv=2, D=128)
    d = _dev(prob)
    o, lse = run_fwd(d)
    cu = prob.cu_seqlens_q.tolist()
    for b in range(3):
        a, e = cu[b], cu[b + 1]
        ob, lb = gb.attn_fwd(d.q[a:e][None], d.k[a:e][None], d.v[a:e][None],
                             scale=d.scale, window=d.window)
        assert torch.equal(ob[0], o[a:e])
        assert torch.equal(lb[0], lse[:, a:e])
    _sync_ok()


def test_forward_is_deterministic():
    prob = inputs.dense(2, 1000, 8, 128)
    d = _dev(prob)
    o1, l1 = run_fwd(d)
    o2, l2 = run_fwd(d)
    _sync_ok()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_backward_reproducibility():
    """deterministic=True: bitwise equal on repeated runs.  Default single
    pass: dk and dv (owned by one CTA each) bitwise equal, dq (fp32 sums in
    scheduling order) equal to within fp32 rounding of the sums, and both
    modes agree to the same precision."""
    prob = inputs.dense(2, 1000, 8, 128, Hkv=2, seed=31, dout_seed=32)
    d = _dev(prob)
    o, lse = run_fwd(d)
    r1 = run_bwd(d, o, lse, deterministic=True)
    r2 = run_bwd(d, o, lse, deterministic=True)
    f1 = run_bwd(d, o, lse)
    f2 = run_bwd(d, o, lse)
    _sync_ok()
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)
    assert torch.equal(f1[1], f2[1]) and torch.equal(f1[2], f2[2])
    for a, b in ((f1[0], f2[0]), (f1[0], r1[0]), (f1[1], r1[1]), (f1[2], r1[2])):
        a64, b64 = a.double(), b.double()
        scale = max(float(b64.abs().max()), GRAD_FLOOR)
        assert float((a64 - b64).abs().max()) <= 1e-2 * scale


def test_packed_gradient_buffer_views():
    """dq, dk, dv written into split views of one packed gradient buffer
    (the layout of the page-1 inputs) match separate buffers."""
    prob = inputs.page1(scale=0.1, seqlen=512)
    d = _dev(prob)
    dout = torch.randn(d.q.shape, generator=torch.Generator().manual_seed(3)).half().to(DEV)
    o, lse = gb.attn_fwd(d.q, d.k, d.v, scale=0.1, window=(-1, 0))
    g = torch.zeros_like(d.bases["qkv"])
    gq, gk, gv = g.split([16, 1, 1], dim=2)
    gq, gk, gv = (t.permute(1, 0, 2, 3) for t in (gq, gk, gv))
    gb.attn_bwd(dout, d.q, d.k, d.v, o, lse, scale=0.1, window=(-1, 0), dq=gq, dk=gk, dv=gv,
                deterministic=True)
    dq, dk, dv = gb.attn_bwd(dout, d.q, d.k, d.v, o, lse, scale=0.1, window=(-1, 0),
                             deterministic=True)
    _sync_ok()
    assert torch.equal(gq, dq) and torch.equal(gk, dk) and torch.equal(gv, dv)


# ---------------------------------------------------------------- merge

@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_merge_matches_oracle_with_empty_sides(dtype):
    import oracle
    g = torch.Generator().manual_seed(9)
    B, S, H, D = 2, 100, 3, 128
    o1 = torch.randn(B, S, H, D, generator=g).to(dtype)
    o2 = torch.randn(B, S, H, D, generator=g).to(dtype)
    l1 = torch.randn(B, H, S, generator=g) * 3
    l2 = torch.randn(B, H, S, generator=g) * 3
    l1[0, 0, :10] = -math.inf
    l2[0, 0, 5:15] = -math.inf
    o, l = gb.attn_merge_lse(o1.to(DEV), l1.to(DEV), o2.to(DEV), l2.to(DEV))
    _sync_ok()
    t = lambda x: to_f64(x).transpose(0, 2, 1, 3) if x.dim() == 4 else to_f64(x)
    ro, rl = oracle.merge_lse(t(o1), t(l1), t(o2), t(l2))
    tol = {torch.float16: 5e-3, torch.bfloat16: 1e-2, torch.float32: 1e-5}[dtype]
    assert np.abs(t(o) - ro).max() <= tol
    fin = np.isfinite(rl)
    assert np.all(np.isneginf(to_f64(l))[~fin])
    assert np.abs(to_f64(l)[fin] - rl[fin]).max() <= 1e-5


def test_merge_in_place_and_thd():
    g = torch.Generator().manual_seed(11)
    T, H, D = 333, 4, 64
    o1 = torch.randn(T, H, D, generator=g).bfloat16().to(DEV)
    o2 = torch.randn(T, H, D, generator=g).bfloat16().to(DEV)
    l1 = torch.randn(H, T, generator=g).to(DEV)
    l2 = torch.randn(H, T, generator=g).to(DEV)
    ref_o, ref_l = gb.attn_merge_lse(o1, l1, o2, l2)
    gb.attn_merge_lse(o1, l1, o2, l2, out=o1, lse_out=l1)
    _sync_ok()
    assert torch.equal(o1, ref_o) and torch.equal(l1, ref_l)


# ---------------------------------------------------------------- watchdog

def test_watchdog_gives_up_and_reports():
    """A wait on a barrier nothing arrives on ends after the limit with an
    error the host reads; the context stays usable."""
    old = gb.set_watchdog_ns(2_000_000)  # 2 ms
    try:
        gb.watchdog_selftest()
        with pytest.raises(gb.AttnError) as ei:
            gb.check_device_error()
        assert ei.value.status == 4
    finally:
        gb.set_watchdog_ns(old)
    gb.check_device_error()  # cleared
    prob = inputs.pr1()
    o, lse = run_fwd(_dev(prob))
    _sync_ok()
    check_fwd(prob, o, lse)


# ----------------------------------------------- reported argument errors

@pytest.mark.parametrize("which,det", [("q", False), ("kv", False), ("kv", True), ("q", True)])
def test_thd_understated_max_seqlen_is_reported(which, det):
    """THD grids are sized from max_seqlen_q / max_seqlen_kv.  A call that
    understates one of them (here 200 for sequences of 300 and 517 rows)
    cannot cover the longer sequences; the kernel of each sequence's last
    grid tile reports that, and attn_check_device_error returns
    INVALID_ARG.  Every address still comes from cu_seqlens, so the call
    reads and writes only inside the tensors.  The forward misses query rows
    (max_seqlen_q); the backward misses key tiles (max_seqlen_kv), and its
    two-kernel form also query rows."""
    prob = inputs.varlen(lengths=[300, 64, 517], Hq=4, Hkv=2, D=128, seed=71, dout_seed=72)
    d = _dev(prob)
    good = kw(d)
    bad = dict(good, **{"max_seqlen_" + which: 200})
    if which == "q":
        gb.attn_fwd(d.q, d.k, d.v, **bad)
    else:
        o, lse = gb.attn_fwd(d.q, d.k, d.v, **good)
        _sync_ok()
        gb.attn_bwd(d.dout, d.q, d.k, d.v, o, lse, deterministic=det, **bad)
    torch.cuda.synchronize()
    with pytest.raises(gb.AttnError) as ei:
        gb.check_device_error()
    assert ei.value.status == 1, str(ei.value)
    assert "max_seqlen_" + which in str(ei.value)
    gb.check_device_error()  # cleared
    o, lse = run_fwd(d)      # and the next correct call is unaffected
    _sync_ok()
    check_fwd(prob, o, lse)


def test_calls_on_a_non_default_current_stream():
    """The binding launches on torch's current stream of the tensors'
    device, here a side stream."""
    prob = inputs.dense(2, 300, 4, 128, Hkv=2, seed=61, dout_seed=62)
    d = _dev(prob)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        o, lse = run_fwd(d)
        dq, dk, dv = run_bwd(d, o, lse)
    side.synchronize()
    _sync_ok()
    check_fwd(prob, o, lse)
    check_bwd(prob, dq, dk, dv)


# ------------------------------------------------------- padded cu_seqlens

@pytest.mark.parametrize("dtype,D,det", [(torch.bfloat16, 128, False), (torch.bfloat16, 128, True),
                                         (torch.float16, 64, False), (torch.float32, 64, False)])
def test_thd_padded_cu_seqlens(dtype, D, det):
    """THD buffers with padding between sequences (cu_seqlens_*_padded of the
    THD+CP thread): sequence b occupies rows [pad[b], pad[b] + L_b).  Outputs
    on the sequence rows equal the unpadded problem's oracle; rows in the
    gaps (finite filler) are never written."""
    lengths = [300, 1, 517, 64, 0, 129]
    prob = inputs.varlen(lengths=lengths, Hq=4, Hkv=2, D=D, dtype=dtype, seed=41, dout_seed=42)
    cu_h = [0]
    for L in lengths:
        cu_h.append(cu_h[-1] + L)
    pads = [0]
    for L in lengths:  # each sequence rounded up to 64 rows, plus 7
        pads.append(pads[-1] + (L + 63) // 64 * 64 + 7)
    Tp = pads[-1]

    def scatter(t, fill):
        out = torch.full((Tp,) + tuple(t.shape[1:]), fill, dtype=t.dtype)
        for b, L in enumerate(lengths):
            out[pads[b]:pads[b] + L] = t[cu_h[b]:cu_h[b] + L]
        return out.to(DEV)

    def gather(t):
        return torch.cat([t[pads[b]:pads[b] + L] for b, L in enumerate(lengths)])

    q, k, v, dout = (scatter(getattr(prob, n), 0.5) for n in ("q", "k", "v", "dout"))
    cu_d = torch.tensor(cu_h, dtype=torch.int32, device=DEV)
    pad_d = torch.tensor(pads, dtype=torch.int32, device=DEV)
    sentinel = 7.0
    o = torch.full_like(q, sentinel)
    lse = torch.full((prob.Hq, Tp), sentinel, dtype=torch.float32, device=DEV)
    dq, dk, dv = (torch.full_like(t, sentinel) for t in (q, k, v))
    args = dict(scale=prob.scale, window=prob.window, cu_seqlens_q=cu_d, cu_seqlens_kv=cu_d,
                max_seqlen_q=max(lengths), max_seqlen_kv=max(lengths),
                cu_seqlens_q_padded=pad_d, cu_seqlens_kv_padded=pad_d)
    gb.attn_fwd(q, k, v, out=o, lse=lse, **args)
    gb.attn_bwd(dout, q, k, v, o, lse, dq=dq, dk=dk, dv=dv, deterministic=det, **args)
    _sync_ok()
    rows = torch.cat([torch.arange(pads[b], pads[b] + L) for b, L in enumerate(lengths)])
    check_fwd(prob, gather(o), lse[:, rows.to(DEV)])
    check_bwd(prob, gather(dq), gather(dk), gather(dv))
    gap = torch.ones(Tp, dtype=torch.bool)
    gap[rows] = False
    gap = gap.to(DEV)
    for t in (o, dq, dk, dv):
        assert torch.all(t[gap] == sentinel)
    assert torch.all(lse[:, gap] == sentinel)


def test_cross_attention_few_queries_many_keys():
    """Cross attention of a few decoder positions over a long encoder
    sequence (the RETURNN pull request's seqlen_kv, beam-search shapes):
    Sq = 7, Skv = 1024, no mask, grouped heads."""
    prob = inputs.dense(3, 7, 8, 128, Hkv=2, Skv=1024, window=(-1, -1), seed=51, dout_seed=52)
    d = _dev(prob)
    o, lse = run_fwd(d)
    dq, dk, dv = run_bwd(d, o, lse)
    _sync_ok()
    check_fwd(prob, o, lse)
    check_bwd(prob, dq, dk, dv)


# -------------------------------------------------------- other head dims

@pytest.mark.parametrize("dtype,det", [(torch.float16, False), (torch.bfloat16, False),
                                       (torch.bfloat16, True), (torch.float32, False)])
@pytest.mark.parametrize("D", [32, 96])
@pytest.mark.parametrize("case", [
    dict(B=2, Sq=150, Skv=150, Hq=4, Hkv=2, window=(-1, 0)),
    dict(B=1, Sq=70, Skv=201, Hq=2, Hkv=1, window=(-1, -1)),
    dict(B=1, Sq=260, Skv=260, Hq=2, Hkv=2, window=(17, 3)),
    dict(B=2, Sq=700, Skv=700, Hq=8, Hkv=8, window=(-1, 0)),
])
def test_head_dims_32_and_96(dtype, D, det, case):
    """Head dims 32 and 96: fp16 / bf16 on the 64- and 128-wide tensor-core
    kernels with zero-padded columns (single pass and two-kernel backward),
    fp32 on the FFMA kernels."""
    prob = inputs.dense(case["B"], case["Sq"], case["Hq"], D, dtype=dtype, window=case["window"],
                        Hkv=case["Hkv"], Skv=case["Skv"], seed=D + case["Sq"])
    d = _dev(prob)
    o, lse = run_fwd(d)
    dq, dk, dv = run_bwd(d, o, lse, deterministic=det)
    _sync_ok()
    check_fwd(prob, o, lse)
    check_bwd(prob, dq, dk, dv)


@pytest.mark.parametrize("D,det", [(32, False), (96, False), (96, True)])
def test_head_dims_32_96_thd_padded_and_split(D, det):
    """Padded head dims with THD (row-by-row stores of partial tiles), padded
    cu_seqlens and grouped heads on a small grid (query-head split)."""
    lengths = [300, 1, 517, 64, 0, 129]
    prob = inputs.varlen(lengths=lengths, Hq=4, Hkv=1, D=D, dtype=torch.bfloat16, seed=D, dout_seed=D + 1)
    d = _dev(prob)
    o, lse = run_fwd(d)
    dq, dk, dv = run_bwd(d, o, lse, deterministic=det)
    _sync_ok()
    check_fwd(prob, o, lse)
    check_bwd(prob, dq, dk, dv)


@pytest.mark.parametrize("D", [32, 96])
def test_head_dims_32_96_strided_views_equal_contiguous(D):
    """A packed sb(h+2h_g)d buffer split into q, k, v views (the page-1
    layout) at the padded head dims: the same results as contiguous copies."""
    prob = inputs.page1(scale=0.1, seqlen=384, q_heads=4, kv_heads=2, head_dim=D, dout_seed=9)
    d = _dev(prob)
    o, lse = run_fwd(d)
    qc, kc, vc = (t.contiguous() for t in (d.q, d.k, d.v))
    oc, lsec = gb.attn_fwd(qc, kc, vc, **kw(d))
    _sync_ok()
    assert torch.equal(o, oc) and torch.equal(lse, lsec)
    check_fwd(prob, o, lse)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("case", [
    dict(B=2, Sq=300, Skv=300, Hq=4, Hkv=2, window=(-1, 0)),
    dict(B=1, Sq=70, Skv=201, Hq=2, Hkv=1, window=(-1, -1)),
    dict(B=1, Sq=520, Skv=520, Hq=2, Hkv=2, window=(40, 3)),
    dict(B=1, Sq=150, Skv=90, Hq=2, Hkv=1, window=(0, 0)),
])
def test_head_dim_256_forward(dtype, case):
    """Head dim 256 (forward only): one query tile per CTA, S and O of the
    tile in TMEM, N = 256 for O += P V."""
    prob = inputs.dense(case["B"], case["Sq"], case["Hq"], 256, dtype=dtype, window=case["window"],
                        Hkv=case["Hkv"], Skv=case["Skv"], seed=256 + case["Sq"], dout_seed=None)
    o, lse = run_fwd(_dev(prob))
    _sync_ok()
    check_fwd(prob, o, lse)


def test_head_dim_256_forward_thd_and_full_size_sampled():
    """Head dim 256 with THD (row-by-row stores of partial tiles) and at a
    long causal sequence, on sampled rows."""
    prob = inputs.varlen(lengths=[300, 1, 517, 64, 0, 129], Hq=4, Hkv=2, D=256, seed=2, dout_seed=None)
    o, lse = run_fwd(_dev(prob))
    _sync_ok()
    check_fwd(prob, o, lse)
    prob = inputs.dense(1, 8192, 8, 256, seed=4, dout_seed=None)
    o, lse = run_fwd(_dev(prob))
    _sync_ok()
    check_fwd(prob, o, lse, row_sel=sample_rows(prob, 48, seed=4))


# ------------------------------------------------------ randomized shapes

def _random_cases(n, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for k in range(n):
        dtype = [torch.float16, torch.bfloat16][k % 2]
        D = [64, 128, 32, 96][(k // 2) % 4]
        Hkv = int(rng.choice([1, 2, 4]))
        Hq = Hkv * int(rng.choice([1, 2, 3]))
        window = [(-1, 0), (-1, -1), (int(rng.integers(0, 200)), 0),
                  (int(rng.integers(0, 90)), int(rng.integers(0, 90)))][int(rng.integers(0, 4))]
        det = bool(rng.integers(0, 2))
        if k % 3 == 2:   # THD
            lengths = [int(x) for x in rng.integers(0, 400, size=int(rng.integers(1, 5)))]
            cases.append(("thd", dict(lengths=lengths, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype, window=window,
                                      seed=k, dout_seed=k + 100), det))
        else:
            B = int(rng.integers(1, 4))
            Sq = int(rng.integers(1, 520))
            Skv = Sq if rng.random() < 0.6 else int(rng.integers(1, 520))
            cases.append(("dense", dict(B=B, S=Sq, H=Hq, D=D, dtype=dtype, window=window, Hkv=Hkv,
                                        Skv=Skv, seed=k, dout_seed=k + 100), det))
    return cases


@pytest.mark.parametrize("layout,args,det", _random_cases(32))
def test_randomized_configs(layout, args, det):
    """Seeded random shapes across dtypes, head dims, layouts, grouped heads,
    windows and both backward forms, against the oracle."""
    prob = inputs.varlen(**args) if layout == "thd" else inputs.dense(**args)
    d = _dev(prob)
    o, lse = run_fwd(d)
    dq, dk, dv = run_bwd(d, o, lse, deterministic=det)
    _sync_ok()
    check_fwd(prob, o, lse)
    check_bwd(prob, dq, dk, dv)
