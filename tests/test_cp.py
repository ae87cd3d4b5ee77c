"""Context parallelism over THD batches (the THD+CP thread), emulated on
one GPU: the library's partition of a padded buffer is the oracle's, bit
for bit; the ring of partial attentions merged by LSE equals one attention
over the whole batch (library and oracle), and so do the gradients of its
backward (per-pair backward with the merged O and LSE, shares summed)."""
import numpy as np
import pytest
import torch

import oracle
import scaled_dot_product_03_gb300 as gb
from scaled_dot_product_03_gb300 import cp
from gpu_helpers import LSE_TOL, O_TOL

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _padded(lengths, multiple):
    pads = [0]
    for L in lengths:
        pads.append(pads[-1] + -(-max(L, 1) // multiple) * multiple)
    return pads


@pytest.mark.parametrize("world", [1, 2, 4, 8])
def test_partitioned_indices_match_oracle(world):
    lengths = [513, 1, 64, 0, 4000, 77]
    pads = _padded(lengths, 2 * world)
    pad_d = torch.tensor(pads, dtype=torch.int32, device=DEV)
    for rank in range(world):
        got = cp.thd_get_partitioned_indices(pad_d, pads[-1], world, rank)
        torch.cuda.synchronize()
        ref = oracle.thd_partitioned_indices(pads, pads[-1], world, rank)
        np.testing.assert_array_equal(got.cpu().numpy().astype(np.int64), ref)


@pytest.mark.parametrize("dtype,D,Hq,Hkv", [(torch.bfloat16, 128, 8, 2), (torch.float16, 64, 4, 4)])
@pytest.mark.parametrize("cp_size", [2, 4])
@pytest.mark.parametrize("causal", [True, False])
def test_ring_attention_matches_full(dtype, D, Hq, Hkv, cp_size, causal):
    lengths = [700, 1, 256, 0, 333]
    pads = _padded(lengths, 2 * cp_size)
    T = pads[-1]
    g = torch.Generator().manual_seed(17)
    # finite filler in the padding rows (they meet zero weights)
    q = torch.randn(T, Hq, D, generator=g).to(dtype)
    k = torch.randn(T, Hkv, D, generator=g).to(dtype)
    v = torch.randn(T, Hkv, D, generator=g).to(dtype)
    cu_h = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    cu_d = torch.tensor(cu_h, device=DEV)
    pad_d = torch.tensor(pads, dtype=torch.int32, device=DEV)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    scale = D ** -0.5
    window = (-1, 0) if causal else (-1, -1)
    o, lse = cp.ring_attention_fwd(qd, kd, vd, cu_d, pad_d, cp_size, causal=causal, scale=scale)
    o_full, lse_full = gb.attn_fwd(qd, kd, vd, scale=scale, window=window, cu_seqlens_q=cu_d,
                                   cu_seqlens_kv=cu_d, max_seqlen_q=max(lengths),
                                   max_seqlen_kv=max(lengths), cu_seqlens_q_padded=pad_d,
                                   cu_seqlens_kv_padded=pad_d)
    torch.cuda.synchronize()
    gb.check_device_error()
    rows = np.concatenate([np.arange(pads[b], pads[b] + L) for b, L in enumerate(lengths)])
    rows_d = torch.tensor(rows, device=DEV)
    ro, rl = oracle.attn_fwd(q.double().numpy()[rows], k.double().numpy()[rows],
                             v.double().numpy()[rows], cu_h, cu_h, scale, window)
    go = o[rows_d].double().cpu().numpy()
    gl = lse[:, rows_d].T.double().cpu().numpy()
    assert np.abs(go - ro).max() <= O_TOL[dtype]
    assert np.abs(gl - rl).max() <= LSE_TOL[dtype]
    # the ring and the single call agree to within their own rounding
    assert float((o[rows_d] - o_full[rows_d]).abs().max()) <= O_TOL[dtype]
    pad_rows = torch.tensor(np.setdiff1d(np.arange(T), rows), device=DEV)
    assert torch.all(o[pad_rows] == 0) and torch.all(torch.isneginf(lse[:, pad_rows]))


def test_thd_row_sums_exact():
    """attn_thd_accumulate / attn_thd_store against the same fp32 arithmetic on
    the CPU (bf16 -> fp32 is exact and both round to nearest even): bit-exact,
    rows outside the sequences untouched by the sums and zeroed by the store."""
    lengths, pads = [5, 0, 17, 3], [0, 8, 8, 32, 40]
    T, H, D = pads[-1] + 4, 3, 64  # 4 tail rows past the last sequence
    g = torch.Generator().manual_seed(23)
    a = torch.randn(T, H, D, generator=g).bfloat16()
    b = torch.randn(T, H, D, generator=g).bfloat16()
    base = torch.randn(T, H, D, generator=g)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32), device=DEV)
    pad = torch.tensor(pads, dtype=torch.int32, device=DEV)
    acc = base.to(DEV)
    cp.thd_accumulate(a.to(DEV), acc, cu, pad, accumulate=False)
    cp.thd_accumulate(b.to(DEV), acc, cu, pad, accumulate=True)
    out = torch.full((T, H, D), 7.0).bfloat16().to(DEV)
    cp.thd_store(acc, out, cu, pad)
    torch.cuda.synchronize()
    inside = np.zeros(T, bool)
    for s0, L in zip(pads, lengths):
        inside[s0:s0 + L] = True
    ins = torch.tensor(inside)
    want = base.clone()
    want[ins] = a[ins].float() + b[ins].float()
    assert torch.equal(acc.cpu(), want)
    want_out = torch.zeros(T, H, D).bfloat16()
    want_out[ins] = want[ins].bfloat16()
    assert torch.equal(out.cpu(), want_out)


@pytest.mark.parametrize("dtype,D,Hq,Hkv", [(torch.bfloat16, 128, 8, 2), (torch.float16, 64, 4, 4)])
@pytest.mark.parametrize("cp_size", [2, 4])
@pytest.mark.parametrize("causal", [True, False])
def test_ring_attention_backward_matches_full(dtype, D, Hq, Hkv, cp_size, causal):
    """The ring's backward (every pair's attention backward with the merged O
    and LSE, shares summed in fp32) against the float64 gradients of one
    attention over the whole batch, and against the library's single call."""
    from gpu_helpers import GRAD_FLOOR, GRAD_REL
    lengths = [700, 1, 256, 0, 333]
    pads = _padded(lengths, 2 * cp_size)
    T = pads[-1]
    g = torch.Generator().manual_seed(29)
    q = torch.randn(T, Hq, D, generator=g).to(dtype)
    k = torch.randn(T, Hkv, D, generator=g).to(dtype)
    v = torch.randn(T, Hkv, D, generator=g).to(dtype)
    do = torch.randn(T, Hq, D, generator=g).to(dtype)
    cu_h = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    cu_d = torch.tensor(cu_h, device=DEV)
    pad_d = torch.tensor(pads, dtype=torch.int32, device=DEV)
    qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV)
    scale = D ** -0.5
    window = (-1, 0) if causal else (-1, -1)
    o, lse = cp.ring_attention_fwd(qd, kd, vd, cu_d, pad_d, cp_size, causal=causal, scale=scale)
    dq, dk, dv = cp.ring_attention_bwd(dod, qd, kd, vd, o, lse, cu_d, pad_d, cp_size, causal=causal,
                                       scale=scale)
    full = dict(scale=scale, window=window, cu_seqlens_q=cu_d, cu_seqlens_kv=cu_d, max_seqlen_q=max(lengths),
                max_seqlen_kv=max(lengths), cu_seqlens_q_padded=pad_d, cu_seqlens_kv_padded=pad_d)
    o1, l1 = gb.attn_fwd(qd, kd, vd, **full)
    s_dq, s_dk, s_dv = gb.attn_bwd(dod, qd, kd, vd, o1, l1, **full)
    torch.cuda.synchronize()
    gb.check_device_error()
    rows = np.concatenate([np.arange(pads[b], pads[b] + L) for b, L in enumerate(lengths)])
    rows_d = torch.tensor(rows, device=DEV)
    r = oracle.attn_bwd(q.double().numpy()[rows], k.double().numpy()[rows], v.double().numpy()[rows],
                        do.double().numpy()[rows], cu_h, cu_h, scale, window)
    for name, got, single, ref in (("dq", dq, s_dq, r[0]), ("dk", dk, s_dk, r[1]), ("dv", dv, s_dv, r[2])):
        tol = GRAD_REL * max(float(np.abs(ref).max()), GRAD_FLOOR)
        ga = got[rows_d].double().cpu().numpy()
        assert np.all(np.isfinite(ga)), name
        assert np.abs(ga - ref).max() <= tol, (name, np.abs(ga - ref).max(), tol)
        assert float((got[rows_d] - single[rows_d]).abs().max()) <= tol, name
    pad_rows = torch.tensor(np.setdiff1d(np.arange(T), rows), device=DEV)
    for t in (dq, dk, dv):
        assert torch.all(t[pad_rows] == 0)
