"""Context parallelism over THD batches (the THD+CP thread), emulated on
one GPU: the library's partition of a padded buffer is the oracle's, bit
for bit, and the ring of partial attentions merged by LSE equals one
attention over the whole batch (library and oracle)."""
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
