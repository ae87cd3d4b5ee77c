"""Context parallelism over THD batches, emulated on one GPU.

"[PyTorch] Add support for cuDNN FusedAttention + THD + CP": each sequence
is cut into 2 x CP chunks, rank r holds chunks r and 2 CP - 1 - r (load
balance under a causal mask), and K/V blocks travel around a ring of ranks;
every rank attends with its own queries to each block it receives and
combines the partial results by their LSE (the order of the ring does not
change the result).  ``ring_attention_fwd`` runs that schedule for all ranks
on one GPU: every (query chunk, key chunk) pair is one ``attn_fwd`` call on
the global buffers, addressed through padded cu_seqlens (chunk c of
sequence b starts at row pad[b] + c * len_b / (2 CP)), and every partial is
folded into its rank's rows with ``attn_merge_lse``.  Under a causal mask a
query chunk sees earlier key chunks in full, its own chunk causally, and
later chunks not at all.  ``ring_attention_bwd`` runs the backward of that
schedule: every pair's attention backward, called with the merged O and
LSE, gives the pair's share of dQ (rows of the query chunk) and of dK, dV
(rows of the key chunk), and each gradient is the fp32 sum of its shares
(``attn_thd_accumulate``), written out with ``attn_thd_store``.  All
arithmetic runs in the library's kernels; this module only plans the calls.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import torch

from . import _DTYPES, _device_of, _stream, _tensor, _lib, attn_bwd, attn_bwd_workspace_size, attn_fwd, attn_merge_lse


def thd_get_partitioned_indices(cu_seqlens_padded: torch.Tensor, total_tokens: int,
                                world_size: int, rank: int) -> torch.Tensor:
    """Rows (int32, on cu_seqlens_padded's device) of a padded THD buffer
    that ``rank`` holds: chunk ``rank`` then chunk ``2 * world_size - 1 -
    rank`` of every sequence (see attn_thd_partitioned_indices)."""
    assert cu_seqlens_padded.dtype == torch.int32 and cu_seqlens_padded.is_cuda
    out = torch.empty(total_tokens // world_size, dtype=torch.int32, device=cu_seqlens_padded.device)
    stream = torch.cuda.current_stream(cu_seqlens_padded.device).cuda_stream
    _lib.check(_lib.load().attn_thd_partitioned_indices(
        cu_seqlens_padded.data_ptr(), cu_seqlens_padded.numel() - 1, int(total_tokens),
        int(world_size), int(rank), out.data_ptr(), stream))
    return out


def ring_pairs(cp_size: int, rank: int, causal: bool) -> List[Tuple[int, int, int, bool]]:
    """The attention calls of ``rank`` in ring order: ``(step, q_chunk,
    kv_chunk, causal_mask)``; at step i the rank holds the K/V of rank
    (rank - i) mod cp_size."""
    n = 2 * cp_size
    own = (rank, n - 1 - rank)
    pairs = []
    for step in range(cp_size):
        src = (rank - step) % cp_size
        for cq in own:
            for ck in (src, n - 1 - src):
                if causal and ck > cq:
                    continue
                pairs.append((step, cq, ck, causal and ck == cq))
    return pairs


def _chunk_views(lengths: Sequence[int], pads: Sequence[int], cp_size: int, device):
    """cu_seqlens and padded starts (int32, device) of chunk c of every
    sequence, for c in 0 .. 2 cp_size - 1, and the longest chunk."""
    n = 2 * cp_size
    cus, starts = [], []
    longest = 0
    for c in range(n):
        cu, st = [0], []
        for b, L in enumerate(lengths):
            size = (pads[b + 1] - pads[b]) // n
            m = max(0, min(size, L - c * size))  # tokens of the chunk (padding excluded)
            cu.append(cu[-1] + m)
            st.append(pads[b] + c * size)
            longest = max(longest, m)
        st.append(pads[-1])
        cus.append(torch.tensor(cu, dtype=torch.int32, device=device))
        starts.append(torch.tensor(st, dtype=torch.int32, device=device))
    return cus, starts, longest


def ring_attention_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                       cu_seqlens: torch.Tensor, cu_seqlens_padded: torch.Tensor, cp_size: int,
                       *, causal: bool = True, scale: Optional[float] = None
                       ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Context-parallel attention of a padded THD batch (q, k, v ``[T, H, D]``,
    every padded length a multiple of ``2 * cp_size``), every rank's ring run
    on this GPU.  Returns ``(o [T, Hq, D], lse [Hq, T])`` in the buffer's row
    order, as one ``attn_fwd`` over the whole batch would (padding rows:
    o = 0, lse = -inf)."""
    lens = (cu_seqlens[1:] - cu_seqlens[:-1]).tolist()      # host copies of the
    pads = cu_seqlens_padded.tolist()                         # (small) offset arrays
    n = 2 * cp_size
    for b in range(len(lens)):
        assert (pads[b + 1] - pads[b]) % n == 0 and lens[b] <= pads[b + 1] - pads[b]
    cus, starts, longest = _chunk_views(lens, pads, cp_size, q.device)
    T, Hq = q.shape[0], q.shape[1]
    o = torch.zeros_like(q)
    lse = torch.full((Hq, T), float("-inf"), dtype=torch.float32, device=q.device)
    part_o = torch.empty_like(q)
    part_lse = torch.empty_like(lse)
    for rank in range(cp_size):
        for _, cq, ck, cmask in ring_pairs(cp_size, rank, causal):
            # the partial covers only chunk cq's rows; the rest stay (0, -inf)
            part_o.zero_()
            part_lse.fill_(float("-inf"))
            attn_fwd(q, k, v, scale=scale, window=(-1, 0) if cmask else (-1, -1),
                     cu_seqlens_q=cus[cq], cu_seqlens_kv=cus[ck], max_seqlen_q=longest,
                     max_seqlen_kv=longest, cu_seqlens_q_padded=starts[cq],
                     cu_seqlens_kv_padded=starts[ck], out=part_o, lse=part_lse)
            attn_merge_lse(o, lse, part_o, part_lse, out=o, lse_out=lse)
    return o, lse


def thd_accumulate(src: torch.Tensor, acc: torch.Tensor, cu_seqlens: torch.Tensor,
                   cu_seqlens_padded: Optional[torch.Tensor] = None, *, accumulate: bool = True) -> None:
    """acc (fp32 [T, H, D], contiguous) += src ([T, H, D] view, or = src when
    ``accumulate`` is False) on the rows inside the sequences (see
    attn_thd_accumulate)."""
    assert acc.dtype == torch.float32 and acc.is_contiguous() and acc.shape == src.shape
    T, H, D = src.shape
    pad = cu_seqlens_padded.data_ptr() if cu_seqlens_padded is not None else None
    with _device_of(src):
        _lib.check(_lib.load().attn_thd_accumulate(_DTYPES[src.dtype], T, H, D, _tensor(src, True), acc.data_ptr(),
                                                   1 if accumulate else 0, cu_seqlens.data_ptr(), pad,
                                                   cu_seqlens.numel() - 1, _stream(src)))


def thd_store(acc: torch.Tensor, dst: torch.Tensor, cu_seqlens: torch.Tensor,
              cu_seqlens_padded: Optional[torch.Tensor] = None) -> None:
    """dst ([T, H, D] view) = acc on the rows inside the sequences, 0 on the
    others (see attn_thd_store)."""
    assert acc.dtype == torch.float32 and acc.is_contiguous() and acc.shape == dst.shape
    T, H, D = dst.shape
    pad = cu_seqlens_padded.data_ptr() if cu_seqlens_padded is not None else None
    with _device_of(dst):
        _lib.check(_lib.load().attn_thd_store(_DTYPES[dst.dtype], T, H, D, acc.data_ptr(), _tensor(dst, True),
                                              cu_seqlens.data_ptr(), pad, cu_seqlens.numel() - 1, _stream(dst)))


def ring_attention_bwd(dout: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                       o: torch.Tensor, lse: torch.Tensor, cu_seqlens: torch.Tensor,
                       cu_seqlens_padded: torch.Tensor, cp_size: int, *, causal: bool = True,
                       scale: Optional[float] = None
                       ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Gradients ``(dq, dk, dv)`` of the context-parallel attention that
    ``ring_attention_fwd`` computes, every rank's ring run on this GPU: for
    each rank and ring step, the attention backward of the step's (query
    chunk, key chunk) pairs with the merged ``o`` and ``lse`` (so each
    recomputes its probabilities from the merged LSE and its row terms from
    the merged O), the shares summed in fp32.  Padding rows get 0."""
    lens = (cu_seqlens[1:] - cu_seqlens[:-1]).tolist()      # host copies of the
    pads = cu_seqlens_padded.tolist()                         # (small) offset arrays
    n = 2 * cp_size
    for b in range(len(lens)):
        assert (pads[b + 1] - pads[b]) % n == 0 and lens[b] <= pads[b + 1] - pads[b]
    cus, starts, longest = _chunk_views(lens, pads, cp_size, q.device)
    acc_q = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    acc_k = torch.empty(k.shape, dtype=torch.float32, device=q.device)
    acc_v = torch.empty(v.shape, dtype=torch.float32, device=q.device)
    part_q, part_k, part_v = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    calls = [(cq, ck, cmask) for rank in range(cp_size) for _, cq, ck, cmask in ring_pairs(cp_size, rank, causal)]
    views = [dict(window=(-1, 0) if cmask else (-1, -1), cu_seqlens_q=cus[cq], cu_seqlens_kv=cus[ck],
                  max_seqlen_q=longest, max_seqlen_kv=longest, cu_seqlens_q_padded=starts[cq],
                  cu_seqlens_kv_padded=starts[ck]) for cq, ck, cmask in calls]
    need = max(attn_bwd_workspace_size(q, k, scale=scale, **kw) for kw in views)
    work = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    seen_q, seen_k = set(), set()
    for (cq, ck, _), kw in zip(calls, views):
        attn_bwd(dout, q, k, v, o, lse, scale=scale, dq=part_q, dk=part_k, dv=part_v, workspace=work, **kw)
        # each chunk's first share is copied, later ones added
        thd_accumulate(part_q, acc_q, cus[cq], starts[cq], accumulate=cq in seen_q)
        thd_accumulate(part_k, acc_k, cus[ck], starts[ck], accumulate=ck in seen_k)
        thd_accumulate(part_v, acc_v, cus[ck], starts[ck], accumulate=ck in seen_k)
        seen_q.add(cq)
        seen_k.add(ck)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    thd_store(acc_q, dq, cu_seqlens, cu_seqlens_padded)
    thd_store(acc_k, dk, cu_seqlens, cu_seqlens_padded)
    thd_store(acc_v, dv, cu_seqlens, cu_seqlens_padded)
    return dq, dk, dv
