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
later chunks not at all.  All arithmetic runs in the library's kernels; this
module only plans the calls.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import torch

from . import _lib, attn_fwd, attn_merge_lse


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
