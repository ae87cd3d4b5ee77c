"""Host planning of the context-parallel ring emulation (CPU): which
(query chunk, key chunk) pairs each rank computes, and the chunk views of a
padded THD buffer.  "[PyTorch] Add support for cuDNN FusedAttention + THD +
CP": every sequence is cut into 2 CP chunks, rank r holds chunks r and
2 CP - 1 - r, and K/V chunks travel around a ring of ranks."""
import itertools

import pytest

from scaled_dot_product_03_gb300.cp import _chunk_views, ring_pairs


@pytest.mark.parametrize("cp_size", [1, 2, 3, 4])
@pytest.mark.parametrize("causal", [True, False])
def test_ring_pairs_cover_every_pair_once(cp_size, causal):
    n = 2 * cp_size
    seen = []
    for rank in range(cp_size):
        own = {rank, n - 1 - rank}
        for step, cq, ck, cmask in ring_pairs(cp_size, rank, causal):
            assert cq in own                       # a rank only computes its own queries
            src = (rank - step) % cp_size          # K/V it holds at this step
            assert ck in (src, n - 1 - src)
            assert cmask == (causal and ck == cq)  # causal mask only on the diagonal
            assert not (causal and ck > cq)        # later chunks are never visited
            seen.append((cq, ck))
    want = [(cq, ck) for cq, ck in itertools.product(range(n), range(n)) if not causal or ck <= cq]
    assert sorted(seen) == sorted(want)


def test_ring_pairs_steps_in_ring_order():
    steps = [s for s, *_ in ring_pairs(4, 1, True)]
    assert steps == sorted(steps) and set(steps) == {0, 1, 2, 3}


@pytest.mark.parametrize("cp_size", [1, 2, 3])
def test_chunk_views_partition_each_sequence(cp_size):
    n = 2 * cp_size
    lengths = [0, 1, 5, 12, 37]
    pads = [0]
    for L in lengths:  # padded length: a multiple of 2 CP, at least L
        pads.append(pads[-1] + max(n, -(-L // n) * n) + n)
    cus, starts, longest = _chunk_views(lengths, pads, cp_size, "cpu")
    assert len(cus) == len(starts) == n
    for b, L in enumerate(lengths):
        size = (pads[b + 1] - pads[b]) // n
        total = 0
        for c in range(n):
            cu, st = cus[c].tolist(), starts[c].tolist()
            m = cu[b + 1] - cu[b]
            assert st[b] == pads[b] + c * size            # chunk c starts c sizes in
            assert m == max(0, min(size, L - c * size))   # padding rows excluded
            assert m <= longest
            total += m
        assert total == L                                 # the chunks cover the sequence
    for c in range(n):
        assert starts[c].tolist()[-1] == pads[-1]
