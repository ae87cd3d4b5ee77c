"""Host-side arithmetic of bench.py (CPU): the visible-pair count behind every
TFLOP/s figure, checked against a count of an explicit boolean mask and the
closed forms of the causal, full and sliding-window cases."""
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _mask_count(S, window):
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    wl, wr = window
    vis = np.ones((S, S), bool)
    if wl >= 0:
        vis &= j >= i - wl
    if wr >= 0:
        vis &= j <= i + wr
    return int(vis.sum())


@pytest.mark.parametrize("S", [1, 2, 7, 128, 1000])
@pytest.mark.parametrize("window", [(-1, 0), (-1, -1), (0, 0), (64, 0), (5, 37), (300, 300)])
def test_n_visible_matches_mask(S, window):
    assert bench.n_visible(S, window) == _mask_count(S, window)


@pytest.mark.parametrize("S", [1, 128, 4096, 16384])
def test_n_visible_closed_forms(S):
    assert bench.n_visible(S, (-1, 0)) == S * (S + 1) // 2
    assert bench.n_visible(S, (-1, -1)) == S * S
    w = 1023
    m = min(S, w + 1)  # rows 0..m-1 see i+1 keys, the rest w+1
    assert bench.n_visible(S, (w, 0)) == m * (m + 1) // 2 + (S - m) * (w + 1)


def test_workload_flops():
    """The headline workload (causal B4 S4096 H16 D128): 4·D flops per visible
    pair forward, 10·D backward (five products including the recompute of S)."""
    B, S, H, D = 4, 4096, 16, 128
    f_fwd, f_bwd, nv = bench.flops(B, S, H, D, (-1, 0))
    assert nv == B * H * S * (S + 1) // 2 == 537001984
    assert f_fwd == 4 * D * nv
    assert f_bwd == 10 * D * nv
    assert f_fwd + f_bwd == 962307555328
