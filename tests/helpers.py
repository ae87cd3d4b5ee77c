"""Test-side marshalling between problems and the float64 oracle.

Only reshapes and upcasts: no attention arithmetic lives here.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).contiguous().numpy()


def packed(prob, name):
    """Tensor ``name`` of ``prob`` as float64 ``[T, H, D]`` token rows."""
    t = prob.tensor(name)
    a = to_f64(t)
    if prob.layout == "dense":
        a = a.reshape(-1, a.shape[2], a.shape[3])
    return a


def cu(prob):
    if prob.layout == "thd":
        return (prob.cu_seqlens_q.cpu().numpy().astype(np.int64),
                prob.cu_seqlens_kv.cpu().numpy().astype(np.int64))
    return oracle.dense_cu(prob.B, prob.Sq), oracle.dense_cu(prob.B, prob.Skv)


def oracle_fwd(prob, row_sel=None):
    cq, ck = cu(prob)
    return oracle.attn_fwd(packed(prob, "q"), packed(prob, "k"), packed(prob, "v"),
                           cq, ck, prob.scale, prob.window, row_sel=row_sel)


def oracle_bwd(prob, row_sel=None, key_sel=None, want_stats=False):
    cq, ck = cu(prob)
    return oracle.attn_bwd(packed(prob, "q"), packed(prob, "k"), packed(prob, "v"),
                           packed(prob, "dout"), cq, ck, prob.scale, prob.window,
                           row_sel=row_sel, key_sel=key_sel, want_stats=want_stats)


def lse_to_library_layout(prob, lse_rows: np.ndarray) -> np.ndarray:
    """Oracle LSE ``[Tq, Hq]`` -> the library's ``[B, Hq, Sq]`` (dense) or
    ``[Hq, Tq]`` (THD)."""
    if prob.layout == "dense":
        return lse_rows.reshape(prob.B, prob.Sq, prob.Hq).transpose(0, 2, 1)
    return lse_rows.T


def rows_to_dense(prob, a: np.ndarray) -> np.ndarray:
    """Oracle ``[T, H, D]`` rows -> ``[B, S, H, D]`` for a dense problem."""
    if prob.layout == "dense":
        return a.reshape(prob.B, -1, a.shape[1], a.shape[2])
    return a
