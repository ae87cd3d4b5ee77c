"""Float64 CPU oracle for fused scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package.  The CUDA library never calls it
and shares no code with it; see ``oracle.c`` for the definitions it follows
and the passages of the source pages each one restates.

Every array handed to the oracle is float64 and contiguous, in the packed
token-row layouts of ``oracle.c``:

* ``q``, ``o``, ``dq``: ``[Tq, Hq, D]``;  ``k``, ``v``, ``dk``, ``dv``: ``[Tkv, Hkv, D]``
* ``lse``: ``[Tq, Hq]``
* ``cu_q``, ``cu_kv``: int64 ``[nseq + 1]`` row offsets of each sequence.

A dense batch ``[B, S, H, D]`` is passed by reshaping to ``[B*S, H, D]`` with
``cu = [0, S, 2S, ...]`` (see :func:`dense_cu`).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc (plain -O2, OpenMP, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_attn_fwd.argtypes = [i32, P, P, i32, i32, i32, P, P, P,
                                            f64, i32, i32, P, P, P]
            lib.oracle_attn_fwd.restype = None
            lib.oracle_attn_bwd.argtypes = [i32, P, P, i32, i32, i32, P, P, P,
                                            P, P, f64, i32, i32, P, P, P, P, P,
                                            P, P]
            lib.oracle_attn_bwd.restype = None
            lib.oracle_merge_lse.argtypes = [i64, i32, P, P, P, P, P, P]
            lib.oracle_merge_lse.restype = None
            lib.oracle_merge_lse_bwd.argtypes = [i64, i32, P, P, P, P, P, P, P, P, P, P]
            lib.oracle_merge_lse_bwd.restype = None
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = i32
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _sel(sel, shape):
    if sel is None:
        return None
    s = np.ascontiguousarray(np.asarray(sel, dtype=np.uint8))
    assert s.shape == shape, (s.shape, shape)
    return s


def dense_cu(batch: int, seqlen: int) -> np.ndarray:
    """Row offsets of a dense batch of ``batch`` sequences of ``seqlen``."""
    return np.arange(batch + 1, dtype=np.int64) * seqlen


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def attn_fwd(q, k, v, cu_q, cu_kv, scale, window=(-1, -1), row_sel=None):
    """Returns ``(o [Tq,Hq,D], lse [Tq,Hq])``; unselected rows are 0 / NaN."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu_q = np.ascontiguousarray(cu_q, dtype=np.int64)
    cu_kv = np.ascontiguousarray(cu_kv, dtype=np.int64)
    Tq, Hq, D = q.shape
    Hkv = k.shape[1]
    assert k.shape == v.shape and k.shape[2] == D and Hq % Hkv == 0
    assert cu_q[-1] == Tq and cu_kv[-1] == k.shape[0] and len(cu_q) == len(cu_kv)
    sel = _sel(row_sel, (Tq, Hq))
    o = np.zeros((Tq, Hq, D))
    lse = np.full((Tq, Hq), np.nan)
    _load().oracle_attn_fwd(len(cu_q) - 1, _ptr(cu_q), _ptr(cu_kv), Hq, Hkv, D,
                            _ptr(q), _ptr(k), _ptr(v), float(scale),
                            int(window[0]), int(window[1]), _ptr(sel),
                            _ptr(o), _ptr(lse))
    return o, lse


def attn_bwd(q, k, v, dout, cu_q, cu_kv, scale, window=(-1, -1),
             row_sel=None, key_sel=None, want_stats=False, dlse=None):
    """Returns ``(dq, dk, dv)`` (plus ``(lse, r)`` with ``want_stats``).
    ``dlse`` ``[Tq, Hq]``: gradient with respect to the LSE output (None: 0)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    cu_q = np.ascontiguousarray(cu_q, dtype=np.int64)
    cu_kv = np.ascontiguousarray(cu_kv, dtype=np.int64)
    Tq, Hq, D = q.shape
    Tkv, Hkv, _ = k.shape
    assert dout.shape == q.shape and Hq % Hkv == 0
    rs, ks = _sel(row_sel, (Tq, Hq)), _sel(key_sel, (Tkv, Hkv))
    if dlse is not None:
        dlse = _f64(dlse)
        assert dlse.shape == (Tq, Hq)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    lse = np.full((Tq, Hq), np.nan) if want_stats else None
    r = np.full((Tq, Hq), np.nan) if want_stats else None
    _load().oracle_attn_bwd(len(cu_q) - 1, _ptr(cu_q), _ptr(cu_kv), Hq, Hkv, D,
                            _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dlse), float(scale),
                            int(window[0]), int(window[1]), _ptr(rs), _ptr(ks),
                            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(lse), _ptr(r))
    if want_stats:
        return dq, dk, dv, lse, r
    return dq, dk, dv


def merge_lse(o1, lse1, o2, lse2):
    """``o*: [..., D]``, ``lse*: [...]`` -> merged ``(o, lse)``."""
    o1, o2 = _f64(o1), _f64(o2)
    lse1, lse2 = _f64(lse1), _f64(lse2)
    shape = o1.shape
    D = shape[-1]
    n = int(np.prod(shape[:-1]))
    assert o2.shape == shape and lse1.shape == shape[:-1] == lse2.shape
    o = np.empty(shape)
    lse = np.empty(shape[:-1])
    _load().oracle_merge_lse(n, D, _ptr(o1), _ptr(lse1), _ptr(o2), _ptr(lse2),
                             _ptr(o), _ptr(lse))
    return o, lse


def merge_lse_bwd(o1, lse1, o2, lse2, dout, dlse=None):
    """Backward of :func:`merge_lse`: ``(do1, dlse1, do2, dlse2)`` for the
    gradients ``dout`` of the merged o and ``dlse`` of the merged lse."""
    o1, o2, dout = _f64(o1), _f64(o2), _f64(dout)
    lse1, lse2 = _f64(lse1), _f64(lse2)
    shape = o1.shape
    D = shape[-1]
    n = int(np.prod(shape[:-1]))
    assert o2.shape == shape == dout.shape and lse1.shape == shape[:-1] == lse2.shape
    if dlse is not None:
        dlse = _f64(dlse)
        assert dlse.shape == shape[:-1]
    do1, do2 = np.empty(shape), np.empty(shape)
    dl1, dl2 = np.empty(shape[:-1]), np.empty(shape[:-1])
    _load().oracle_merge_lse_bwd(n, D, _ptr(o1), _ptr(lse1), _ptr(o2), _ptr(lse2),
                                 _ptr(dout), _ptr(dlse), _ptr(do1), _ptr(dl1),
                                 _ptr(do2), _ptr(dl2))
    return do1, dl1, do2, dl2


# ---------------------------------------------------------------------------
# Context parallelism over THD ("[PyTorch] Add support for cuDNN
# FusedAttention + THD + CP": every sequence is split into CP*2 chunks and
# each rank is given 2 of them for load balance; K/V move around a ring of
# ranks and each rank merges its partial results; the order of the ring
# does not matter).  Plain loops, float64, on gathered copies of the chunks.

def thd_partitioned_indices(cu_seqlens_padded, total_tokens, world_size, rank):
    """Rows of the padded THD buffer held by ``rank``: for every sequence,
    the rows of chunk ``rank`` then of chunk ``2 * world_size - 1 - rank``
    of its 2 * world_size equal chunks."""
    pads = [int(x) for x in cu_seqlens_padded]
    assert pads[-1] == total_tokens
    n = 2 * world_size
    rows = []
    for b in range(len(pads) - 1):
        size = (pads[b + 1] - pads[b]) // n
        for c in (rank, n - 1 - rank):
            rows.extend(range(pads[b] + c * size, pads[b] + (c + 1) * size))
    return np.array(rows, dtype=np.int64)


def ring_attention_fwd(q, k, v, cu_seqlens, cu_seqlens_padded, cp_size, scale, causal=True):
    """Every rank's ring, as float64 partial attentions merged by LSE.
    q, k, v: padded THD ``[T, H, D]``; returns ``(o [T, Hq, D], lse [T, Hq])``
    with o = 0, lse = -inf on padding rows.  A query chunk at sequence
    offset a against a key chunk at offset c sees key j from query i iff
    a + i >= c + j (causal), i.e. window (-1, a - c); pairs with a < c see
    nothing."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    lens = np.diff(np.asarray(cu_seqlens, dtype=np.int64))
    pads = [int(x) for x in cu_seqlens_padded]
    T, Hq, D = q.shape
    n = 2 * cp_size
    o = np.zeros((T, Hq, D))
    lse = np.full((T, Hq), -np.inf)
    for rank in range(cp_size):
        for b, L in enumerate(lens):
            size = (pads[b + 1] - pads[b]) // n
            for cq in (rank, n - 1 - rank):
                a = cq * size
                nq = max(0, min(size, L - a))
                if nq == 0:
                    continue
                rows = np.arange(pads[b] + a, pads[b] + a + nq)
                acc_o, acc_l = np.zeros((nq, Hq, D)), np.full((nq, Hq), -np.inf)
                for step in range(cp_size):           # K/V of rank (rank - step) mod CP
                    src = (rank - step) % cp_size
                    for ck in (src, n - 1 - src):
                        c = ck * size
                        nk = max(0, min(size, L - c))
                        if nk == 0 or (causal and a < c):
                            continue
                        kr = np.arange(pads[b] + c, pads[b] + c + nk)
                        window = (-1, a - c) if causal else (-1, -1)
                        po, pl = attn_fwd(q[rows], k[kr], v[kr], np.array([0, nq]),
                                          np.array([0, nk]), scale, window)
                        acc_o, acc_l = merge_lse(acc_o, acc_l, po, pl)
                o[rows], lse[rows] = acc_o, acc_l
    return o, lse
