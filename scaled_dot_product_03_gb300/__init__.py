"""Fused scaled-dot-product attention for GB300 (sm_103a).

Python binding of the C ABI in ``include/gbattn.h``: the functions here only
marshal torch tensors into pointers, strides and sizes and call the library
on the current CUDA stream.  PyTorch supplies device memory for outputs the
caller does not pass.  Every step of the computation runs in the library's
CUDA kernels; there is no other implementation to fall back on.

* :func:`attn_fwd`  -- O and LSE (``softmax(scale * q k^T + mask) v``).
* :func:`attn_bwd`  -- dq, dk, dv from dO and the saved LSE.
* :func:`attn_merge_lse` -- merge two partial attentions by their LSE.
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import torch

from . import _lib

__all__ = ["attn_fwd", "attn_bwd", "attn_bwd_noalloc", "attn_merge_lse", "attn_bwd_workspace_size",
           "check_device_error", "set_watchdog_ns", "watchdog_selftest", "AttnError",
           "profile_begin", "profile_read",
           "params_for"]

AttnError = _lib.AttnError

_DTYPES = {torch.float16: _lib.ATTN_F16, torch.bfloat16: _lib.ATTN_BF16,
           torch.float32: _lib.ATTN_F32}


def _stream(t: torch.Tensor):
    return ctypes_void(torch.cuda.current_stream(t.device).cuda_stream)


def _device_of(t: torch.Tensor):
    """Makes the tensor's device current for the call: the library launches
    on the current device and its stream argument must belong to it."""
    return torch.cuda.device(t.device)


def ctypes_void(x):
    import ctypes
    return ctypes.c_void_p(x)


def _tensor(t: Optional[torch.Tensor], thd: bool) -> "_lib.AttnTensor":
    at = _lib.AttnTensor()
    if t is None:
        return at
    at.ptr = t.data_ptr()
    st = t.stride()
    if thd:
        assert t.dim() == 3, "THD tensors are [T, H, D]"
        at.stride[:] = (0, st[0], st[1], st[2])
    else:
        assert t.dim() == 4, "dense tensors are [B, S, H, D]"
        at.stride[:] = tuple(st)
    return at


def params_for(q, k, *, scale=None, window=(-1, -1), cu_seqlens_q=None, cu_seqlens_kv=None,
               max_seqlen_q=None, max_seqlen_kv=None, deterministic=False,
               cu_seqlens_q_padded=None, cu_seqlens_kv_padded=None) -> "_lib.AttnParams":
    """The ``attn_params`` struct describing q (and k, v) views.  THD
    ``cu_seqlens_*_padded`` (int32, device): first row of each sequence in a
    padded buffer."""
    p = _lib.AttnParams()
    p.deterministic = 1 if deterministic else 0
    if q.dtype not in _DTYPES:
        raise TypeError("unsupported dtype %s" % q.dtype)
    p.dtype = _DTYPES[q.dtype]
    thd = cu_seqlens_q is not None
    D = q.shape[-1]
    p.D = D
    p.scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    p.window_left, p.window_right = int(window[0]), int(window[1])
    if thd:
        if cu_seqlens_kv is None:
            cu_seqlens_kv = cu_seqlens_q
        p.layout = _lib.ATTN_LAYOUT_THD
        p.B = cu_seqlens_q.numel() - 1
        p.Sq, p.Hq = q.shape[0], q.shape[1]
        p.Skv, p.Hkv = k.shape[0], k.shape[1]
        p.cu_seqlens_q = cu_seqlens_q.data_ptr()
        p.cu_seqlens_kv = cu_seqlens_kv.data_ptr()
        if cu_seqlens_q_padded is not None:
            p.cu_seqlens_q_padded = cu_seqlens_q_padded.data_ptr()
            if cu_seqlens_kv_padded is None:
                cu_seqlens_kv_padded = cu_seqlens_q_padded
        if cu_seqlens_kv_padded is not None:
            p.cu_seqlens_kv_padded = cu_seqlens_kv_padded.data_ptr()
        if max_seqlen_q is None:  # needs a device->host read of cu_seqlens
            max_seqlen_q = int((cu_seqlens_q[1:] - cu_seqlens_q[:-1]).max()) if p.B else 0
        if max_seqlen_kv is None:
            max_seqlen_kv = int((cu_seqlens_kv[1:] - cu_seqlens_kv[:-1]).max()) if p.B else 0
        p.max_seqlen_q, p.max_seqlen_kv = int(max_seqlen_q), int(max_seqlen_kv)
    else:
        p.layout = _lib.ATTN_LAYOUT_DENSE4D
        p.B, p.Sq, p.Hq = q.shape[0], q.shape[1], q.shape[2]
        p.Skv, p.Hkv = k.shape[1], k.shape[2]
    return p


def _lse_shape(p):
    if p.layout == _lib.ATTN_LAYOUT_THD:
        return (p.Hq, p.Sq)
    return (p.B, p.Hq, p.Sq)


def attn_fwd(q, k, v, *, scale=None, window=(-1, -1), cu_seqlens_q=None, cu_seqlens_kv=None,
             max_seqlen_q=None, max_seqlen_kv=None, out=None, lse=None,
             cu_seqlens_q_padded=None, cu_seqlens_kv_padded=None
             ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Forward attention.  Dense: q ``[B, Sq, Hq, D]``, k/v ``[B, Skv, Hkv, D]``
    (any strides, d contiguous).  THD (``cu_seqlens_q`` given): q ``[Tq, Hq, D]``,
    k/v ``[Tkv, Hkv, D]``.  ``window=(left, right)``, -1 unbounded, (-1, 0)
    causal.  Returns ``(o, lse)`` with lse fp32 ``[B, Hq, Sq]`` / ``[Hq, Tq]``."""
    p = params_for(q, k, scale=scale, window=window, cu_seqlens_q=cu_seqlens_q,
                   cu_seqlens_kv=cu_seqlens_kv, max_seqlen_q=max_seqlen_q,
                   max_seqlen_kv=max_seqlen_kv, cu_seqlens_q_padded=cu_seqlens_q_padded,
                   cu_seqlens_kv_padded=cu_seqlens_kv_padded)
    thd = p.layout == _lib.ATTN_LAYOUT_THD
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(_lse_shape(p), dtype=torch.float32, device=q.device)
    lib = _lib.load()
    with _device_of(q):
        _lib.check(lib.attn_fwd(p, _tensor(q, thd), _tensor(k, thd), _tensor(v, thd),
                                _tensor(out, thd), lse.data_ptr(), _stream(q)))
    return out, lse


def attn_bwd_workspace_size(q, k, **kw) -> int:
    p = params_for(q, k, **kw)
    return int(_lib.load().attn_bwd_workspace_size(p))


def attn_bwd(dout, q, k, v, out, lse, *, scale=None, window=(-1, -1), cu_seqlens_q=None,
             cu_seqlens_kv=None, max_seqlen_q=None, max_seqlen_kv=None, dq=None, dk=None,
             dv=None, workspace=None, deterministic=False, dlse=None,
             cu_seqlens_q_padded=None, cu_seqlens_kv_padded=None
             ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Backward attention: ``(dq, dk, dv)`` for upstream gradient ``dout``
    (and ``dlse``, the gradient with respect to the forward's LSE output,
    fp32 in its layout; None: zero), recomputing P from q, k and ``lse``.  ``workspace`` (uint8
    device tensor of at least :func:`attn_bwd_workspace_size` bytes, with the
    same ``deterministic``) is allocated when not given.  ``deterministic``
    selects the bitwise-reproducible two-kernel backward instead of the
    single pass whose fp32 dq sums may differ in their last bits between
    runs."""
    p = params_for(q, k, scale=scale, window=window, cu_seqlens_q=cu_seqlens_q,
                   cu_seqlens_kv=cu_seqlens_kv, max_seqlen_q=max_seqlen_q,
                   max_seqlen_kv=max_seqlen_kv, deterministic=deterministic,
                   cu_seqlens_q_padded=cu_seqlens_q_padded,
                   cu_seqlens_kv_padded=cu_seqlens_kv_padded)
    thd = p.layout == _lib.ATTN_LAYOUT_THD
    lib = _lib.load()
    if dq is None:
        dq = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if dk is None:
        dk = torch.empty(k.shape, dtype=k.dtype, device=k.device)
    if dv is None:
        dv = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    need = int(lib.attn_bwd_workspace_size(p))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    ws = (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    if dlse is None:
        with _device_of(q):
            _lib.check(lib.attn_bwd(p, _tensor(q, thd), _tensor(k, thd), _tensor(v, thd),
                                    _tensor(out, thd), _tensor(dout, thd), lse.data_ptr(),
                                    _tensor(dq, thd), _tensor(dk, thd), _tensor(dv, thd), *ws,
                                    _stream(q)))
    else:
        assert dlse.dtype == torch.float32 and dlse.is_contiguous() and dlse.shape == lse.shape
        with _device_of(q):
            _lib.check(lib.attn_bwd_dlse(p, _tensor(q, thd), _tensor(k, thd), _tensor(v, thd),
                                         _tensor(out, thd), _tensor(dout, thd), lse.data_ptr(),
                                         dlse.data_ptr(), _tensor(dq, thd), _tensor(dk, thd),
                                         _tensor(dv, thd), *ws, _stream(q)))
    return dq, dk, dv


def attn_bwd_noalloc(dout, q, k, v, out, lse, *, scale=None, window=(-1, -1),
                     cu_seqlens_q=None, cu_seqlens_kv=None, max_seqlen_q=None,
                     max_seqlen_kv=None, dq=None, dk=None, dv=None, deterministic=False,
                     cu_seqlens_q_padded=None, cu_seqlens_kv_padded=None
                     ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """:func:`attn_bwd` for callers that cannot allocate device scratch: the
    library's own fixed scratch array (``_lib.NOALLOC_SCRATCH_BYTES`` bytes per
    device) replaces the workspace.  Calls share that array, so calls that
    could overlap on the GPU must be serialised.  (This wrapper still lets
    torch allocate dq/dk/dv when they are not passed.)"""
    p = params_for(q, k, scale=scale, window=window, cu_seqlens_q=cu_seqlens_q,
                   cu_seqlens_kv=cu_seqlens_kv, max_seqlen_q=max_seqlen_q,
                   max_seqlen_kv=max_seqlen_kv, deterministic=deterministic,
                   cu_seqlens_q_padded=cu_seqlens_q_padded,
                   cu_seqlens_kv_padded=cu_seqlens_kv_padded)
    thd = p.layout == _lib.ATTN_LAYOUT_THD
    if dq is None:
        dq = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if dk is None:
        dk = torch.empty(k.shape, dtype=k.dtype, device=k.device)
    if dv is None:
        dv = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    lib = _lib.load()
    with _device_of(q):
        _lib.check(lib.attn_bwd_noalloc(p, _tensor(q, thd), _tensor(k, thd), _tensor(v, thd),
                                        _tensor(out, thd), _tensor(dout, thd), lse.data_ptr(),
                                        _tensor(dq, thd), _tensor(dk, thd), _tensor(dv, thd),
                                        _stream(q)))
    return dq, dk, dv


def attn_merge_lse(o1, lse1, o2, lse2, *, out=None, lse_out=None
                   ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Merge two partial attentions over disjoint key sets by their LSE.
    Dense: o ``[B, S, H, D]`` with lse ``[B, H, S]``; THD: o ``[T, H, D]``
    with lse ``[H, T]``.  ``out`` / ``lse_out`` may be ``o1`` / ``lse1``
    (in place)."""
    if out is None:
        out = torch.empty(o1.shape, dtype=o1.dtype, device=o1.device)
    if lse_out is None:
        lse_out = torch.empty(lse1.shape, dtype=torch.float32, device=lse1.device)
    if o1.dim() == 3:
        T, H, D = o1.shape
        B, S = 1, T
        views = [x.unsqueeze(0) for x in (o1, o2, out)]
    else:
        B, S, H, D = o1.shape
        views = [o1, o2, out]
    for l in (lse1, lse2, lse_out):
        assert l.dtype == torch.float32 and l.is_contiguous() and l.numel() == B * H * S
    if o1.dtype not in _DTYPES:
        raise TypeError("unsupported dtype %s" % o1.dtype)
    lib = _lib.load()
    with _device_of(o1):
        _lib.check(lib.attn_merge_lse(_DTYPES[o1.dtype], B, S, H, D, _tensor(views[0], False),
                                      lse1.data_ptr(), _tensor(views[1], False), lse2.data_ptr(),
                                      _tensor(views[2], False), lse_out.data_ptr(), _stream(o1)))
    return out, lse_out


def attn_merge_lse_bwd(o1, lse1, o2, lse2, dout, dlse=None, *, do1=None, dlse1=None, do2=None,
                       dlse2=None):
    """Backward of :func:`attn_merge_lse`: ``(do1, dlse1, do2, dlse2)`` for
    the gradients ``dout`` of the merged o and ``dlse`` of the merged lse
    (None: zero).  Shapes as for :func:`attn_merge_lse`."""
    do1 = torch.empty(o1.shape, dtype=o1.dtype, device=o1.device) if do1 is None else do1
    do2 = torch.empty(o2.shape, dtype=o2.dtype, device=o2.device) if do2 is None else do2
    dlse1 = torch.empty_like(lse1) if dlse1 is None else dlse1
    dlse2 = torch.empty_like(lse2) if dlse2 is None else dlse2
    if o1.dim() == 3:
        T, H, D = o1.shape
        B, S = 1, T
        views = [x.unsqueeze(0) for x in (o1, o2, dout, do1, do2)]
    else:
        B, S, H, D = o1.shape
        views = [o1, o2, dout, do1, do2]
    lses = [lse1, lse2, dlse1, dlse2] + ([] if dlse is None else [dlse])
    for l in lses:
        assert l.dtype == torch.float32 and l.is_contiguous() and l.numel() == B * H * S
    if o1.dtype not in _DTYPES:
        raise TypeError("unsupported dtype %s" % o1.dtype)
    lib = _lib.load()
    with _device_of(o1):
        _lib.check(lib.attn_merge_lse_bwd(_DTYPES[o1.dtype], B, S, H, D, _tensor(views[0], False),
                                          lse1.data_ptr(), _tensor(views[1], False), lse2.data_ptr(),
                                          _tensor(views[2], False),
                                          None if dlse is None else dlse.data_ptr(),
                                          _tensor(views[3], False), dlse1.data_ptr(),
                                          _tensor(views[4], False), dlse2.data_ptr(), _stream(o1)))
    return do1, dlse1, do2, dlse2


def profile_begin(max_launches: int) -> None:
    """Start timing each kernel launch of the calling thread (see
    attn_profile_begin in include/gbattn.h)."""
    _lib.check(_lib.load().attn_profile_begin(int(max_launches)))


def profile_read(capacity: int = 4096):
    """Stop timing; returns ``[(kind_name, milliseconds), ...]`` per launch."""
    import ctypes
    ms = (ctypes.c_float * capacity)()
    kind = (ctypes.c_int * capacity)()
    n = _lib.load().attn_profile_read(ctypes.cast(ms, ctypes.c_void_p),
                                      ctypes.cast(kind, ctypes.c_void_p), capacity)
    if n < 0:
        raise AttnError(_lib.ATTN_ERR_CUDA, "attn_profile_read failed")
    return [(_lib.KERNEL_KINDS.get(kind[i], str(kind[i])), float(ms[i])) for i in range(n)]


def check_device_error(device=None) -> None:
    """Raises :class:`AttnError` if a kernel watchdog fired since the last check."""
    s = torch.cuda.current_stream(device)
    _lib.check(_lib.load().attn_check_device_error(ctypes_void(s.cuda_stream)))


def set_watchdog_ns(ns: int) -> int:
    return int(_lib.load().attn_set_watchdog_ns(int(ns)))


def watchdog_selftest(device=None) -> None:
    s = torch.cuda.current_stream(device)
    _lib.check(_lib.load().attn_watchdog_selftest(ctypes_void(s.cuda_stream)))
