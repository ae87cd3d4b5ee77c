"""Seeded synthetic inputs shaped like the source pages' workloads.

This module only draws random numbers and arranges them in memory (views,
packing, cu_seqlens).  It holds none of the attention arithmetic, so the CUDA
path and the float64 oracle can both be fed from it.  Every tensor is drawn
on the CPU from ``torch.Generator().manual_seed(seed)`` (the pages seed with
``torch.manual_seed(0)`` and draw with ``torch.randn``), cast to the workload
dtype, and only then moved to a device, so both sides see identical bytes.

Workloads (one constructor each):

* :func:`pr1` -- forward only, fp16, B=1, S=128, 4 query heads sharing 1 KV
  head, D=64, causal, scale 1/8, contiguous (b, s, h, d).
* :func:`page1` -- "[PyTorch] fused CUDNN attention kernel not properly
  handling strides": one packed fp16 tensor [2048, 1, 16+2, 64] split on the
  head dim into q, k, v (an sb(h+2h_g)d layout, strides (1152, 1152, 64, 1)),
  causal, scale 1.0 or 0.1.
* :func:`page3` -- "Significant Accuracy Difference between Compiled and
  Eager Flex Attention": fp32 x ~ N(0,1) [1, 512, 256] through a 256->768
  linear whose weights and biases are all 0.1, split into q, k, v of 4 heads
  of 64; non-causal, scale 1/8, dO = ones.
* :func:`dense` -- contiguous (b, s, h, d) bf16 causal self-attention (the
  S=1024/H=16/D=64 case and the 16384-tokens-per-batch D=128 sweep).
* :func:`varlen` -- packed THD batch addressed by cu_seqlens ("[PyTorch] Add
  support for cuDNN FusedAttention + THD + CP"): 16 sequences with lengths
  uniform in [128, 4096], 32 query heads over 8 KV heads, D=128, causal.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, Optional, Tuple

import torch

__all__ = ["Attn", "pr1", "page1", "page3", "dense", "varlen", "random_case"]


def _gen(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed))


def _randn(shape, g: torch.Generator, dtype: torch.dtype) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32).to(dtype)


@dataclass
class Attn:
    """One attention problem.

    Dense: ``q`` is ``[B, Sq, Hq, D]``, ``k``/``v`` ``[B, Skv, Hkv, D]``, any
    strides (views into ``bases``).  THD: ``q`` is ``[Tq, Hq, D]``, ``k``/``v``
    ``[Tkv, Hkv, D]`` with ``cu_seqlens_q/kv`` (int32, ``B + 1`` entries) and
    ``Sq``/``Skv`` holding the longest sequence.  ``window`` is
    ``(left, right)`` with -1 meaning unbounded; ``(-1, 0)`` is causal.
    """

    name: str
    dtype: torch.dtype
    layout: str
    B: int
    Sq: int
    Skv: int
    Hq: int
    Hkv: int
    D: int
    scale: float
    window: Tuple[int, int]
    bases: Dict[str, torch.Tensor]
    views: Dict[str, Tuple[str, tuple, tuple, int]]
    cu_seqlens_q: Optional[torch.Tensor] = None
    cu_seqlens_kv: Optional[torch.Tensor] = None
    extra: dict = field(default_factory=dict)

    def tensor(self, name: str) -> Optional[torch.Tensor]:
        if name not in self.views:
            return None
        base, size, stride, off = self.views[name]
        return self.bases[base].as_strided(size, stride, off)

    @property
    def q(self):
        return self.tensor("q")

    @property
    def k(self):
        return self.tensor("k")

    @property
    def v(self):
        return self.tensor("v")

    @property
    def dout(self):
        return self.tensor("dout")

    @property
    def total_q(self) -> int:
        return self.q.shape[0] if self.layout == "thd" else self.B * self.Sq

    @property
    def total_kv(self) -> int:
        return self.k.shape[0] if self.layout == "thd" else self.B * self.Skv

    def to(self, device) -> "Attn":
        """Same problem with every base moved to ``device`` (views rebuilt
        with the same strides and offsets, so no layout changes)."""
        bases = {n: b.to(device) for n, b in self.bases.items()}
        return Attn(self.name, self.dtype, self.layout, self.B, self.Sq,
                    self.Skv, self.Hq, self.Hkv, self.D, self.scale,
                    self.window, bases, dict(self.views),
                    None if self.cu_seqlens_q is None else self.cu_seqlens_q.to(device),
                    None if self.cu_seqlens_kv is None else self.cu_seqlens_kv.to(device),
                    dict(self.extra))

    def lengths(self):
        """Per-sequence (Lq, Lkv) pairs."""
        if self.layout == "thd":
            cq = self.cu_seqlens_q.cpu().tolist()
            ck = self.cu_seqlens_kv.cpu().tolist()
            return [(cq[i + 1] - cq[i], ck[i + 1] - ck[i]) for i in range(self.B)]
        return [(self.Sq, self.Skv)] * self.B


def _contig(name, t):
    return {name: t}, {name: (name, tuple(t.shape), tuple(t.stride()), 0)}


def _problem(name, dtype, layout, B, Sq, Skv, Hq, Hkv, D, scale, window,
             tensors: Dict[str, torch.Tensor], **kw) -> Attn:
    bases, views = {}, {}
    for n, t in tensors.items():
        b, v = _contig(n, t.contiguous())
        bases.update(b)
        views.update(v)
    return Attn(name, dtype, layout, B, Sq, Skv, Hq, Hkv, D, scale, window,
                bases, views, **kw)


def pr1(seed: int = 0) -> Attn:
    g = _gen(seed)
    B, S, Hq, Hkv, D = 1, 128, 4, 1, 64
    q = _randn((B, S, Hq, D), g, torch.float16)
    k = _randn((B, S, Hkv, D), g, torch.float16)
    v = _randn((B, S, Hkv, D), g, torch.float16)
    return _problem("pr1_fp16_s128_mqa_causal", torch.float16, "dense", B, S,
                    S, Hq, Hkv, D, 1.0 / math.sqrt(D), (-1, 0),
                    {"q": q, "k": k, "v": v})


def page1(scale: float = 1.0, seed: int = 0, seqlen: int = 2048,
          q_heads: int = 16, kv_heads: int = 1, head_dim: int = 64,
          dout_seed: Optional[int] = None) -> Attn:
    """Packed ``qkv[s, 1, h + 2 h_g, d]`` split on dim 2 into q, k, v views.

    The views are sbhd tensors; they are exposed in (b, s, h, d) order by a
    permute, which changes no memory, so their element strides are
    (b, s, h, d) = (1152, 1152, 64, 1) at the page's sizes.  With
    ``dout_seed`` an upstream gradient ``[1, s, h, d]`` (contiguous) is drawn
    from its own generator for the backward.
    """
    g = _gen(seed)
    H = q_heads + 2 * kv_heads
    qkv = _randn((seqlen, 1, H, head_dim), g, torch.float16)
    st = qkv.stride()  # (H*d, H*d, d, 1)
    bstride = (st[1], st[0], st[2], st[3])  # (b, s, h, d)
    views = {
        "q": ("qkv", (1, seqlen, q_heads, head_dim), bstride, 0),
        "k": ("qkv", (1, seqlen, kv_heads, head_dim), bstride, q_heads * head_dim),
        "v": ("qkv", (1, seqlen, kv_heads, head_dim), bstride,
              (q_heads + kv_heads) * head_dim),
    }
    bases = {"qkv": qkv}
    if dout_seed is not None:
        dout = _randn((1, seqlen, q_heads, head_dim), _gen(dout_seed), torch.float16)
        bases["dout"] = dout
        views["dout"] = ("dout", tuple(dout.shape), tuple(dout.stride()), 0)
    return Attn("page1_fp16_packed_sbhd_s%d_scale%g" % (seqlen, scale),
                torch.float16, "dense", 1, seqlen, seqlen, q_heads, kv_heads,
                head_dim, float(scale), (-1, 0), bases, views)


def page3(seed: int = 0) -> Attn:
    """x ~ N(0,1) [1, 512, 256] -> linear(256, 768) with all weights and
    biases 0.1 -> split into q, k, v [1, 512, 4, 64] views of the packed
    projection (strides (393216, 768, 64, 1)); dO = ones.

    The projection is input preparation, evaluated in float64 and rounded to
    fp32 once; ``extra['x']`` keeps x for tests that use it.
    """
    g = _gen(seed)
    n_batch, n_ctx, d_model, n_head = 1, 512, 256, 4
    x = torch.randn((n_batch, n_ctx, d_model), generator=g, dtype=torch.float32)
    w = torch.full((3 * d_model, d_model), 0.1, dtype=torch.float64)
    bias = torch.full((3 * d_model,), 0.1, dtype=torch.float64)
    packed = (x.to(torch.float64) @ w.T + bias).to(torch.float32)
    D = d_model // n_head
    st = packed.stride()  # (n_ctx*768, 768, 1)
    stride = (st[0], st[1], D, 1)
    size = (n_batch, n_ctx, n_head, D)
    views = {"q": ("packed", size, stride, 0),
             "k": ("packed", size, stride, d_model),
             "v": ("packed", size, stride, 2 * d_model),
             "dout": ("dout", size, (n_ctx * n_head * D, n_head * D, D, 1), 0)}
    bases = {"packed": packed, "dout": torch.ones(size, dtype=torch.float32)}
    return Attn("page3_fp32_linear01_s512_h4", torch.float32, "dense", n_batch,
                n_ctx, n_ctx, n_head, n_head, D, 1.0 / math.sqrt(D), (-1, -1),
                bases, views, extra={"x": x})


def dense(B: int, S: int, H: int, D: int, dtype=torch.bfloat16,
          window=(-1, 0), seed: int = 0, dout_seed: Optional[int] = 1,
          Hkv: Optional[int] = None, Skv: Optional[int] = None,
          scale: Optional[float] = None, name: Optional[str] = None) -> Attn:
    """Contiguous (b, s, h, d) self-attention with N(0,1) data."""
    Hkv = H if Hkv is None else Hkv
    Skv = S if Skv is None else Skv
    g = _gen(seed)
    q = _randn((B, S, H, D), g, dtype)
    k = _randn((B, Skv, Hkv, D), g, dtype)
    v = _randn((B, Skv, Hkv, D), g, dtype)
    t = {"q": q, "k": k, "v": v}
    if dout_seed is not None:
        t["dout"] = _randn((B, S, H, D), _gen(dout_seed), dtype)
    nm = name or "dense_%s_b%d_s%d_h%d_d%d" % (str(dtype).split(".")[-1], B, S, H, D)
    return _problem(nm, dtype, "dense", B, S, Skv, H, Hkv, D,
                    1.0 / math.sqrt(D) if scale is None else float(scale),
                    tuple(window), t)


def varlen(nseq: int = 16, min_len: int = 128, max_len: int = 4096,
           Hq: int = 32, Hkv: int = 8, D: int = 128, dtype=torch.bfloat16,
           window=(-1, 0), len_seed: int = 0, seed: int = 1,
           dout_seed: Optional[int] = 2, lengths=None) -> Attn:
    """Packed THD batch: lengths ~ U[min_len, max_len] (integers, from
    ``len_seed``) unless given, cu_seqlens int32 [nseq + 1]."""
    if lengths is None:
        lengths = torch.randint(min_len, max_len + 1, (nseq,),
                                generator=_gen(len_seed)).tolist()
    lengths = [int(x) for x in lengths]
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    T = int(cu[-1])
    g = _gen(seed)
    q = _randn((T, Hq, D), g, dtype)
    k = _randn((T, Hkv, D), g, dtype)
    v = _randn((T, Hkv, D), g, dtype)
    t = {"q": q, "k": k, "v": v}
    if dout_seed is not None:
        t["dout"] = _randn((T, Hq, D), _gen(dout_seed), dtype)
    mx = max(lengths) if lengths else 0
    return _problem("thd_%s_n%d_hq%d_hkv%d_d%d" % (str(dtype).split(".")[-1],
                                                  len(lengths), Hq, Hkv, D),
                    dtype, "thd", len(lengths), mx, mx, Hq, Hkv, D,
                    1.0 / math.sqrt(D), tuple(window), t,
                    cu_seqlens_q=cu, cu_seqlens_kv=cu.clone())


def random_case(seed: int, B=1, Sq=64, Skv=None, Hq=2, Hkv=1, D=64,
                dtype=torch.float16, window=(-1, 0), order="bshd",
                scale=None, with_dout=True) -> Attn:
    """Small dense problem whose q/k/v/dout are laid out in memory in the
    given ``order`` ("bshd", "sbhd" or "bhsd") and exposed as (b, s, h, d)
    views, so the same values arrive with different strides."""
    Skv = Sq if Skv is None else Skv
    g = _gen(seed)
    perm = {"bshd": (0, 1, 2, 3), "sbhd": (1, 0, 2, 3), "bhsd": (0, 2, 1, 3)}[order]
    inv = [perm.index(i) for i in range(4)]
    bases, views = {}, {}
    for n, (s, h) in (("q", (Sq, Hq)), ("k", (Skv, Hkv)), ("v", (Skv, Hkv)),
                      ("dout", (Sq, Hq))):
        if n == "dout" and not with_dout:
            continue
        logical = _randn((B, s, h, D), g, dtype)
        stored = logical.permute(*perm).contiguous()
        bview = stored.permute(*inv)
        bases[n] = stored
        views[n] = (n, tuple(bview.shape), tuple(bview.stride()), 0)
    return Attn("random_%s_%d" % (order, seed), dtype, "dense", B, Sq, Skv, Hq,
                Hkv, D, 1.0 / math.sqrt(D) if scale is None else float(scale),
                tuple(window), bases, views)
