"""Helpers of the GPU parity tests: run the library on a problem, compare
with the oracle.  Tolerances follow the stated bars: fp16 O <= 5e-3, bf16
O <= 1e-2, LSE <= 1e-3, fp32 O <= 1e-4; gradients <= 2e-2 * max|grad|."""
from __future__ import annotations

import numpy as np
import torch

import scaled_dot_product_03_gb300 as gb
from helpers import lse_to_library_layout, oracle_bwd, oracle_fwd, to_f64

O_TOL = {torch.float16: 5e-3, torch.bfloat16: 1e-2, torch.float32: 1e-4}
LSE_TOL = {torch.float16: 1e-3, torch.bfloat16: 1e-3}
# half an ulp of the output type relative to |O| (8 and 11 significant bits)
O_ROUND_REL = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}
# fp32 LSE: 1e-4 plus the rounding of an fp32 number of the LSE's size
# (scores of magnitude ~200 on the page-3 workload make fp32 rounding alone
# reach ~1.4e-4 there), per element
LSE_F32_ABS, LSE_F32_REL = 1e-4, 2.0 ** -20
GRAD_REL = 2e-2
# Gradients that are exactly zero (a row that sees a single key has dS = 0)
# are compared against this floor of max|grad| instead of 0.
GRAD_FLOOR = 1e-3


def kw(prob):
    k = dict(scale=prob.scale, window=prob.window)
    if prob.layout == "thd":
        k.update(cu_seqlens_q=prob.cu_seqlens_q, cu_seqlens_kv=prob.cu_seqlens_kv,
                 max_seqlen_q=prob.Sq, max_seqlen_kv=prob.Skv)
    return k


def run_fwd(dprob):
    o, lse = gb.attn_fwd(dprob.q, dprob.k, dprob.v, **kw(dprob))
    return o, lse


def run_bwd(dprob, o, lse, deterministic=False):
    return gb.attn_bwd(dprob.dout, dprob.q, dprob.k, dprob.v, o, lse, deterministic=deterministic,
                       **kw(dprob))


def rows_of(prob, t):
    """Library output ``[B,S,H,D]`` / ``[T,H,D]`` -> float64 ``[rows, H, D]``."""
    a = to_f64(t)
    return a.reshape(-1, a.shape[-2], a.shape[-1])


def lse_rows(prob, lse):
    a = lse.detach().cpu().to(torch.float64).numpy()
    if prob.layout == "dense":
        return a.transpose(0, 2, 1).reshape(-1, prob.Hq)
    return a.T


def max_abs(a, b, mask=None):
    with np.errstate(invalid="ignore"):  # -inf - -inf outside the mask
        d = np.abs(a - b)
    if mask is not None:
        d = d[mask]
    return float(d.max()) if d.size else 0.0


def check_fwd(prob, o, lse, row_sel=None, o_tol=None, lse_tol=None):
    """Compare (o, lse) of the library with the oracle on all rows (or the
    selected (row, head) pairs).  Returns the errors."""
    ro, rl = oracle_fwd(prob, row_sel=row_sel)
    go, gl = rows_of(prob, o), lse_rows(prob, lse)
    sel = np.ones(rl.shape, bool) if row_sel is None else row_sel.astype(bool)
    # rows without any visible key: exactly 0 and -inf
    empty = sel & np.isneginf(rl)
    assert np.all(np.isneginf(gl[empty])), "empty rows must have lse = -inf"
    assert np.all(go[empty] == 0), "empty rows must have o = 0"
    full = sel & ~np.isneginf(rl)
    assert np.all(np.isfinite(gl[full])) and np.all(np.isfinite(go[full]))
    e_o = max_abs(go, ro, full)
    e_l = max_abs(gl, rl, full)
    o_tol = O_TOL[prob.dtype] if o_tol is None else o_tol
    if e_o > o_tol and prob.dtype in O_ROUND_REL:
        # The 16-bit output's own rounding: a row of large |O| (few visible
        # keys) can exceed the flat bound by rounding alone, as the stated
        # reading of the tolerance allows; such a row must stay within the
        # flat bound plus the output type's half-ulp, |err| <= tol + rel |O|,
        # and the raw max-abs is reported beside it.
        with np.errstate(invalid="ignore"):
            d = np.abs(go - ro)[full]
            bound = o_tol + O_ROUND_REL[prob.dtype] * np.abs(ro[full])
        worst = float((d - bound).max())
        print("O max-abs %.4g above %.3g; within tol + half-ulp of |O| (margin %.3g)" % (e_o, o_tol, -worst))
        assert worst <= 0, "O error exceeds %.3g + %.3g |O| by %.3g (max-abs %.3g)" % (
            o_tol, O_ROUND_REL[prob.dtype], worst, e_o)
    else:
        assert e_o <= o_tol, "O max-abs error %.3g > %.3g" % (e_o, o_tol)
    if lse_tol is None and prob.dtype == torch.float32:
        with np.errstate(invalid="ignore"):
            d = np.abs(gl - rl)[full]
            bound = LSE_F32_ABS + LSE_F32_REL * np.abs(rl[full])
        worst = float((d - bound).max()) if d.size else -1.0
        assert worst <= 0, "fp32 LSE error exceeds 1e-4 + 2^-20 |LSE| by %.3g" % worst
    else:
        lse_tol = LSE_TOL[prob.dtype] if lse_tol is None else lse_tol
        assert e_l <= lse_tol, "LSE max-abs error %.3g > %.3g" % (e_l, lse_tol)
    return e_o, e_l


def check_bwd(prob, dq, dk, dv, row_sel=None, key_sel=None, rel=GRAD_REL):
    rdq, rdk, rdv = oracle_bwd(prob, row_sel=row_sel, key_sel=key_sel)
    errs = {}
    for name, g, r, sel in (("dq", dq, rdq, row_sel), ("dk", dk, rdk, key_sel),
                            ("dv", dv, rdv, key_sel)):
        ga = rows_of(prob, g)
        m = np.ones(ga.shape[:2], bool) if sel is None else sel.astype(bool)
        ref = r[m]
        scale = max(float(np.abs(ref).max()) if ref.size else 0.0, GRAD_FLOOR)
        err = max_abs(ga, r, m)
        assert np.all(np.isfinite(ga[m])), name
        assert err <= rel * scale, "%s max-abs error %.3g > %.3g * %.3g" % (name, err, rel, scale)
        errs[name] = (err, scale)
    return errs


def sample_rows(prob, n_per_head, seed=0):
    """Random (row, head) selection of ``n_per_head`` rows per head, always
    including each sequence's first and last row."""
    rng = np.random.default_rng(seed)
    T = prob.total_q
    sel = np.zeros((T, prob.Hq), np.uint8)
    for h in range(prob.Hq):
        sel[rng.choice(T, size=min(n_per_head, T), replace=False), h] = 1
    starts = [0]
    if prob.layout == "thd":
        starts = prob.cu_seqlens_q.cpu().tolist()
    else:
        starts = [b * prob.Sq for b in range(prob.B + 1)]
    for a, e in zip(starts[:-1], starts[1:]):
        if e > a:
            sel[a, :] = 1
            sel[e - 1, :] = 1
    return sel


def sample_keys(prob, units, n_per_unit, seed=0):
    """Key selection: ``n_per_unit`` keys (plus first/last) of each (sequence,
    kv head) unit in ``units``."""
    rng = np.random.default_rng(seed)
    sel = np.zeros((prob.total_kv, prob.Hkv), np.uint8)
    if prob.layout == "thd":
        cu = prob.cu_seqlens_kv.cpu().tolist()
    else:
        cu = [b * prob.Skv for b in range(prob.B + 1)]
    for b, hk in units:
        a, e = cu[b], cu[b + 1]
        if e <= a:
            continue
        idx = rng.choice(np.arange(a, e), size=min(n_per_unit, e - a), replace=False)
        sel[idx, hk] = 1
        sel[a, hk] = sel[e - 1, hk] = 1
    return sel
