"""Pins of the float64 oracle against facts fixed by the pages and by the
mathematics, independent of the oracle's own code path.  CPU only.

Each test names what it pins; together they are chosen so that a plausible
slip anywhere in the oracle (a wrong scale, a dropped term of the softmax
gradient, a swapped head index, an off-by-one in the mask, a wrong log base)
fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from scaled_dot_product_03_gb300 import inputs
from helpers import cu, oracle_bwd, oracle_fwd, packed

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng


def _rand(shape, seed):
    return rng(seed).standard_normal(shape)


def _dense(B, Sq, Skv, Hq, Hkv, D, seed=0):
    q = _rand((B * Sq, Hq, D), seed)
    k = _rand((B * Skv, Hkv, D), seed + 1)
    v = _rand((B * Skv, Hkv, D), seed + 2)
    return q, k, v, oracle.dense_cu(B, Sq), oracle.dense_cu(B, Skv)


# -- 1. identical V rows: the output is that row, for any mask and scale ----

@pytest.mark.parametrize("window", [(-1, -1), (-1, 0), (3, 0), (2, 5)])
def test_identical_value_rows_return_that_row(window):
    q, k, v, cq, ck = _dense(2, 9, 9, 4, 2, 8, seed=1)
    c = _rand((2, 8), 7)
    v[:] = np.repeat(c[None], v.shape[0], 0)  # every key row of head h: c[h]
    o, lse = oracle.attn_fwd(q, k, v, cq, ck, 0.37, window)
    for h in range(4):
        np.testing.assert_allclose(o[:, h, :], np.broadcast_to(c[h // 2], o[:, h, :].shape),
                                   rtol=0, atol=1e-14)


# -- 2. a single visible key: o = v_j and LSE = scale <q, k_j> -----------------

def test_single_visible_key():
    q, k, v, cq, ck = _dense(1, 6, 6, 2, 2, 8, seed=3)
    scale = 0.3
    o, lse = oracle.attn_fwd(q, k, v, cq, ck, scale, (-1, 0))
    # causal row 0 sees only key 0
    np.testing.assert_allclose(o[0], v[0], atol=1e-15)
    np.testing.assert_allclose(lse[0], scale * np.einsum("hd,hd->h", q[0], k[0]), atol=1e-14)
    # window (0, 0): every row sees only itself
    o, lse = oracle.attn_fwd(q, k, v, cq, ck, scale, (0, 0))
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse, scale * np.einsum("thd,thd->th", q, k), atol=1e-14)


def test_empty_rows_give_zero_and_minus_inf():
    # window (0, 0) with Skv < Sq: rows i >= Skv see nothing
    q, k, v, cq, ck = _dense(1, 6, 3, 1, 1, 4, seed=5)
    o, lse = oracle.attn_fwd(q, k, v, cq, ck, 1.0, (0, 0))
    assert np.all(o[3:] == 0) and np.all(np.isneginf(lse[3:]))
    assert np.all(np.isfinite(lse[:3]))


# -- 3. library routine: torch's float64 CPU SDPA and autograd ----------------

def _torch_ref(q, k, v, dout, Sq, Skv, B, scale, window):
    """torch.nn.functional.scaled_dot_product_attention on float64 CPU
    tensors with an explicit boolean mask; gradients by autograd."""
    Hq, Hkv, D = q.shape[1], k.shape[1], q.shape[2]
    G = Hq // Hkv
    tq = torch.tensor(q).reshape(B, Sq, Hq, D).transpose(1, 2).requires_grad_()
    tk = torch.tensor(k).reshape(B, Skv, Hkv, D).transpose(1, 2).requires_grad_()
    tv = torch.tensor(v).reshape(B, Skv, Hkv, D).transpose(1, 2).requires_grad_()
    i = torch.arange(Sq)[:, None]
    j = torch.arange(Skv)[None, :]
    mask = torch.ones(Sq, Skv, dtype=torch.bool)
    if window[0] >= 0:
        mask &= j >= i - window[0]
    if window[1] >= 0:
        mask &= j <= i + window[1]
    out = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(G, 1), tv.repeat_interleave(G, 1),
        attn_mask=mask, scale=scale)
    out.backward(torch.tensor(dout).reshape(B, Sq, Hq, D).transpose(1, 2))
    back = lambda t: t.transpose(1, 2).reshape(-1, t.shape[1], D).detach().numpy()
    return back(out), back(tq.grad), back(tk.grad), back(tv.grad)


@pytest.mark.parametrize("B,Sq,Skv,Hq,Hkv,D,window,scale", [
    (2, 7, 7, 4, 1, 8, (-1, 0), 0.35),
    (1, 13, 13, 2, 2, 16, (-1, -1), 0.25),
    (1, 11, 17, 6, 2, 8, (-1, 0), 0.5),   # Sq != Skv, top-left causal
    (2, 12, 12, 3, 3, 4, (4, 0), 1.0),    # sliding window
    (1, 10, 10, 2, 1, 8, (2, 3), 0.7),    # two-sided window
])
def test_matches_torch_sdpa_float64(B, Sq, Skv, Hq, Hkv, D, window, scale):
    q, k, v, cq, ck = _dense(B, Sq, Skv, Hq, Hkv, D, seed=11)
    dout = _rand(q.shape, 99)
    o_ref, dq_ref, dk_ref, dv_ref = _torch_ref(q, k, v, dout, Sq, Skv, B, scale, window)
    o, lse = oracle.attn_fwd(q, k, v, cq, ck, scale, window)
    dq, dk, dv = oracle.attn_bwd(q, k, v, dout, cq, ck, scale, window)
    for a, b in ((o, o_ref), (dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)
    # LSE against torch.logsumexp of the masked scaled scores
    Hk = Hkv
    G = Hq // Hk
    for b in range(B):
        for h in range(Hq):
            s = scale * q[b * Sq:(b + 1) * Sq, h] @ k[b * Skv:(b + 1) * Skv, h // G].T
            i = np.arange(Sq)[:, None]
            j = np.arange(Skv)[None, :]
            m = np.ones_like(s, dtype=bool)
            if window[0] >= 0:
                m &= j >= i - window[0]
            if window[1] >= 0:
                m &= j <= i + window[1]
            ref = torch.logsumexp(torch.tensor(np.where(m, s, -np.inf)), dim=1).numpy()
            np.testing.assert_allclose(lse[b * Sq:(b + 1) * Sq, h], ref, rtol=1e-12, atol=1e-12)


# -- 4. finite differences: the backward is the derivative of the forward ----

@pytest.mark.parametrize("window", [(-1, -1), (-1, 0), (1, 1)])
def test_gradients_match_central_differences(window):
    q, k, v, cq, ck = _dense(1, 5, 5, 2, 1, 4, seed=21)
    dout = _rand(q.shape, 22)
    scale = 0.6
    dq, dk, dv = oracle.attn_bwd(q, k, v, dout, cq, ck, scale, window)

    def f(q_, k_, v_):
        o, _ = oracle.attn_fwd(q_, k_, v_, cq, ck, scale, window)
        return float(np.sum(o * dout))

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            fp = f(args["q"], args["k"], args["v"])
            args[name] = xm
            fm = f(args["q"], args["k"], args["v"])
            fd[idx] = (fp - fm) / (2 * h)
        err = np.abs(fd - g).max() / max(1.0, np.abs(g).max())
        assert err < 1e-6, (name, err)


# -- 5. closed form of the page-3 workload ------------------------------------

def test_page3_closed_form():
    """Every weight and bias of the page's projection is 0.1, so token t's
    q, k and v rows are the constant vector c_t * 1 (c_t = the fp32-rounded
    projection of x_t).  With D = 64 and scale 1/8 the scores are
    s_tu = 8 c_t c_u, the same for every head, and output, LSE and gradients
    (dO = ones) follow from 1-D sums over u."""
    prob = inputs.page3()
    q, k, v, dout = (packed(prob, n) for n in ("q", "k", "v", "dout"))
    cq, ck = cu(prob)
    c = q[:, 0, 0]
    assert np.all(q == c[:, None, None]) and np.all(k == q) and np.all(v == q)
    D = prob.D
    s = prob.scale * D * np.outer(c, c)                   # [t, u]
    m = s.max(axis=1, keepdims=True)
    lse_cf = (m + np.log(np.exp(s - m).sum(axis=1, keepdims=True)))[:, 0]
    p = np.exp(s - lse_cf[:, None])
    o_cf = p @ c                                          # o_t (every column)
    dP = D * c[None, :]                                   # <1, v_u> = D c_u
    dS = p * (dP - (p * dP).sum(axis=1, keepdims=True))
    dq_cf = prob.scale * dS @ c
    dk_cf = prob.scale * dS.T @ c
    dv_cf = p.sum(axis=0)                                 # sum_t p_tu * 1

    o, lse = oracle.attn_fwd(q, k, v, cq, ck, prob.scale, prob.window)
    dq, dk, dv = oracle.attn_bwd(q, k, v, dout, cq, ck, prob.scale, prob.window)
    H = prob.Hq
    tol = dict(rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(o, np.broadcast_to(o_cf[:, None, None], o.shape), **tol)
    np.testing.assert_allclose(lse, np.broadcast_to(lse_cf[:, None], (len(c), H)), **tol)
    np.testing.assert_allclose(dq, np.broadcast_to(dq_cf[:, None, None], dq.shape), **tol)
    np.testing.assert_allclose(dk, np.broadcast_to(dk_cf[:, None, None], dk.shape), **tol)
    np.testing.assert_allclose(dv, np.broadcast_to(dv_cf[:, None, None], dv.shape), **tol)
    # the page's remark that the scores are extreme: |s| reaches the hundreds
    assert np.abs(s).max() > 100


# -- 6. merge of disjoint key sets equals the full attention ------------------

def test_merge_local_global_equals_causal():
    """Page 3's v1 split: a sliding-window-causal part (q - kv <= band) over
    all rows and a causal part on the query rows shifted by band + 1, whose
    visible keys are exactly those with q - kv > band; merge_attn of the two
    on the shifted rows, the local part alone on the first band + 1 rows,
    equals full causal attention."""
    S, H, D, band, scale = 40, 3, 8, 6, 0.4
    q, k, v, cq, ck = _dense(1, S, S, H, H, D, seed=31)
    o_full, lse_full = oracle.attn_fwd(q, k, v, cq, ck, scale, (-1, 0))
    o_loc, lse_loc = oracle.attn_fwd(q, k, v, cq, ck, scale, (band, 0))
    sh = band + 1
    o_glb, lse_glb = oracle.attn_fwd(q[sh:], k, v, np.array([0, S - sh]), ck,
                                     scale, (-1, 0))
    o_m, lse_m = oracle.merge_lse(o_loc[sh:], lse_loc[sh:], o_glb, lse_glb)
    o = np.concatenate([o_loc[:sh], o_m])
    lse = np.concatenate([lse_loc[:sh], lse_m])
    np.testing.assert_allclose(o, o_full, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse_full, rtol=1e-12, atol=1e-13)


def test_merge_is_order_independent_ring():
    """Ring attention over key chunks does not depend on the visiting order
    ("Ring attention doesn't care the order of iteration"): partials over
    three disjoint key chunks merged in any order give the full result."""
    S, H, D, scale = 24, 2, 8, 0.5
    q, k, v, cq, ck = _dense(1, S, S, H, H, D, seed=41)
    full = oracle.attn_fwd(q, k, v, cq, ck, scale, (-1, -1))
    edges = [0, 5, 14, 24]
    parts = []
    for a, b in zip(edges[:-1], edges[1:]):
        parts.append(oracle.attn_fwd(q, k[a:b], v[a:b], cq, np.array([0, b - a]),
                                     scale, (-1, -1)))
    for order in ([0, 1, 2], [2, 0, 1], [1, 2, 0]):
        o, lse = parts[order[0]]
        for i in order[1:]:
            o, lse = oracle.merge_lse(o, lse, *parts[i])
        np.testing.assert_allclose(o, full[0], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, full[1], rtol=1e-12, atol=1e-13)


def test_merge_with_empty_sides():
    o1 = _rand((4, 3), 1)
    lse1 = np.array([0.3, -np.inf, 2.0, -np.inf])
    o2 = _rand((4, 3), 2)
    lse2 = np.array([-np.inf, 1.5, 2.0, -np.inf])
    o, lse = oracle.merge_lse(o1, lse1, o2, lse2)
    np.testing.assert_allclose(o[0], o1[0])
    np.testing.assert_allclose(o[1], o2[1])
    np.testing.assert_allclose(o[2], 0.5 * (o1[2] + o2[2]))
    assert lse[0] == 0.3 and lse[1] == 1.5
    np.testing.assert_allclose(lse[2], 2.0 + math.log(2.0))
    assert np.all(o[3] == 0) and np.isneginf(lse[3])


# -- 6b. gradient through the LSE output and through the merge ---------------
# The flex-attention issue returns the LSE and combines two partial results
# through it (merge_attn); training such a split needs the gradient of a loss
# that reaches the scores through LSE as well as O, and the backward of the
# merge.

def _fd(f, arrays, h=1e-6):
    """Central differences of f(*arrays) with respect to every element."""
    out = []
    for n in range(len(arrays)):
        g = np.zeros_like(arrays[n])
        for idx in np.ndindex(arrays[n].shape):
            xp = [a.copy() for a in arrays]
            xm = [a.copy() for a in arrays]
            xp[n][idx] += h
            xm[n][idx] -= h
            g[idx] = (f(*xp) - f(*xm)) / (2 * h)
        out.append(g)
    return out


@pytest.mark.parametrize("window", [(-1, -1), (-1, 0), (1, 1)])
def test_lse_gradient_matches_central_differences(window):
    q, k, v, cq, ck = _dense(1, 5, 5, 2, 1, 4, seed=61)
    dout = _rand(q.shape, 62)
    dlse = _rand(q.shape[:2], 63)
    scale = 0.6
    dq, dk, dv = oracle.attn_bwd(q, k, v, dout, cq, ck, scale, window, dlse=dlse)

    def f(q_, k_, v_):
        o, lse = oracle.attn_fwd(q_, k_, v_, cq, ck, scale, window)
        return float(np.sum(o * dout) + np.sum(lse * dlse))

    for name, fd, g in zip("qkv", _fd(f, [q, k, v]), (dq, dk, dv)):
        err = np.abs(fd - g).max() / max(1.0, np.abs(g).max())
        assert err < 1e-6, (name, err)


def test_lse_gradient_matches_torch_autograd():
    """The same loss written with torch's softmax and logsumexp (float64,
    autograd), grouped heads and a causal mask."""
    B, S, Hq, Hkv, D, scale = 1, 9, 4, 2, 8, 0.45
    q, k, v, cq, ck = _dense(B, S, S, Hq, Hkv, D, seed=64)
    dout, dlse = _rand(q.shape, 65), _rand(q.shape[:2], 66)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    G = Hq // Hkv
    kk, vv = tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1)   # [S, Hq, D]
    s = scale * torch.einsum("ihd,jhd->hij", tq, kk)
    mask = torch.ones(S, S, dtype=torch.bool).tril()
    s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)                       # [Hq, S]
    o = torch.einsum("hij,jhd->ihd", torch.softmax(s, dim=-1), vv)
    loss = (o * torch.tensor(dout)).sum() + (lse.T * torch.tensor(dlse)).sum()
    loss.backward()
    dq, dk, dv = oracle.attn_bwd(q, k, v, dout, cq, ck, scale, (-1, 0), dlse=dlse)
    for a, t in ((dq, tq), (dk, tk), (dv, tv)):
        np.testing.assert_allclose(a, t.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_merge_backward_matches_central_differences():
    n, D = 6, 3
    o1, o2 = _rand((n, D), 71), _rand((n, D), 72)
    l1, l2 = _rand((n,), 73), _rand((n,), 74) * 2.0
    dout, dlse = _rand((n, D), 75), _rand((n,), 76)
    do1, dl1, do2, dl2 = oracle.merge_lse_bwd(o1, l1, o2, l2, dout, dlse)

    def f(a1, b1, a2, b2):
        o, lse = oracle.merge_lse(a1, b1, a2, b2)
        return float(np.sum(o * dout) + np.sum(lse * dlse))

    for name, fd, g in zip(("o1", "lse1", "o2", "lse2"), _fd(f, [o1, l1, o2, l2]),
                           (do1, dl1, do2, dl2)):
        np.testing.assert_allclose(g, fd, rtol=1e-7, atol=1e-8, err_msg=name)


def test_merge_backward_with_empty_sides():
    """A side without keys gets no gradient; the other side then is the
    merged row itself, so it receives dO unchanged and the LSE gradient as
    is; both sides empty: nothing anywhere."""
    o1, o2, dout = _rand((3, 4), 81), _rand((3, 4), 82), _rand((3, 4), 83)
    l1 = np.array([-np.inf, 0.7, -np.inf])
    l2 = np.array([1.1, -np.inf, -np.inf])
    dlse = np.array([0.3, -0.8, 0.5])
    do1, dl1, do2, dl2 = oracle.merge_lse_bwd(o1, l1, o2, l2, dout, dlse)
    assert np.all(do1[0] == 0) and dl1[0] == 0
    np.testing.assert_allclose(do2[0], dout[0])
    np.testing.assert_allclose(dl2[0], dlse[0])
    assert np.all(do2[1] == 0) and dl2[1] == 0
    np.testing.assert_allclose(do1[1], dout[1])
    np.testing.assert_allclose(dl1[1], dlse[1])
    assert np.all(do1[2] == 0) and np.all(do2[2] == 0) and dl1[2] == 0 and dl2[2] == 0


def test_local_global_split_trains_like_causal():
    """Page 3's v1 split trained end to end: the gradients of a loss on the
    merged O and LSE, taken back through merge_attn and through both partial
    attentions (each with its LSE gradient), equal those of full causal
    attention."""
    S, H, D, band, scale = 40, 3, 8, 6, 0.4
    q, k, v, cq, ck = _dense(1, S, S, H, H, D, seed=91)
    dout, dlse = _rand(q.shape, 92), _rand(q.shape[:2], 93)
    sh = band + 1
    cg = np.array([0, S - sh])
    o_loc, lse_loc = oracle.attn_fwd(q, k, v, cq, ck, scale, (band, 0))
    o_glb, lse_glb = oracle.attn_fwd(q[sh:], k, v, cg, ck, scale, (-1, 0))
    do_lt, dl_lt, do_g, dl_g = oracle.merge_lse_bwd(o_loc[sh:], lse_loc[sh:], o_glb, lse_glb,
                                                    dout[sh:], dlse[sh:])
    do_l = np.concatenate([dout[:sh], do_lt])
    dl_l = np.concatenate([dlse[:sh], dl_lt])
    dq_l, dk_l, dv_l = oracle.attn_bwd(q, k, v, do_l, cq, ck, scale, (band, 0), dlse=dl_l)
    dq_g, dk_g, dv_g = oracle.attn_bwd(q[sh:], k, v, do_g, cg, ck, scale, (-1, 0), dlse=dl_g)
    dq = dq_l.copy()
    dq[sh:] += dq_g
    dq_f, dk_f, dv_f = oracle.attn_bwd(q, k, v, dout, cq, ck, scale, (-1, 0), dlse=dlse)
    for a, b in ((dq, dq_f), (dk_l + dk_g, dk_f), (dv_l + dv_g, dv_f)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)


# -- 7. identities of the softmax gradient -----------------------------------

def test_row_term_equals_dout_dot_out():
    """The definitional row term sum_j p_ij dP_ij equals <dO_i, O_i> (the
    form a fused backward computes), and the backward's LSE is the
    forward's."""
    q, k, v, cq, ck = _dense(2, 9, 9, 4, 2, 8, seed=51)
    dout = _rand(q.shape, 52)
    o, lse = oracle.attn_fwd(q, k, v, cq, ck, 0.4, (-1, 0))
    _, _, _, lse_b, r = oracle.attn_bwd(q, k, v, dout, cq, ck, 0.4, (-1, 0),
                                        want_stats=True)
    np.testing.assert_allclose(r, np.einsum("thd,thd->th", dout, o), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse_b, lse, rtol=0, atol=0)


@pytest.mark.parametrize("window", [(-1, 0), (-1, -1), (3, 1)])
def test_gradient_sums(window):
    """sum_j dS_ij = 0 for every row, hence sum_j dk_j = 0 per kv head and
    sequence; sum_j dv_j = sum of dO over the rows that see some key, over
    the group's query heads; and dq = 0 when all key rows are equal."""
    B, S, Hq, Hkv, D = 2, 8, 4, 2, 6
    q, k, v, cq, ck = _dense(B, S, S, Hq, Hkv, D, seed=61)
    dout = _rand(q.shape, 62)
    dq, dk, dv = oracle.attn_bwd(q, k, v, dout, cq, ck, 0.5, window)
    G = Hq // Hkv
    for b in range(B):
        rows = slice(b * S, (b + 1) * S)
        np.testing.assert_allclose(dk[rows].sum(axis=0), 0, atol=1e-12)
        for hk in range(Hkv):
            want = dout[rows, hk * G:(hk + 1) * G].sum(axis=(0, 1))
            np.testing.assert_allclose(dv[rows, hk].sum(axis=0), want, atol=1e-12)
    k_eq = np.repeat(k[:1], k.shape[0], 0)
    dq, _, _ = oracle.attn_bwd(q, k_eq, v, dout, cq, ck, 0.5, window)
    np.testing.assert_allclose(dq, 0, atol=1e-13)


# -- 8. batch and packing independence ----------------------------------------

def test_batch_and_packing_independence():
    """Each sequence of a batch or of a THD pack is computed on its own:
    the packed result equals the per-sequence results, and permuting the
    sequences permutes the results."""
    lens = [5, 9, 1, 7]
    Hq, Hkv, D = 4, 2, 8
    T = sum(lens)
    q, k, v = _rand((T, Hq, D), 71), _rand((T, Hkv, D), 72), _rand((T, Hkv, D), 73)
    dout = _rand((T, Hq, D), 74)
    cuv = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    o, lse = oracle.attn_fwd(q, k, v, cuv, cuv, 0.3, (-1, 0))
    g = oracle.attn_bwd(q, k, v, dout, cuv, cuv, 0.3, (-1, 0))
    for b, (a, e) in enumerate(zip(cuv[:-1], cuv[1:])):
        one = np.array([0, e - a])
        o1, l1 = oracle.attn_fwd(q[a:e], k[a:e], v[a:e], one, one, 0.3, (-1, 0))
        g1 = oracle.attn_bwd(q[a:e], k[a:e], v[a:e], dout[a:e], one, one, 0.3, (-1, 0))
        np.testing.assert_array_equal(o[a:e], o1)
        np.testing.assert_array_equal(lse[a:e], l1)
        for x, x1 in zip(g, g1):
            np.testing.assert_array_equal(x[a:e], x1)


# -- 9. selections compute exactly the selected outputs ------------------------

def test_row_and_key_selection_match_full():
    q, k, v, cq, ck = _dense(2, 10, 10, 4, 2, 8, seed=81)
    dout = _rand(q.shape, 82)
    o, lse = oracle.attn_fwd(q, k, v, cq, ck, 0.5, (-1, 0))
    dq, dk, dv = oracle.attn_bwd(q, k, v, dout, cq, ck, 0.5, (-1, 0))
    rs = rng(5).random(q.shape[:2]) < 0.3
    ks = rng(6).random(k.shape[:2]) < 0.3
    o_s, lse_s = oracle.attn_fwd(q, k, v, cq, ck, 0.5, (-1, 0), row_sel=rs)
    dq_s, dk_s, dv_s = oracle.attn_bwd(q, k, v, dout, cq, ck, 0.5, (-1, 0),
                                       row_sel=rs, key_sel=ks)
    np.testing.assert_array_equal(o_s[rs], o[rs])
    np.testing.assert_array_equal(lse_s[rs], lse[rs])
    np.testing.assert_array_equal(dq_s[rs], dq[rs])
    np.testing.assert_array_equal(dk_s[ks], dk[ks])
    np.testing.assert_array_equal(dv_s[ks], dv[ks])


# -- 10. the page-1 view layout ------------------------------------------------

def test_page1_views_have_the_printed_strides():
    """The packed qkv split reproduces the strides the issue prints."""
    want = open(os.path.join(GOLDEN, "page1_strides.txt")).read().split("\n")
    want = [ln for ln in want if ln and not ln.startswith("#")]
    strides = tuple(int(x) for x in want[0].split())
    prob = inputs.page1()
    for n in ("q", "k", "v"):
        t = prob.tensor(n)
        sbhd = (t.stride(1), t.stride(0), t.stride(2), t.stride(3))
        assert sbhd == strides, (n, sbhd)
    assert prob.k.storage_offset() == 16 * 64 and prob.v.storage_offset() == 17 * 64


# -- 11. context parallelism over THD (the THD+CP thread) --------------------

def _padded(lengths, multiple):
    pads = [0]
    for L in lengths:
        pads.append(pads[-1] + -(-max(L, 1) // multiple) * multiple)
    return pads


@pytest.mark.parametrize("world", [1, 2, 3, 4])
def test_partitioned_indices_cover_and_balance(world):
    """Every row of the padded buffer belongs to exactly one rank, every rank
    holds the same number of rows, two chunks per sequence, and (the point
    of the split) the same causal work: the sum over its rows of the number
    of keys a row sees under a causal mask."""
    lengths = [8 * world, 24 * world, 2 * world]
    pads = _padded(lengths, 2 * world)
    T = pads[-1]
    parts = [oracle.thd_partitioned_indices(pads, T, world, r) for r in range(world)]
    allrows = np.sort(np.concatenate(parts))
    np.testing.assert_array_equal(allrows, np.arange(T))
    assert len({len(p) for p in parts}) == 1
    work = []
    for p in parts:
        w = 0
        for row in p:
            b = int(np.searchsorted(pads, row, side="right") - 1)
            w += row - pads[b] + 1           # keys seen by this row (causal)
        work.append(w)
    assert len(set(work)) == 1, work


def test_partitioned_indices_within_rank_order_table():
    """The rows each rank holds, in order, written out by hand for two ranks
    and three sequences padded to 8, 4 and 12 rows: every sequence is cut
    into four equal chunks; rank r lists, sequence by sequence, its chunk r
    and then the mirrored chunk 3 - r (the reading of the THD+CP thread's
    load-balanced split used throughout)."""
    pads = [0, 8, 12, 24]
    want = {
        0: [0, 1, 6, 7, 8, 11, 12, 13, 14, 21, 22, 23],
        1: [2, 3, 4, 5, 9, 10, 15, 16, 17, 18, 19, 20],
    }
    for rank, rows in want.items():
        got = oracle.thd_partitioned_indices(pads, 24, 2, rank)
        assert got.tolist() == rows, (rank, got.tolist())


@pytest.mark.parametrize("cp", [2, 3])
@pytest.mark.parametrize("causal", [True, False])
def test_ring_attention_equals_full_attention(cp, causal):
    """The ring of partial attentions merged by LSE equals one attention over
    each whole sequence; padding rows stay (0, -inf)."""
    lengths = [37, 1, 64, 0, 50]
    pads = _padded(lengths, 2 * cp)
    T, H, Hkv, D, scale = pads[-1], 4, 2, 8, 0.45
    g = np.random.default_rng(5)
    q, k, v = g.standard_normal((T, H, D)), g.standard_normal((T, Hkv, D)), g.standard_normal((T, Hkv, D))
    cu_l = np.concatenate([[0], np.cumsum(lengths)])
    o, lse = oracle.ring_attention_fwd(q, k, v, cu_l, pads, cp, scale, causal)
    rows = np.concatenate([np.arange(pads[b], pads[b] + L) for b, L in enumerate(lengths)])
    o_full, lse_full = oracle.attn_fwd(q[rows], k[rows], v[rows], cu_l, cu_l, scale,
                                       (-1, 0) if causal else (-1, -1))
    np.testing.assert_allclose(o[rows], o_full, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse[rows], lse_full, rtol=1e-12, atol=1e-13)
    pad_rows = np.setdiff1d(np.arange(T), rows)
    assert np.all(o[pad_rows] == 0) and np.all(np.isneginf(lse[pad_rows]))
