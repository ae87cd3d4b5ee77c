"""GPU parity of the backward through the LSE output (``attn_bwd_dlse``) and
of the LSE-merge backward (``attn_merge_lse_bwd``) against the float64
oracle, and the flex-attention issue's local + global split
("Significant Accuracy Difference between Compiled and Eager Flex
Attention", merge_attn) trained end to end through the library: the
gradients taken back through the merge and through both partial attentions
equal those of full causal attention."""
import numpy as np
import pytest
import torch

import oracle
import scaled_dot_product_03_gb300 as gb
from scaled_dot_product_03_gb300 import inputs
from gpu_helpers import GRAD_FLOOR, GRAD_REL, kw, rows_of, run_fwd
from helpers import cu, lse_to_library_layout, packed

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _sync_ok():
    torch.cuda.synchronize()
    gb.check_device_error()


def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64).float() * scale


def _check(name, got, ref, rel=GRAD_REL):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), name
    scale = max(float(np.abs(ref).max()) if ref.size else 0.0, GRAD_FLOOR)
    err = float(np.abs(got - ref).max()) if ref.size else 0.0
    assert err <= rel * scale, "%s max-abs error %.3g > %.3g * %.3g" % (name, err, rel, scale)


_CASES = {
    "bf16_d128_causal_gqa": lambda: inputs.dense(2, 300, 4, 128, Hkv=2, seed=3, dout_seed=4),
    "fp16_d64_window": lambda: inputs.dense(1, 257, 2, 64, dtype=torch.float16, Hkv=1,
                                            window=(40, 0), seed=5, dout_seed=6),
    "fp32_d64_full": lambda: inputs.dense(1, 200, 2, 64, dtype=torch.float32, window=(-1, -1),
                                          seed=7, dout_seed=8),
    "thd_bf16_d128": lambda: inputs.varlen(lengths=[300, 1, 517, 64], Hq=4, Hkv=2, D=128,
                                           seed=9, dout_seed=10),
}


@pytest.mark.parametrize("case,det", [("bf16_d128_causal_gqa", False), ("bf16_d128_causal_gqa", True),
                                      ("fp16_d64_window", False), ("fp32_d64_full", False),
                                      ("thd_bf16_d128", False), ("thd_bf16_d128", True)])
def test_bwd_with_lse_gradient(case, det):
    prob = _CASES[case]()
    d = prob.to(DEV)
    o, lse = run_fwd(d)
    dl_rows = _rand((prob.total_q, prob.Hq), 77).double().numpy()
    dlse = torch.tensor(np.ascontiguousarray(lse_to_library_layout(prob, dl_rows)),
                        dtype=torch.float32, device=DEV)
    got = gb.attn_bwd(d.dout, d.q, d.k, d.v, o, lse, dlse=dlse, deterministic=det, **kw(d))
    _sync_ok()
    cq, ck = cu(prob)
    ref = oracle.attn_bwd(packed(prob, "q"), packed(prob, "k"), packed(prob, "v"),
                          packed(prob, "dout"), cq, ck, prob.scale, prob.window, dlse=dl_rows)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        _check(name, rows_of(prob, g), r)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_merge_backward_matches_oracle(dtype):
    B, S, H, D = 2, 100, 3, 64
    o1, o2, dout = (_rand((B, S, H, D), s).to(dtype) for s in (11, 12, 13))
    l1, l2 = _rand((B, H, S), 14, 2.0), _rand((B, H, S), 15, 2.0)
    l1[0, 0, :5] = -float("inf")       # left side empty
    l2[0, 0, 3:8] = -float("inf")      # right side empty (3, 4: both)
    dlse = _rand((B, H, S), 16)
    got = gb.attn_merge_lse_bwd(o1.to(DEV), l1.to(DEV), o2.to(DEV), l2.to(DEV), dout.to(DEV),
                                dlse.to(DEV))
    _sync_ok()
    bh = lambda t: t.double().permute(0, 2, 1, 3).numpy()   # [B, H, S, D] like lse
    r_do1, r_dl1, r_do2, r_dl2 = oracle.merge_lse_bwd(bh(o1), l1.double().numpy(), bh(o2),
                                                      l2.double().numpy(), bh(dout),
                                                      dlse.double().numpy())
    rel = {torch.float16: 5e-3, torch.bfloat16: 1e-2, torch.float32: 1e-5}[dtype]
    _check("do1", bh(got[0].cpu()), r_do1, rel)
    _check("do2", bh(got[2].cpu()), r_do2, rel)
    _check("dlse1", got[1].cpu().double().numpy(), r_dl1, 1e-4)
    _check("dlse2", got[3].cpu().double().numpy(), r_dl2, 1e-4)
    # empty sides receive exact zeros
    assert torch.all(got[0][0, :5, 0] == 0) and torch.all(got[1][0, 0, :5] == 0)
    assert torch.all(got[2][0, 3:8, 0] == 0) and torch.all(got[3][0, 0, 3:8] == 0)


@pytest.mark.parametrize("which", ["page3_fp32", "bf16_d128"])
def test_local_global_split_trains_like_causal(which):
    if which == "page3_fp32":
        prob, band = inputs.page3(), 64
    else:
        prob, band = inputs.dense(1, 1024, 4, 128, seed=21, dout_seed=22), 100
    prob.window = (-1, 0)
    d = prob.to(DEV)
    scale, sh = d.scale, band + 1
    o_loc, l_loc = gb.attn_fwd(d.q, d.k, d.v, scale=scale, window=(band, 0))
    qg = d.q[:, sh:]
    o_glb, l_glb = gb.attn_fwd(qg, d.k, d.v, scale=scale, window=(-1, 0))
    l_lt = l_loc[:, :, sh:].contiguous()
    # gradients of a loss on the merged O and LSE
    dO = d.dout
    dL = _rand(tuple(l_loc.shape), 23).to(DEV)
    do_lt, dl_lt, do_g, dl_g = gb.attn_merge_lse_bwd(o_loc[:, sh:], l_lt, o_glb, l_glb,
                                                     dO[:, sh:].contiguous(),
                                                     dL[:, :, sh:].contiguous())
    do_l = torch.cat([dO[:, :sh], do_lt], dim=1)
    dl_l = torch.cat([dL[:, :, :sh], dl_lt], dim=2).contiguous()
    dq_l, dk_l, dv_l = gb.attn_bwd(do_l, d.q, d.k, d.v, o_loc, l_loc, scale=scale,
                                   window=(band, 0), dlse=dl_l)
    dq_g, dk_g, dv_g = gb.attn_bwd(do_g, qg, d.k, d.v, o_glb, l_glb, scale=scale,
                                   window=(-1, 0), dlse=dl_g)
    _sync_ok()
    dq = dq_l.double()
    dq[:, sh:] += dq_g.double()
    dk, dv = dk_l.double() + dk_g.double(), dv_l.double() + dv_g.double()
    cq, ck = cu(prob)
    dl_rows = dL.cpu().double().permute(0, 2, 1).reshape(-1, prob.Hq).numpy()
    ref = oracle.attn_bwd(packed(prob, "q"), packed(prob, "k"), packed(prob, "v"),
                          packed(prob, "dout"), cq, ck, prob.scale, (-1, 0), dlse=dl_rows)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        _check(name, g.cpu().numpy().reshape(r.shape), r)
