"""attn_bwd_noalloc: the backward pass for callers that cannot allocate
device memory (code holding only tensor pointers, or code that must not
allocate after its set-up).  It uses the library's fixed scratch array
instead of a caller workspace; these tests check that it gives what
attn_bwd gives, on two calls in a row (the second call must not see the
first call's leftovers), and that problems larger than the scratch are
refused.  Collected last so that a stop at the first failure has already
run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import scaled_dot_product_03_gb300 as gb
from scaled_dot_product_03_gb300 import _lib, inputs
from gpu_helpers import GRAD_FLOOR, GRAD_REL, kw

pytestmark = pytest.mark.gpu


def _compare(prob):
    d = prob.to("cuda")
    o, lse = gb.attn_fwd(d.q, d.k, d.v, **kw(d))
    ref = gb.attn_bwd(d.dout, d.q, d.k, d.v, o, lse, **kw(d))
    got = gb.attn_bwd_noalloc(d.dout, d.q, d.k, d.v, o, lse, **kw(d))
    torch.cuda.synchronize()
    gb.check_device_error()
    for name, r, g in zip(("dq", "dk", "dv"), ref, got):
        r64, g64 = r.double().cpu().numpy(), g.double().cpu().numpy()
        assert np.all(np.isfinite(g64)), name
        scale = max(float(np.abs(r64).max()), GRAD_FLOOR)
        err = float(np.abs(g64 - r64).max())
        assert err <= GRAD_REL * scale, "%s: %.3g > %.3g * %.3g" % (name, err, GRAD_REL, scale)


def test_noalloc_matches_attn_bwd_on_two_calls_in_a_row():
    # first call: dense bf16, grouped heads, causal
    _compare(inputs.dense(2, 700, 8, 128, Hkv=2, seed=21, dout_seed=22))
    # second call: a different THD fp16 problem reusing the same scratch
    _compare(inputs.varlen(lengths=[300, 1, 517, 64], Hq=4, Hkv=1, D=64,
                           dtype=torch.float16, seed=23, dout_seed=24))


def test_noalloc_refuses_problems_larger_than_its_scratch():
    lib = _lib.load()
    p = _lib.AttnParams()
    p.dtype, p.layout = _lib.ATTN_BF16, _lib.ATTN_LAYOUT_DENSE4D
    # 64 x 65536 rows x 16 heads of fp32 row terms: 256 MiB of scratch
    p.B, p.Sq, p.Skv, p.Hq, p.Hkv, p.D = 64, 65536, 65536, 16, 16, 128
    p.scale, p.window_left, p.window_right = 0.125, -1, 0
    assert lib.attn_bwd_workspace_size(ctypes.byref(p)) > _lib.NOALLOC_SCRATCH_BYTES
    t = _lib.AttnTensor()
    t.ptr = 4096
    t.stride[:] = (65536 * 2048, 2048, 128, 1)
    st = lib.attn_bwd_noalloc(ctypes.byref(p), t, t, t, t, t, 4096, t, t, t, None)
    assert st == _lib.ATTN_ERR_UNSUPPORTED
    assert b"scratch" in lib.attn_last_error_string()
