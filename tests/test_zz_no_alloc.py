"""attn_bwd_noalloc: the backward pass for callers that cannot allocate
device memory (code holding only tensor pointers, or code that must not
allocate after its set-up).  It uses the library's fixed scratch array
instead of a caller workspace; these tests check it against the float64
oracle and against attn_bwd, on two calls in a row (the second call must not
see the first call's leftovers).  The refusal of problems larger than the
scratch needs no GPU and is tested with the C-ABI checks on the CPU.
Collected last so that a stop at the first failure has already run every
other test."""
import numpy as np
import pytest
import torch

import scaled_dot_product_03_gb300 as gb
from scaled_dot_product_03_gb300 import inputs
from gpu_helpers import GRAD_FLOOR, GRAD_REL, check_bwd, kw

pytestmark = pytest.mark.gpu


def _compare(prob):
    d = prob.to("cuda")
    o, lse = gb.attn_fwd(d.q, d.k, d.v, **kw(d))
    got = gb.attn_bwd_noalloc(d.dout, d.q, d.k, d.v, o, lse, **kw(d))
    ref = gb.attn_bwd(d.dout, d.q, d.k, d.v, o, lse, **kw(d))
    torch.cuda.synchronize()
    gb.check_device_error()
    # against the oracle, at the tolerance of every backward test
    check_bwd(prob, *got)
    # and against the entry point with a caller workspace
    for name, r, g in zip(("dq", "dk", "dv"), ref, got):
        r64, g64 = r.double().cpu().numpy(), g.double().cpu().numpy()
        assert np.all(np.isfinite(g64)), name
        scale = max(float(np.abs(r64).max()), GRAD_FLOOR)
        err = float(np.abs(g64 - r64).max())
        assert err <= GRAD_REL * scale, "%s: %.3g > %.3g * %.3g" % (name, err, GRAD_REL, scale)


def test_noalloc_matches_oracle_on_two_calls_in_a_row():
    # first call: dense bf16, grouped heads, causal
    _compare(inputs.dense(2, 700, 8, 128, Hkv=2, seed=21, dout_seed=22))
    # second call: a different THD fp16 problem reusing the same scratch
    _compare(inputs.varlen(lengths=[300, 1, 517, 64], Hq=4, Hkv=1, D=64,
                           dtype=torch.float16, seed=23, dout_seed=24))
