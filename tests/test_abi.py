"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from scaled_dot_product_03_gb300 import _lib
from scaled_dot_product_03_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbattn.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return _lib.load()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"GBATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def test_header_declares_the_binding_exports():
    assert sorted(declared_symbols()) == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    # and nothing of the internal namespace leaks out
    out = os.popen("nm -D --defined-only %s" % _lib.LIB_PATH).read()
    exported = set(re.findall(r" T (\w+)", out))
    assert exported >= set(declared_symbols())
    assert not [s for s in exported if "gbattn" in s]


def test_params_struct_matches_header():
    """The ctypes attn_params has the header's fields, in the header's order."""
    with open(os.path.join(ROOT, "include", "gbattn.h")) as f:
        text = f.read()
    body = text[text.index("typedef struct {\n    attn_dtype dtype;"):]
    body = body[:body.index("} attn_params;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = []
    for decl in body.split(";")[:-1]:
        decl = decl.strip().split("{", 1)[-1].strip()
        parts = decl.replace("*", " ").split()
        names += [n.strip(",") for n in parts[1:] if n.strip(",") and n != "const"
                  and n not in ("int32_t", "int", "float")]
    assert names == [f[0] for f in _lib.AttnParams._fields_]


def _params(**kw):
    p = _lib.AttnParams()
    p.dtype, p.layout = _lib.ATTN_BF16, _lib.ATTN_LAYOUT_DENSE4D
    p.B, p.Sq, p.Skv, p.Hq, p.Hkv, p.D = 2, 128, 128, 4, 2, 64
    p.scale, p.window_left, p.window_right = 0.125, -1, 0
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def _t(ptr=4096, strides=(32768, 256, 64, 1)):
    t = _lib.AttnTensor()
    t.ptr = ptr
    t.stride[:] = strides
    return t


@pytest.mark.parametrize("kw,status", [
    (dict(deterministic=2), _lib.ATTN_ERR_INVALID_ARG),
    (dict(cu_seqlens_q_padded=4096), _lib.ATTN_ERR_INVALID_ARG),   # padding needs THD
    (dict(D=80), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(D=0), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(Hq=3, Hkv=2), _lib.ATTN_ERR_INVALID_ARG),
    (dict(Hkv=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(window_left=-2), _lib.ATTN_ERR_INVALID_ARG),
    (dict(dtype=7), _lib.ATTN_ERR_INVALID_ARG),
    (dict(layout=5), _lib.ATTN_ERR_INVALID_ARG),
    (dict(B=-1), _lib.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), _lib.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(scale=-0.5), _lib.ATTN_ERR_INVALID_ARG),
    (dict(layout=_lib.ATTN_LAYOUT_THD), _lib.ATTN_ERR_INVALID_ARG),  # no cu_seqlens
])
def test_invalid_params_rejected_without_launch(lib, kw, status):
    p = _params(**kw)
    st = lib.attn_fwd(ctypes.byref(p), _t(), _t(), _t(), _t(), 4096, None)
    assert st == status
    assert lib.attn_last_error_string()
    assert lib.attn_bwd_workspace_size(ctypes.byref(p)) == 0


@pytest.mark.parametrize("tensor_kw,status", [
    (dict(ptr=4096 + 2), _lib.ATTN_ERR_UNSUPPORTED),               # not 16-byte aligned
    (dict(strides=(32768, 260, 65, 1)), _lib.ATTN_ERR_UNSUPPORTED),  # strides not 16 B
    (dict(strides=(32768, 256, 64, 2)), _lib.ATTN_ERR_UNSUPPORTED),  # d not contiguous
    (dict(ptr=0), _lib.ATTN_ERR_INVALID_ARG),
])
def test_bad_views_rejected_without_copy(lib, tensor_kw, status):
    p = _params()
    st = lib.attn_fwd(ctypes.byref(p), _t(**tensor_kw), _t(), _t(), _t(), 4096, None)
    assert st == status, lib.attn_last_error_string()


def test_empty_problem_is_a_no_op(lib):
    for kw in (dict(B=0), dict(Sq=0)):
        p = _params(**kw)
        assert lib.attn_fwd(ctypes.byref(p), _t(ptr=0), _t(ptr=0), _t(ptr=0), _t(ptr=0),
                            0, None) == _lib.ATTN_OK


def test_workspace_size(lib):
    p = _params()
    n = lib.attn_bwd_workspace_size(ctypes.byref(p))
    rows = p.B * p.Sq
    assert n >= 4 * rows * p.Hq  # row terms
    assert n % 256 == 0
    p32 = _params(dtype=_lib.ATTN_F32)
    assert lib.attn_bwd_workspace_size(ctypes.byref(p32)) >= 4 * rows * p.Hq
    # 16-bit, D = 128: the single pass adds an fp32 dq accumulator, the
    # deterministic form needs the row terms only (one query head per
    # key/value head: no query-head split)
    for dt in (_lib.ATTN_F16, _lib.ATTN_BF16):
        pf = _params(dtype=dt, D=128, Hkv=4)
        # row terms, the accumulator and the 256-byte work-counter block
        assert lib.attn_bwd_workspace_size(ctypes.byref(pf)) >= 4 * rows * pf.Hq * (1 + 128) + 256
        pf.deterministic = 1
        nd = lib.attn_bwd_workspace_size(ctypes.byref(pf))
        assert 4 * rows * pf.Hq <= nd < 4 * rows * pf.Hq + 256
    # grouped heads on a small grid (2 key tiles x 2 key/value heads x 2
    # sequences): the query heads of a group are split in two, and both
    # backward forms add the fp32 partial dK, dV of each split
    for det in (0, 1):
        pg = _params(D=128, Hq=4, Hkv=2, deterministic=det)
        n = lib.attn_bwd_workspace_size(ctypes.byref(pg))
        parts = 2 * 2 * (pg.B * pg.Skv) * pg.Hkv * 128 * 4
        base = 4 * rows * pg.Hq * (1 if det else 1 + 128)
        assert base + parts <= n < base + parts + 512, (det, n)
    pf = _params(dtype=_lib.ATTN_BF16, D=128)
    pf.deterministic = 2
    assert lib.attn_bwd_workspace_size(ctypes.byref(pf)) == 0


def test_lse_gradient_backward_rejects_like_attn_bwd(lib):
    """attn_bwd_dlse validates exactly as attn_bwd (nothing is launched)."""
    t = _t()
    for kw, status in ((dict(deterministic=2), _lib.ATTN_ERR_INVALID_ARG),
                       (dict(D=80), _lib.ATTN_ERR_UNSUPPORTED)):
        p = _params(**kw)
        st = lib.attn_bwd_dlse(ctypes.byref(p), t, t, t, t, t, 4096, 4096, t, t, t, 4096, 1 << 20,
                               None)
        assert st == status, lib.attn_last_error_string()
    p = _params()
    st = lib.attn_bwd_dlse(ctypes.byref(p), t, t, t, t, t, None, 4096, t, t, t, 4096, 1 << 20, None)
    assert st == _lib.ATTN_ERR_INVALID_ARG  # lse missing


def test_merge_backward_rejects_bad_args(lib):
    t, z = _t(), _t(ptr=0)
    args = lambda dt, B, D, do1=t: (dt, B, 4, 2, D, t, 4096, t, 4096, t, None, do1, 4096, t, 4096, None)
    assert lib.attn_merge_lse_bwd(*args(9, 1, 64)) == _lib.ATTN_ERR_INVALID_ARG
    assert lib.attn_merge_lse_bwd(*args(1, 1, 300)) == _lib.ATTN_ERR_UNSUPPORTED
    assert lib.attn_merge_lse_bwd(*args(1, 1, 64, do1=z)) == _lib.ATTN_ERR_INVALID_ARG
    assert lib.attn_merge_lse_bwd(*args(1, 0, 64)) == _lib.ATTN_OK  # empty: nothing to do


def test_merge_rejects_bad_args(lib):
    t = _t()
    assert lib.attn_merge_lse(9, 1, 1, 1, 64, t, 4096, t, 4096, t, 4096, None) == \
        _lib.ATTN_ERR_INVALID_ARG
    assert lib.attn_merge_lse(1, 1, 1, 1, 300, t, 4096, t, 4096, t, 4096, None) == \
        _lib.ATTN_ERR_UNSUPPORTED
    assert lib.attn_merge_lse(1, 0, 5, 1, 64, t, 4096, t, 4096, t, 4096, None) == _lib.ATTN_OK


def test_partitioned_indices_rejects_bad_args(lib):
    f = lib.attn_thd_partitioned_indices
    assert f(4096, 1, 16, 0, 0, 4096, None) == _lib.ATTN_ERR_INVALID_ARG   # world 0
    assert f(4096, 1, 16, 2, 2, 4096, None) == _lib.ATTN_ERR_INVALID_ARG   # rank >= world
    assert f(4096, 1, 18, 4, 0, 4096, None) == _lib.ATTN_ERR_INVALID_ARG   # 18 % 8 != 0
    assert f(None, 1, 16, 2, 0, 4096, None) == _lib.ATTN_ERR_INVALID_ARG   # NULL offsets
    assert f(None, 0, 0, 2, 1, None, None) == _lib.ATTN_OK                 # empty: nothing


def test_thd_row_sums_reject_bad_args(lib):
    """attn_thd_accumulate / attn_thd_store validate before any launch."""
    def tensor(ptr=4096, row=256, head=64):
        t = _lib.AttnTensor()
        t.ptr = ptr
        t.stride[:] = (0, row, head, 1)
        return t
    cu, acc = 4096, 8192
    for fn, call in (("accumulate", lambda dt, T, H, D, t, a, c, B: lib.attn_thd_accumulate(dt, T, H, D, t, a, 1, c, None, B, None)),
                     ("store", lambda dt, T, H, D, t, a, c, B: lib.attn_thd_store(dt, T, H, D, a, t, c, None, B, None))):
        assert call(9, 4, 2, 64, tensor(), acc, cu, 1) == _lib.ATTN_ERR_INVALID_ARG, fn      # dtype
        assert call(1, 4, 2, 12, tensor(), acc, cu, 1) == _lib.ATTN_ERR_INVALID_ARG, fn      # D % 8
        assert call(1, 4, 2, 264, tensor(), acc, cu, 1) == _lib.ATTN_ERR_INVALID_ARG, fn     # D > 256
        assert call(1, -1, 2, 64, tensor(), acc, cu, 1) == _lib.ATTN_ERR_INVALID_ARG, fn     # T < 0
        assert call(1, 4, 2, 64, tensor(), acc, None, 1) == _lib.ATTN_ERR_INVALID_ARG, fn    # cu_seqlens
        assert call(1, 4, 2, 64, tensor(), acc, cu, 0) == _lib.ATTN_ERR_INVALID_ARG, fn      # B
        assert call(1, 4, 2, 64, tensor(ptr=4098), acc, cu, 1) == _lib.ATTN_ERR_INVALID_ARG, fn  # alignment
        assert call(1, 4, 2, 64, tensor(row=252), acc, cu, 1) == _lib.ATTN_ERR_INVALID_ARG, fn   # row stride
        assert call(1, 4, 2, 64, tensor(), 8196, cu, 1) == _lib.ATTN_ERR_INVALID_ARG, fn     # acc alignment
        assert call(1, 0, 2, 64, tensor(), acc, cu, 1) == _lib.ATTN_OK, fn                   # empty: no-op


def test_header_is_c99_and_layout_matches_binding(tmp_path):
    """The header compiles as plain C99 with warnings as errors, and a C
    compiler lays attn_params and attn_tensor out exactly as the ctypes
    binding does (sizes and every field offset)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [f[0] for f in _lib.AttnParams._fields_]
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stddef.h>\n#include <stdio.h>\n#include "gbattn.h"\n'
        "int main(void) {\n"
        '    printf("attn_params %zu\\n", sizeof(attn_params));\n'
        '    printf("attn_tensor %zu %zu\\n", sizeof(attn_tensor), offsetof(attn_tensor, stride));\n'
        + "".join('    printf("%s %%zu\\n", offsetof(attn_params, %s));\n' % (f, f) for f in fields)
        + "    return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.check_call([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                           str(src), "-o", str(exe)])
    out = dict(line.split(" ", 1) for line in subprocess.check_output([str(exe)], text=True).splitlines())
    assert int(out["attn_params"]) == ctypes.sizeof(_lib.AttnParams)
    size_t, stride_off = (int(x) for x in out["attn_tensor"].split())
    assert size_t == ctypes.sizeof(_lib.AttnTensor) and stride_off == _lib.AttnTensor.stride.offset
    for f in fields:
        assert int(out[f]) == getattr(_lib.AttnParams, f).offset, f


def test_noalloc_refuses_problems_larger_than_its_scratch(lib):
    """attn_bwd_noalloc refuses a problem whose workspace would not fit the
    library's fixed scratch before it touches any device state, so this runs
    without a GPU (the pointers are never dereferenced)."""
    p = _lib.AttnParams()
    p.dtype, p.layout = _lib.ATTN_BF16, _lib.ATTN_LAYOUT_DENSE4D
    # 64 x 65536 rows x 16 heads of fp32 row terms: 256 MiB of scratch
    p.B, p.Sq, p.Skv, p.Hq, p.Hkv, p.D = 64, 65536, 65536, 16, 16, 128
    p.scale, p.window_left, p.window_right = 0.125, -1, 0
    assert lib.attn_bwd_workspace_size(ctypes.byref(p)) > _lib.NOALLOC_SCRATCH_BYTES
    t = _t(strides=(65536 * 2048, 2048, 128, 1))
    st = lib.attn_bwd_noalloc(ctypes.byref(p), t, t, t, t, t, 4096, t, t, t, None)
    assert st == _lib.ATTN_ERR_UNSUPPORTED
    assert b"scratch" in lib.attn_last_error_string()


@pytest.mark.parametrize("which", [0, 1, 2])
def test_strides_beyond_tensor_map_reach_rejected(lib, which):
    """A stride of 2^40 bytes or more cannot be stepped by a tensor map: the
    call fails with UNSUPPORTED before anything is enqueued (forward and
    backward alike), while the same stride on a dim of extent 1 is never
    stepped and is accepted by the checks."""
    big = (1 << 40) // 2  # elements of 2 bytes
    strides = [32768, 256, 64, 1]
    strides[which] = big
    bad = _t(strides=tuple(strides))
    p = _params()
    st = lib.attn_fwd(ctypes.byref(p), bad, _t(), _t(), _t(), 4096, None)
    assert st == _lib.ATTN_ERR_UNSUPPORTED, lib.attn_last_error_string()
    assert b"2^40" in lib.attn_last_error_string()
    t = _t()
    st = lib.attn_bwd(ctypes.byref(p), t, t, t, t, t, 4096, t, t, bad, 4096, 1 << 30, None)
    assert st == _lib.ATTN_ERR_UNSUPPORTED, lib.attn_last_error_string()
    # extent-1 dims: B = 1 makes stride[0] irrelevant
    if which == 0:
        p1 = _params(B=1)
        st = lib.attn_fwd(ctypes.byref(p1), bad, bad, bad, bad, 0, None)
        assert st == _lib.ATTN_ERR_INVALID_ARG  # only the NULL lse is left to reject


def test_head_dim_256_is_a_16_bit_forward_only(lib):
    """Head dim 256 runs on the fp16 / bf16 tensor-core forward; the backward
    (whose 256-column dK and dV accumulators do not fit the tensor memory) and
    fp32 are refused before anything is enqueued."""
    p = _params(D=256)
    assert lib.attn_bwd_workspace_size(ctypes.byref(p)) == 0
    t = _t(strides=(32768 * 4, 1024, 256, 1))
    st = lib.attn_bwd(ctypes.byref(p), t, t, t, t, t, 4096, t, t, t, 4096, 1 << 20, None)
    assert st == _lib.ATTN_ERR_UNSUPPORTED and b"forward only" in lib.attn_last_error_string()
    p32 = _params(D=256, dtype=_lib.ATTN_F32)
    st = lib.attn_fwd(ctypes.byref(p32), t, t, t, t, 4096, None)
    assert st == _lib.ATTN_ERR_UNSUPPORTED
    assert lib.attn_fwd(ctypes.byref(_params(D=192)), t, t, t, t, 4096, None) == _lib.ATTN_ERR_UNSUPPORTED


def test_invariant_divisor_division_matches_integer_division(tmp_path):
    """FastDiv (division by a launch-invariant divisor as a multiply and
    shifts, used by the streaming kernels' index arithmetic) equals unsigned
    integer division for divisors 1..4096, large and power-of-two divisors,
    and numerators across the whole 32-bit range.  Host code of the same
    header the kernels include, compiled with nvcc (no GPU needed)."""
    import shutil
    import subprocess
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("no nvcc")
    src = tmp_path / "fastdiv.cu"
    src.write_text(
        '#include <cstdio>\n#include <cstdint>\n#include "common.cuh"\n'
        "int main() {\n"
        "    uint32_t ds[4200]; int nd = 0;\n"
        "    for (uint32_t d = 1; d <= 4096; ++d) ds[nd++] = d;\n"
        "    const uint32_t big[] = {65535u, 65536u, 65537u, 1000003u, 16777216u, 2147483647u, 2147483648u,\n"
        "                            3000000019u, 4294967295u};\n"
        "    for (uint32_t d : big) ds[nd++] = d;\n"
        "    uint64_t x = 88172645463325252ull; long bad = 0;\n"
        "    for (int i = 0; i < nd; ++i) {\n"
        "        const gbattn::FastDiv f(ds[i]);\n"
        "        const uint32_t edge[] = {0u, 1u, ds[i] - 1u, ds[i], ds[i] + 1u, 4294967295u, 2147483648u};\n"
        "        for (uint32_t n : edge) bad += f.div(n) != n / ds[i];\n"
        "        for (int k = 0; k < 2000; ++k) {\n"
        "            x ^= x << 13; x ^= x >> 7; x ^= x << 17;\n"
        "            const uint32_t n = (uint32_t)x;\n"
        "            bad += f.div(n) != n / ds[i];\n"
        "        }\n"
        "    }\n"
        '    printf("%ld\\n", bad);\n'
        "    return bad != 0;\n}\n")
    exe = tmp_path / "fastdiv"
    csrc = os.path.join(ROOT, "scaled_dot_product_03_gb300", "csrc")
    subprocess.check_call([nvcc, "-std=c++17", "-I", csrc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "0", out.stdout
