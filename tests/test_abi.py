"""The C ABI library: it loads, exports what include/vsa.h declares, and its
host-side argument checks answer correctly.  No GPU is needed: none of these
calls launches a kernel."""
import ctypes
import os
import re

import pytest

from trainable_block_sparse_gb300 import build, vsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return vsa.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "vsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(vsa_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/vsa.h but not exported"


def _cfg(**kw):
    base = dict(batch=1, heads=2, T=8, H=8, W=8, head_dim=64, topk=2)
    base.update(kw)
    return vsa.make_config(base.pop("batch"), base.pop("heads"), base.pop("T"), base.pop("H"),
                           base.pop("W"), base.pop("head_dim"), **base)


@pytest.mark.parametrize("kw,status", [
    ({}, vsa.OK),
    ({"T": 6}, vsa.ERR_SHAPE),
    ({"W": 0}, vsa.ERR_SHAPE),
    ({"head_dim": 96}, vsa.ERR_UNSUPPORTED),
    ({"topk": 0}, vsa.ERR_INVALID_ARG),
    ({"topk": 9}, vsa.ERR_INVALID_ARG),          # more than the 8 cubes
    ({"batch": 0}, vsa.ERR_INVALID_ARG),
    ({"select": "mass", "kmin": 9, "kmax": 8}, vsa.ERR_INVALID_ARG),
    ({"select": "mass", "mass": 0.0}, vsa.ERR_INVALID_ARG),
    ({"select": "mass", "kmax": 300}, vsa.ERR_INVALID_ARG),
    ({"select": "mass"}, vsa.OK),
    ({"T": 4096, "H": 64, "W": 64}, vsa.ERR_SHAPE),  # too many cubes
    ({"grad_dtype": "bf16"}, vsa.OK),
])
def test_validate(lib, kw, status):
    cfg = _cfg(**kw)
    assert lib.vsa_validate(ctypes.byref(cfg)) == status


def test_unknown_gradient_dtype_is_rejected(lib):
    cfg = _cfg()
    cfg.grad_dtype = 2
    assert lib.vsa_validate(ctypes.byref(cfg)) == vsa.ERR_INVALID_ARG
    with pytest.raises(ValueError, match="grad_dtype"):
        _cfg(grad_dtype="fp16")


def test_null_config_and_pointers(lib):
    assert lib.vsa_validate(None) == vsa.ERR_INVALID_ARG
    cfg = _cfg()
    # null tensors are rejected on the host, before any launch
    assert lib.vsa_permute(ctypes.byref(cfg), None, None, 0, None) == vsa.ERR_INVALID_ARG
    assert lib.vsa_forward(ctypes.byref(cfg), *([None] * 7), 1, None, None) == vsa.ERR_INVALID_ARG


def test_coarse_select_inputs_are_all_or_none(lib):
    """q, k, v: all given (pooled here) or all NULL (qc, kc, vc are the means)."""
    cfg = _cfg()
    p = ctypes.c_void_p(0x1000)
    outs = [p] * 8  # qc, kc, vc, oc, lse_c, idx, cnt, ws
    for qkv in ([p, p, None], [None, p, None], [p, None, p]):
        assert lib.vsa_coarse_select(ctypes.byref(cfg), *qkv, *outs, None) == vsa.ERR_INVALID_ARG
    # the pooled form still needs every output
    assert lib.vsa_coarse_select(ctypes.byref(cfg), None, None, None, *([p] * 7), None,
                                 None) == vsa.ERR_INVALID_ARG
    # and checks alignment on the host
    odd = ctypes.c_void_p(0x2008)
    assert lib.vsa_coarse_select(ctypes.byref(cfg), None, None, None, odd, *([p] * 7),
                                 None) == vsa.ERR_ALIGNMENT


def test_misaligned_pointer_is_rejected(lib):
    cfg = _cfg()
    a = ctypes.c_void_p(0x1000)
    b = ctypes.c_void_p(0x2008)  # not 16-byte aligned
    assert lib.vsa_permute(ctypes.byref(cfg), a, b, 0, None) == vsa.ERR_ALIGNMENT
    assert lib.vsa_permute(ctypes.byref(cfg), a, a, 0, None) == vsa.ERR_INVALID_ARG


def test_buffer_sizes(lib):
    cfg = _cfg()
    L = vsa.saved_layout(cfg)
    # pieces are 256-byte aligned, in order, and fit the total
    offs = [L.qc, L.kc, L.vc, L.oc, L.lse_c, L.idx, L.cnt, L.lse_f, L.q16, L.k16, L.v16,
            L.o_f]
    assert all(o % 256 == 0 for o in offs)
    assert offs == sorted(offs) and L.total > offs[-1]
    assert L.list_cap == 2
    n_tok = 2 * 512
    assert L.lse_f - L.cnt >= 2 * 8 * 4 and L.q16 - L.lse_f >= n_tok * 4
    assert L.total - L.o_f >= n_tok * 64 * 2
    fwd = vsa.workspace_bytes(cfg, False)
    bwd = vsa.workspace_bytes(cfg, True)
    assert 0 < fwd < bwd
    bad = _cfg(T=5)
    assert lib.vsa_saved_bytes(ctypes.byref(bad), None) == 0
    assert lib.vsa_workspace_bytes(ctypes.byref(bad), 1) == 0
    # staged fp16 copies of Q, K, V, one [B, heads, N, D] each
    assert L.k16 - L.q16 >= n_tok * 64 * 2 and L.o_f - L.v16 >= n_tok * 64 * 2


def test_inference_saved_buffer_drops_what_only_training_needs(lib):
    # head_dim 64 (raster): the inference forward reads q, k, v in place and
    # writes no O_f: the buffer ends where the staged copies begin; the offsets
    # are the training layout's
    cfg = _cfg()
    full = vsa.saved_layout(cfg)
    inf = vsa.saved_layout(cfg, with_backward=False)
    assert lib.vsa_saved_bytes_for(ctypes.byref(cfg), 1, None) == full.total
    assert lib.vsa_saved_bytes(ctypes.byref(cfg), None) == full.total
    for name in ("q16", "k16", "v16", "qc", "kc", "vc", "oc", "lse_c", "idx", "cnt", "o_f",
                 "lse_f"):
        assert getattr(inf, name) == getattr(full, name)
    assert inf.total == full.q16
    n_tok = 2 * 512
    assert full.total - inf.total >= 4 * n_tok * 64 * 2
    # raster head_dim 128: the inference forward stages, so only O_f goes
    cfg128 = _cfg(head_dim=128)
    full128 = vsa.saved_layout(cfg128)
    assert vsa.saved_layout(cfg128, with_backward=False).total == full128.o_f
    # cube layout head_dim 128 reads in place again
    cube128 = _cfg(head_dim=128, layout="cube")
    assert vsa.saved_layout(cube128, with_backward=False).total == \
        vsa.saved_layout(cube128).q16
    bad = _cfg(T=5)
    assert lib.vsa_saved_bytes_for(ctypes.byref(bad), 0, None) == 0


def test_status_strings(lib):
    for s in range(8):
        assert len(lib.vsa_status_string(s)) > 0
    assert lib.vsa_status_string(99) == b"unknown status"


def test_wait_probe_arguments_are_checked_on_the_host(lib):
    ws = ctypes.c_void_p(0x1000)
    assert lib.vsa_probe_wait_timeout(None, 1000, None) == vsa.ERR_INVALID_ARG
    assert lib.vsa_probe_wait_timeout(ws, 0, None) == vsa.ERR_INVALID_ARG
    assert lib.vsa_probe_wait_timeout(ws, 20_000_000, None) == vsa.ERR_INVALID_ARG
    assert lib.vsa_probe_wait_timeout(ctypes.c_void_p(0x1008), 1000, None) == vsa.ERR_ALIGNMENT


# ------------------------------------------- the autograd entry point's checks

def _bf(*shape, dtype=None):
    import torch
    return torch.zeros(*shape, dtype=dtype or torch.bfloat16)


def _five(shape=(1, 2, 512, 64), **over):
    t = {n: _bf(*shape) for n in ("q", "k", "v", "gc", "gf")}
    t.update(over)
    return t


@pytest.mark.parametrize("case,exc,match", [
    ("fp16_q", TypeError, "q must be bfloat16"),
    ("fp32_gf", TypeError, "gf must be bfloat16"),
    ("not_tensor", TypeError, "k must be a torch.Tensor"),
    ("three_d", ValueError, "must be 4-D"),
    ("shape_k", ValueError, "k has shape"),
    ("shape_gc", ValueError, "gc has shape"),
    ("tokens", ValueError, "T\\*H\\*W"),
    ("video_shape", ValueError, "video_shape"),
    ("layout", ValueError, "layout"),
    ("cpu", ValueError, "CUDA tensor"),
])
def test_video_sparse_attention_refuses_before_any_launch(case, exc, match):
    """Inputs the kernels would misread raise on the host; no kernel runs
    (these tensors are on the CPU, and the refusals come first)."""
    import torch
    vs = (8, 8, 8)
    kw = {}
    if case == "fp16_q":
        t = _five(q=_bf(1, 2, 512, 64, dtype=torch.float16))
    elif case == "fp32_gf":
        t = _five(gf=_bf(1, 2, 512, 64, dtype=torch.float32))
    elif case == "not_tensor":
        t = _five(k=[[0.0]])
    elif case == "three_d":
        t = _five(shape=(2, 512, 64))
    elif case == "shape_k":
        t = _five(k=_bf(1, 2, 512, 128))
    elif case == "shape_gc":
        t = _five(gc=_bf(1, 1, 512, 64))
    elif case == "tokens":
        t = _five()
        vs = (8, 8, 4)
    elif case == "video_shape":
        t = _five()
        vs = (8, 64)
    elif case == "layout":
        t = _five()
        kw = {"layout": "zigzag"}
    else:
        t = _five()
    with pytest.raises(exc, match=match):
        vsa.video_sparse_attention(t["q"], t["k"], t["v"], t["gc"], t["gf"], vs, topk=2, **kw)


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c++", "c++17")])
def test_header_is_plain_c_and_cpp(lang, std):
    """include/vsa.h compiles on its own as C99 and as C++17 (no CUDA or torch
    types in the boundary)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                       "vsa.h")
    r = subprocess.run([cc, "-fsyntax-only", "-Wall", "-Werror", "-x", lang, f"-std={std}", hdr],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
