"""The FMA-pipe exponential of the softmax kernels (ex2_poly).

CPU: the coefficients compiled into csrc/sm103_ptx.cuh are the float32
roundings of the fit in exp2_fit.py, and a float32 emulation of the whole
function (range reduction, Horner steps, exponent add) stays within the fit's
bound over the input range.  GPU: the device function itself, run through
vsa_probe_exp2, against float64 exp2, and the ex2-unit path beside it."""
import os
import re

import numpy as np
import pytest
import torch

from trainable_block_sparse_gb300 import build, exp2_fit, vsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BOUND = 7.5e-5


def _header_coefficients():
    src = open(os.path.join(ROOT, "trainable_block_sparse_gb300", "csrc", "sm103_ptx.cuh")).read()
    body = src[src.index("float ex2_poly("):]
    body = body[: body.index("\n}\n")]
    lits = re.findall(r"(0x[0-9a-fA-F.]+p[-+]?\d+)f\)?;\s*//\s*c(\d)", body)
    return {int(k): float.fromhex(v) for v, k in lits}


def _emulate(x):
    f32 = np.float32
    c = [f32(v) for v in exp2_fit.float32_coefficients()]
    x = np.maximum(x.astype(np.float32), f32(-126.0))
    t = (x + f32(12582912.0)).astype(np.float32)
    f = (x - (t - f32(12582912.0))).astype(np.float32)
    p = c[3]
    for k in (2, 1, 0):  # fused multiply-add: one rounding per step
        p = (p.astype(np.float64) * f.astype(np.float64) + np.float64(c[k])).astype(np.float32)
    n = t.view(np.int32) - np.int32(0x4B400000)
    return (p.view(np.int32) + (n << 23)).view(np.float32)


def test_compiled_coefficients_are_the_fit():
    got = _header_coefficients()
    want = exp2_fit.float32_coefficients()
    assert sorted(got) == [0, 1, 2, 3]
    for k in range(4):
        assert got[k] == want[k], (k, got[k], want[k])


def test_fit_error_bound():
    _, err = exp2_fit.fit()
    assert err < BOUND


def test_emulated_function_within_bound():
    x = np.concatenate([np.linspace(-125.9, 127.9, 400001), np.arange(-125, 128) + 0.5,
                        np.arange(-125, 128).astype(np.float64)])
    y = _emulate(x).astype(np.float64)
    rel = np.abs(y / np.exp2(x.astype(np.float32).astype(np.float64)) - 1)
    assert rel.max() < BOUND + 1e-6, rel.max()
    # below the clamp the result is negligible, never garbage
    lo = _emulate(np.array([-126.0, -200.0, -np.inf], dtype=np.float32))
    assert np.all(np.abs(lo) <= 2.0 ** -125)


@pytest.mark.gpu
def test_device_exponentials_against_float64():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    L = vsa.lib()
    x = torch.cat([torch.linspace(-125.9, 127.9, 1 << 20, dtype=torch.float64),
                   torch.tensor([-126.0, -300.0, float("-inf"), 0.0, 8.0])]).float().cuda()
    ref = torch.exp2(x.double())
    for which, bound in ((0, 2e-6), (1, BOUND + 1e-6)):
        y = torch.empty_like(x)
        assert L.vsa_probe_exp2(vsa._ptr(x), vsa._ptr(y), x.numel(), which, vsa._stream()) == vsa.OK
        torch.cuda.synchronize()
        body = x >= -125.0
        rel = (y[body].double() / ref[body] - 1).abs().max().item()
        assert rel < bound, (which, rel)
        assert torch.all(y[~body].abs() <= 2.0 ** -125), which
