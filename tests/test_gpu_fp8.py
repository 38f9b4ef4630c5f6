"""The e4m3 (fp8) variant of the fine forward, head_dim 128, inference.

Its accuracy is e4m3's (3 significand bits for Q, K, V and P), so it is
compared with the fp64 oracle and its errors are reported (printed), not
held to the fp16 path's bounds: e4m3 rounding of Q and K moves each logit by
~0.07, which slices with very peaked attention do not average out (measured:
O rel-L2 1.4e-2 on the 720p slice, up to 5.4e-2 on one Wan-1.3B slice).  The
asserted bounds only catch gross failures: a misplaced tile, a wrong layout
or a lost scale factor makes the error O(1).  The index lists come from the fp32 coarse stage and must match the
oracle bit for bit, as in the fp16 path.  Layers: the Wan-1.3B layer (every
slice, every cube) and one whole slice of the 720p layer.
"""
import numpy as np
import pytest
import torch

from oracle import vsa_oracle as O
from tests.helpers import cuda_inputs, errors
from tests.test_gpu_forward import gapped
from tests.test_gpu_full_parity import P720_SLICE, all_slices
from trainable_block_sparse_gb300 import build, vsa

pytestmark = pytest.mark.gpu

REL_L2_O = 1e-1    # O (gated combine) against the fp64 oracle: gross failures only
REL_L2_LSE = 2e-2  # lse_f


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def fp8_layer(inp, slices):
    wl = inp.wl
    cfg = vsa.config_for(wl)
    t = cuda_inputs(inp)
    bufs = vsa.Buffers(cfg, "cuda", with_backward=False)
    o = vsa.forward_fp8(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs)
    torch.cuda.synchronize()
    assert bufs.device_status() == vsa.OK
    B, H, N, D, nc, cap = wl.batch, wl.heads, wl.tokens, wl.head_dim, wl.cubes, wl.list_capacity
    idx = bufs.view("idx", torch.int32, (B, H, nc, cap))
    cnt = bufs.view("cnt", torch.int32, (B, H, nc))
    lse = bufs.view("lse_f", torch.float32, (B, H, N))
    out = {}
    for b, h in slices:
        out[(b, h)] = {"o": O.tile(o[b, h].to("cpu", torch.float64).numpy(), wl.T, wl.H, wl.W),
                       "idx": idx[b, h].cpu().numpy(), "cnt": cnt[b, h].cpu().numpy(),
                       "lse_f": lse[b, h].cpu().double().numpy()}
    return out


def check(inp, slices, pool, tag):
    wl = inp.wl
    got = fp8_layer(inp, slices)
    ref = pool.layer(inp, slices, tag, backward=False)
    worst = {"o": (0.0, 0.0), "lse_f": (0.0, 0.0)}
    for key in slices:
        g, r = got[key], ref[key]
        assert np.array_equal(g["cnt"], r["cnt"]), f"counts differ in slice {key}"
        assert np.array_equal(g["idx"], r["idx"]), f"index lists differ in slice {key}"
        for n, bound in (("o", REL_L2_O), ("lse_f", REL_L2_LSE)):
            ma, rel = errors(g[n], r[n].reshape(g[n].shape))
            assert np.isfinite(g[n]).all(), f"{n} {key}: non-finite values"
            assert rel <= bound, f"{n} {key}: rel-L2 {rel:.3e} (bound {bound}), max-abs {ma:.3e}"
            worst[n] = max(worst[n], (rel, ma))
    print(f"\n{wl.name} e4m3 fine stage against the fp64 oracle: "
          f"O rel-L2 {worst['o'][0]:.3e} max-abs {worst['o'][1]:.3e}; "
          f"lse_f rel-L2 {worst['lse_f'][0]:.3e} max-abs {worst['lse_f'][1]:.3e}")


def test_fp8_wan13b_every_slice(oracle_pool):
    inp = gapped("wan13b")
    check(inp, all_slices(inp.wl), oracle_pool, "wan13b_fp8")


def test_fp8_p720_one_slice(oracle_pool):
    check(gapped("p720"), [P720_SLICE], oracle_pool, "p720_fp8")


def test_fp8_refuses_head_dim_64():
    inp = gapped("tiny")
    cfg = vsa.config_for(inp.wl)
    t = cuda_inputs(inp)
    bufs = vsa.Buffers(cfg, "cuda", with_backward=False)
    with pytest.raises(vsa.VSAError) as e:
        vsa.forward_fp8(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs)
    assert e.value.status == vsa.ERR_UNSUPPORTED
