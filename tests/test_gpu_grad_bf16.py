"""bf16 gradient outputs (vsa_config_t.grad_dtype = VSA_GRAD_BF16).

The kernels compute every gradient in fp32 exactly as for fp32 outputs and
round once at the store, so the bf16 outputs must equal the fp32 outputs
rounded to nearest even, bit for bit.  The fp32 outputs themselves are held to
the oracle by the backward parity tests; together the two give the bf16 path
its parity.  Covered: the whole backward in raster and cube layout, an item
with no selected blocks (only the pooled gradient reaches its rows), both
head dims, a dynamic-selection layer, two heads of the 720p layer, and the
combine and fine backward entry points on their own."""
import pytest
import torch

from tests.helpers import cuda_inputs, enforce_gaps
from tests.test_gpu_forward import _custom, gapped
from trainable_block_sparse_gb300 import build, synth, vsa

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dgc", "dgf")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _backward(inp, layout, grad_dtype):
    cfg = vsa.config_for(inp.wl, layout, grad_dtype=grad_dtype)
    t = cuda_inputs(inp)
    if layout == "cube":
        for n in ("q", "k", "v", "gc", "gf", "do"):
            t[n] = vsa.permute(cfg, t[n])
    bufs = vsa.Buffers(cfg, "cuda", with_backward=True)
    vsa.forward(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs, with_backward=True)
    grads = vsa.backward(cfg, t["gc"], t["gf"], t["do"], bufs)
    torch.cuda.synchronize()
    assert bufs.device_status() == vsa.OK
    return grads


def check_rounding(inp, layout="raster"):
    g32 = _backward(inp, layout, "fp32")
    g16 = _backward(inp, layout, "bf16")
    for n, a, b in zip(NAMES, g32, g16):
        assert a.dtype == torch.float32 and b.dtype == torch.bfloat16
        rounded = a.to(torch.bfloat16)
        if not torch.equal(rounded, b):
            bad = (rounded != b).sum().item()
            diff = (rounded.float() - b.float()).abs().max().item()
            raise AssertionError(f"{n}: {bad} of {b.numel()} elements differ from the rounded "
                                 f"fp32 gradient (max diff {diff:.3e})")
        assert torch.count_nonzero(b) > 0, f"{n} is all zero"


@pytest.mark.parametrize("layout", ["raster", "cube"])
def test_tiny(layout):
    check_rounding(gapped("tiny"), layout)


@pytest.mark.parametrize("name", ["pretrain", "dynamic"])
def test_training_layers(name):
    check_rounding(gapped(name))


@pytest.mark.parametrize("thw,D,topk", [((4, 4, 12), 64, 2), ((8, 4, 12), 128, 5)])
def test_edge_shapes(thw, D, topk):
    check_rounding(_custom(*thw, D, topk, seed=21 + topk))


def test_unselected_key_cubes():
    """Key cubes no query selected take the pooled-only store path."""
    wl = synth.Workload("edge_unselected", 1, 1, 64, 8, 8, 8, "topk", topk=1, seed=31)
    inp = synth.Inputs(wl, with_grad=True)
    enforce_gaps(inp)
    check_rounding(inp)


def test_720p_two_heads():
    check_rounding(gapped("p720", heads=2))


def test_stage_entry_points():
    """vsa_combine_bwd and vsa_fine_bwd called on their own."""
    inp = gapped("tiny")
    wl = inp.wl
    t = cuda_inputs(inp)
    out = {}
    for gd in ("fp32", "bf16"):
        cfg = vsa.config_for(wl, grad_dtype=gd)
        bufs = vsa.Buffers(cfg, "cuda", with_backward=True)
        vsa.forward(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs, with_backward=True)
        B, H, N, D, nc, cap = wl.batch, wl.heads, wl.tokens, wl.head_dim, wl.cubes, \
            wl.list_capacity
        o_f = bufs.view("o_f", torch.float16, (B, H, N, D))
        oc = bufs.view("oc", torch.float32, (B, H, nc, D))
        dgc, dgf, dof, doc, delta, gscale = vsa.combine_bwd(cfg, t["do"], t["gc"], t["gf"], o_f,
                                                            oc, bufs.ws)
        v16 = [bufs.view(n, torch.float16, (B, H, N, D)) for n in ("q16", "k16", "v16")]
        dq, dk, dv = vsa.fine_bwd(cfg, *v16, bufs.view("idx", torch.int32, (B, H, nc, cap)),
                                  bufs.view("cnt", torch.int32, (B, H, nc)),
                                  bufs.view("lse_f", torch.float32, (B, H, N)), dof, delta,
                                  None, None, None, bufs.ws, gscale=gscale)
        torch.cuda.synchronize()
        assert bufs.device_status() == vsa.OK
        out[gd] = (dgc, dgf, dq, dk, dv)
    for n, a, b in zip(("dgc", "dgf", "dq", "dk", "dv"), out["fp32"], out["bf16"]):
        assert b.dtype == torch.bfloat16
        assert torch.equal(a.to(torch.bfloat16), b), n
