"""Backward parity of the CUDA path against the fp64 oracle's analytic
gradients (selection held fixed): dQ, dK, dV, dG_c, dG_f within max-abs 2e-2
and relative-L2 1e-2; also the component entry points (combine backward,
coarse backward) on their own."""
import numpy as np
import pytest
import torch

from oracle import vsa_oracle as O
from tests.helpers import assert_close, cuda_inputs, enforce_gaps, to_np
from tests.test_gpu_forward import cubes_of, gapped, slices_of
from trainable_block_sparse_gb300 import build, synth, vsa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_fwd_bwd(inp, layout="raster"):
    wl = inp.wl
    cfg = vsa.config_for(wl, layout)
    t = cuda_inputs(inp)
    if layout == "cube":
        for n in ("q", "k", "v", "gc", "gf", "do"):
            t[n] = vsa.permute(cfg, t[n])
    bufs = vsa.Buffers(cfg, "cuda", with_backward=True)
    vsa.forward(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs, with_backward=True)
    grads = vsa.backward(cfg, t["gc"], t["gf"], t["do"], bufs)
    torch.cuda.synchronize()
    assert bufs.device_status() == vsa.OK
    if layout == "cube":
        grads = tuple(_untile_f32(cfg, g) for g in grads)
    return [to_np(g) for g in grads]


def _untile_f32(cfg, g):
    # fp32 gradients in cube order -> raster, on the host (test plumbing only)
    wl_T, wl_H, wl_W = cfg.T, cfg.H, cfg.W
    return torch.from_numpy(O.untile(g.cpu().double().numpy(), wl_T, wl_H, wl_W))


def check_backward(inp, layout="raster", full=False):
    wl = inp.wl
    dq, dk, dv, dgc, dgf = run_fwd_bwd(inp, layout)
    for b, h in slices_of(wl, full):
        hd = O.head_of(inp, b, h)
        cubes = cubes_of(wl, full, seed=7 * b + h)
        got = {n: [] for n in ("dq", "dgc", "dgf", "dk", "dv")}
        ref = {n: [] for n in got}
        for c in cubes:
            rows = synth.raster_rows_of_cube(wl, c)
            rq, rgc, rgf = hd.grad_query_cube(c)
            rk, rv = hd.grad_key_cube(c)
            for n, r, g in (("dq", rq, dq), ("dgc", rgc, dgc), ("dgf", rgf, dgf),
                            ("dk", rk, dk), ("dv", rv, dv)):
                ref[n].append(r)
                got[n].append(g[b, h, rows])
        for n in got:
            assert_close(f"{n} slice {(b, h)}", np.stack(got[n]), np.stack(ref[n]))


def test_backward_tiny_full():
    check_backward(gapped("tiny"), full=True)


def test_backward_tiny_cube_layout():
    check_backward(gapped("tiny"), layout="cube", full=True)


@pytest.mark.parametrize("name", ["pretrain", "dynamic"])
def test_backward_sampled(name):
    check_backward(gapped(name))


@pytest.mark.slow
def test_backward_sampled_720p():
    check_backward(gapped("p720"))


@pytest.mark.parametrize("thw,D,topk", [((4, 4, 12), 64, 2), ((8, 4, 12), 128, 5),
                                        ((4, 8, 8), 64, 4)])
def test_backward_edge_shapes(thw, D, topk):
    from tests.test_gpu_forward import _custom
    check_backward(_custom(*thw, D, topk, seed=21 + topk), full=True)


def test_autograd_function_matches_entry_points():
    inp = gapped("tiny")
    wl = inp.wl
    t = cuda_inputs(inp)
    leaves = {n: t[n].clone().requires_grad_(True) for n in ("q", "k", "v", "gc", "gf")}
    o = vsa.video_sparse_attention(leaves["q"], leaves["k"], leaves["v"], leaves["gc"],
                                   leaves["gf"], (wl.T, wl.H, wl.W), topk=wl.topk)
    o.backward(t["do"])
    dq, dk, dv, dgc, dgf = run_fwd_bwd(inp)
    for n, ref in (("q", dq), ("k", dk), ("v", dv), ("gc", dgc), ("gf", dgf)):
        got = to_np(leaves[n].grad)
        # the autograd path rounds gradients to the inputs' dtype (bf16)
        assert np.max(np.abs(got - ref)) <= 2.0 ** -8 * np.max(np.abs(ref)) + 1e-6


def test_empty_key_cubes_get_only_the_pooled_gradient():
    """A key cube no query selected: dK, dV come from the coarse stage alone."""
    wl = synth.Workload("edge_unselected", 1, 1, 64, 8, 8, 8, "topk", topk=1, seed=31)
    inp = synth.Inputs(wl, with_grad=True)
    enforce_gaps(inp)
    hd = O.head_of(inp, 0, 0)
    unselected = sorted(set(range(wl.cubes)) - set(hd.idx[:, 0].tolist()))
    assert unselected, "this seed should leave some key cube unselected"
    dq, dk, dv, dgc, dgf = run_fwd_bwd(inp)
    for j in unselected:
        rows = synth.raster_rows_of_cube(wl, j)
        rk, rv = hd.grad_key_cube(j)
        assert_close("dk", dk[0, 0, rows], rk)
        assert_close("dv", dv[0, 0, rows], rv)
        np.testing.assert_allclose(rk, np.repeat(hd.dkc[j][None] / 64, 64, 0), atol=1e-12)


@pytest.mark.parametrize("name,heads", [("p720", 4), ("dynamic", None)])
def test_repeated_layers_are_bitwise_identical(name, heads):
    """The fine kernels' CTAs take items from a shared counter as they free up,
    so which CTA runs an item changes from run to run; every item is computed
    by one CTA alone, so the forward and backward outputs must not change."""
    inp = gapped(name, heads=heads) if heads else gapped(name)
    cfg = vsa.config_for(inp.wl)
    t = cuda_inputs(inp)
    runs = []
    for _ in range(3):
        bufs = vsa.Buffers(cfg, "cuda", with_backward=True)
        o = vsa.forward(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs, with_backward=True)
        grads = vsa.backward(cfg, t["gc"], t["gf"], t["do"], bufs)
        torch.cuda.synchronize()
        assert bufs.device_status() == vsa.OK
        runs.append([o.clone()] + [g.clone() for g in grads])
    for later in runs[1:]:
        for a, b in zip(runs[0], later):
            assert torch.equal(a, b)


def test_layer_replays_from_a_cuda_graph():
    """vsa_forward and vsa_backward captured into a CUDA graph (the backward's
    list building forks to a second stream and joins back inside the capture)
    replay to the eager results, bit for bit."""
    inp = gapped("pretrain")
    cfg = vsa.config_for(inp.wl)
    t = cuda_inputs(inp)
    bufs = vsa.Buffers(cfg, "cuda", with_backward=True)

    def layer():
        o = vsa.forward(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs, with_backward=True)
        return [o] + list(vsa.backward(cfg, t["gc"], t["gf"], t["do"], bufs))

    eager = [x.clone() for x in layer()]
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer()  # warm-up on the capture's stream
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(graph):
        outs = layer()
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        assert bufs.device_status() == vsa.OK
        for a, b in zip(eager, outs):
            assert torch.equal(a, b)
