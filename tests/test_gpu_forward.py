"""Forward parity of the CUDA path against the fp64 oracle.

Index lists must match bit for bit (inputs are drawn so that no selection
boundary is closer than 1e-3 in logit); floating-point outputs must be within
max-abs 2e-2 and relative-L2 1e-2 of the oracle.  Small layers are compared
element by element; full-size layers on sampled (batch, head) slices and
cubes, in the same launch configuration the benchmark times.
"""
import functools

import numpy as np
import pytest
import torch

from oracle import vsa_oracle as O
from tests.helpers import assert_close, cuda_inputs, enforce_gaps, to_np
from trainable_block_sparse_gb300 import build, synth, vsa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@functools.lru_cache(maxsize=6)
def gapped(name, **over):
    wl = synth.WORKLOADS[name].replace(**over) if over else synth.WORKLOADS[name]
    inp = synth.Inputs(wl, with_grad=True)
    enforce_gaps(inp)
    return inp


def run_forward(inp, layout="raster", with_backward=True):
    wl = inp.wl
    cfg = vsa.config_for(wl, layout)
    t = cuda_inputs(inp)
    if layout == "cube":
        for n in ("q", "k", "v", "gc", "gf"):
            t[n] = vsa.permute(cfg, t[n])
    bufs = vsa.Buffers(cfg, "cuda", with_backward=with_backward)
    o = vsa.forward(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs,
                    with_backward=with_backward)
    torch.cuda.synchronize()
    assert bufs.device_status() == vsa.OK
    B, H, N, D, nc, cap = wl.batch, wl.heads, wl.tokens, wl.head_dim, wl.cubes, wl.list_capacity
    views = {
        "idx": bufs.view("idx", torch.int32, (B, H, nc, cap)),
        "cnt": bufs.view("cnt", torch.int32, (B, H, nc)),
        "qc": bufs.view("qc", torch.float32, (B, H, nc, D)),
        "oc": bufs.view("oc", torch.float32, (B, H, nc, D)),
        "lse_c": bufs.view("lse_c", torch.float32, (B, H, nc)),
        "lse_f": bufs.view("lse_f", torch.float32, (B, H, N)),
    }
    if with_backward:
        views["o_f"] = bufs.view("o_f", torch.float16, (B, H, N, D))
    if layout == "cube":
        o = vsa.permute(cfg, o, inverse=True)
    return cfg, t, bufs, o, views


def slices_of(wl, full):
    if full:
        return [(b, h) for b in range(wl.batch) for h in range(wl.heads)]
    return sorted({(0, 0), (wl.batch - 1, wl.heads - 1), (0, wl.heads // 2)})


def cubes_of(wl, full, seed=0):
    if full:
        return list(range(wl.cubes))
    r = np.random.default_rng(seed)
    extra = r.choice(wl.cubes, size=3, replace=False).tolist()
    return sorted({0, 1, wl.cubes - 1, wl.cubes // 2, *extra})


def check_forward(inp, layout="raster", full=False, with_backward=True):
    """with_backward=False checks the inference path (bf16 inputs read in place,
    no O_f)."""
    wl = inp.wl
    cfg, t, bufs, o, v = run_forward(inp, layout, with_backward)
    o_np = to_np(o)
    for b, h in slices_of(wl, full):
        hd = O.head_of(inp, b, h)
        # selection: bit-exact lists and counts for every query cube of the slice
        cnt = v["cnt"][b, h].cpu().numpy()
        idx = v["idx"][b, h].cpu().numpy()
        assert np.array_equal(cnt, hd.cnt), f"counts differ in slice {(b, h)}"
        assert np.array_equal(idx, hd.idx), f"index lists differ in slice {(b, h)}"
        assert_close("O_c", to_np(v["oc"][b, h]), hd.coarse["out"])
        assert_close("lse_c", to_np(v["lse_c"][b, h]), hd.coarse["lse"])
        # fp32 sum of 64 terms: error <= 63 * 2^-24 * mean |x| of the cube
        qc_bound = 63 * 2.0 ** -24 * float(np.abs(hd.qt).reshape(wl.cubes, 64, -1)
                                           .mean(axis=1).max())
        assert_close("Q_c", to_np(v["qc"][b, h]), hd.qc, atol=max(1e-5, qc_bound), rtol_l2=1e-6)
        cubes = cubes_of(wl, full, seed=b * 1000 + h)
        of_g = (to_np(v["o_f"][b, h]).reshape(wl.cubes, 64, wl.head_dim) if with_backward
                else None)
        lse_g = to_np(v["lse_f"][b, h]).reshape(wl.cubes, 64)
        ref_o, got_o, ref_of, got_of, ref_l, got_l = [], [], [], [], [], []
        for c in cubes:
            _, of, lse = hd.rows(c)
            if with_backward:
                ref_of.append(of)
                got_of.append(of_g[c])
            ref_l.append(lse)
            got_l.append(lse_g[c])
            ref_o.append(hd.output_tiled(c))
            got_o.append(o_np[b, h, synth.raster_rows_of_cube(wl, c)])
        if with_backward:
            assert_close("O_f", np.stack(got_of), np.stack(ref_of))
        assert_close("lse_f", np.stack(got_l), np.stack(ref_l))
        assert_close("O", np.stack(got_o), np.stack(ref_o))


def test_forward_tiny_full():
    check_forward(gapped("tiny"), full=True)


def test_forward_tiny_cube_layout():
    check_forward(gapped("tiny"), layout="cube", full=True)


@pytest.mark.parametrize("layout", ["raster", "cube"])
def test_inference_forward_tiny(layout):
    """The inference path (bf16 inputs read in place): 5-D cube copies in raster
    layout, 2-D copies in cube layout."""
    check_forward(gapped("tiny"), layout=layout, full=True, with_backward=False)


@pytest.mark.parametrize("thw,D,topk", [((4, 4, 12), 64, 2), ((8, 4, 12), 128, 5),
                                        ((4, 4, 4), 128, 1)])
def test_inference_forward_edge_shapes(thw, D, topk):
    check_forward(_custom(*thw, D, topk, seed=7 + topk), full=True, with_backward=False)


@pytest.mark.parametrize("thw,topk", [((8, 4, 12), 5), ((4, 4, 4), 1)])
def test_inference_forward_cube_layout_head_dim_128(thw, topk):
    check_forward(_custom(*thw, 128, topk, seed=9 + topk), layout="cube", full=True,
                  with_backward=False)


@pytest.mark.parametrize("layout", ["raster", "cube"])
def test_fine_stage_in_place_head_dim_128(layout):
    """vsa_fine_fwd_bf16 itself at head_dim 128 (5-D cube copies in raster
    layout), fed the oracle's lists and O_c, on every cube of the tiny-shaped
    layer at D = 128."""
    inp = _custom(8, 8, 8, 128, 3, seed=17)
    wl = inp.wl
    cfg = vsa.config_for(wl, layout)
    heads = {(0, h): O.head_of(inp, 0, h) for h in range(wl.heads)}
    idx = np.stack([[heads[(0, h)].idx for h in range(wl.heads)]])
    cnt = np.stack([[heads[(0, h)].cnt for h in range(wl.heads)]])
    oc = np.stack([[heads[(0, h)].coarse["out"] for h in range(wl.heads)]])
    t = cuda_inputs(inp)
    if layout == "cube":
        for n in ("q", "k", "v", "gc", "gf"):
            t[n] = vsa.permute(cfg, t[n])
    ws = torch.empty(vsa.workspace_bytes(cfg, False), dtype=torch.uint8, device="cuda")
    vsa.lib().vsa_reset_device_status(vsa._ptr(ws), vsa._stream())
    o, lse = vsa.fine_fwd_bf16(cfg, t["q"], t["k"], t["v"], torch.from_numpy(idx).int().cuda(),
                               torch.from_numpy(cnt).int().cuda(), t["gc"], t["gf"],
                               torch.from_numpy(oc).float().cuda(), ws)
    torch.cuda.synchronize()
    assert vsa.lib().vsa_check_device_status(vsa._ptr(ws), vsa._stream()) == vsa.OK
    if layout == "cube":
        o = vsa.permute(cfg, o, inverse=True)
    o_np, lse_np = to_np(o), to_np(lse)
    for h, hd in ((h, heads[(0, h)]) for h in range(wl.heads)):
        for c in range(wl.cubes):
            _, _, lse_r = hd.rows(c)
            assert_close("O", o_np[0, h, synth.raster_rows_of_cube(wl, c)], hd.output_tiled(c))
            assert_close("lse_f", lse_np[0, h, c * 64:(c + 1) * 64], lse_r)


def test_inference_forward_accepts_values_beyond_fp16():
    """No staged fp16 copy on the inference path: a Q value above 65504 is
    computed, not refused (the oracle agrees)."""
    inp = _custom(4, 4, 8, 64, 1, seed=15)
    inp.q = inp.q.clone()
    inp.q[0, 1, 77, 5] = 1.0e5
    big = inp.q[0, 1, 77, 5].item()
    enforce_gaps(inp)
    assert inp.q[0, 1, 77, 5].item() == big > 65504.0
    check_forward(inp, full=True, with_backward=False)


@pytest.mark.parametrize("name", ["pretrain", "wan13b", "dynamic"])
def test_forward_sampled(name):
    check_forward(gapped(name))


@pytest.mark.slow
def test_forward_sampled_720p():
    check_forward(gapped("p720"))


def test_permute_is_oracle_tiling():
    inp = gapped("tiny")
    wl = inp.wl
    cfg = vsa.config_for(wl)
    q = inp.q.cuda()
    qt = vsa.permute(cfg, q)
    ref = np.stack([O.tile(O.f64(inp.q[0, h]), wl.T, wl.H, wl.W) for h in range(wl.heads)])
    assert np.array_equal(to_np(qt)[0], ref)  # bit-exact: a pure rearrangement
    assert torch.equal(vsa.permute(cfg, qt, inverse=True), q)


@pytest.mark.parametrize("name", ["tiny", "dynamic"])
def test_coarse_select_from_staged_means(name):
    """vsa_coarse_select with q, k, v NULL reads the means vsa_stage wrote and
    gives what the pooling call gives, bit for bit."""
    inp = gapped(name)
    cfg = vsa.config_for(inp.wl)
    t = cuda_inputs(inp)
    ws = torch.empty(vsa.workspace_bytes(cfg, False), dtype=torch.uint8, device="cuda")
    qc, kc, vc, oc, lse, idx, cnt = vsa.coarse_select(cfg, t["q"], t["k"], t["v"], ws)
    means = [vsa.stage(cfg, t[n], ws, want_pooled=True)[1] for n in ("q", "k", "v")]
    for a, b in zip((qc, kc, vc), means):
        assert torch.equal(a, b)
    oc2, lse2, idx2, cnt2 = vsa.coarse_select_pooled(cfg, *means, ws)
    torch.cuda.synchronize()
    for a, b in ((oc, oc2), (lse, lse2), (idx, idx2), (cnt, cnt2)):
        assert torch.equal(a, b)


def test_pooled_means_within_fp32_summation_bound():
    inp = gapped("pretrain")
    wl = inp.wl
    cfg = vsa.config_for(wl)
    q = inp.q.cuda()
    ws = torch.empty(vsa.workspace_bytes(cfg, False), dtype=torch.uint8, device="cuda")
    qc = vsa.coarse_select(cfg, q, q, q, ws)[0]
    q16, qc2 = vsa.stage(cfg, q, ws, want_pooled=True)
    assert torch.equal(qc, qc2)
    # the staged copy is the fp16 value of every bf16 input, in cube order: exact
    # in the normal fp16 range, within half a subnormal step (2^-25) below it
    ref = vsa.permute(cfg, q).float()
    normal = ref.abs() >= 2.0 ** -14
    assert torch.equal(q16.float()[normal], ref[normal])
    assert (q16.float() - ref).abs().max().item() <= 2.0 ** -25
    for b, h in slices_of(wl, False):
        x = O.tile(O.f64(inp.q[b, h]), wl.T, wl.H, wl.W).reshape(wl.cubes, 64, wl.head_dim)
        exact = x.mean(axis=1)
        bound = 63 * 2.0 ** -24 * np.abs(x).mean(axis=1) + 1e-30
        assert np.all(np.abs(to_np(qc[b, h]) - exact) <= bound)


@pytest.mark.parametrize("name", ["tiny", "pretrain"])
def test_fine_stage_with_injected_oracle_lists(name):
    """The fine stage alone, fed the oracle's lists, pooled O_c and tiled inputs."""
    inp = gapped(name)
    wl = inp.wl
    cfg = vsa.config_for(wl, layout="cube")
    heads = {(b, h): O.head_of(inp, b, h) for b, h in slices_of(wl, True)}
    idx = np.stack([[heads[(b, h)].idx for h in range(wl.heads)] for b in range(wl.batch)])
    cnt = np.stack([[heads[(b, h)].cnt for h in range(wl.heads)] for b in range(wl.batch)])
    oc = np.stack([[heads[(b, h)].coarse["out"] for h in range(wl.heads)] for b in range(wl.batch)])

    def tiled(x):
        return torch.from_numpy(O.tile(O.f64(x), wl.T, wl.H, wl.W)).to(torch.bfloat16).cuda()

    q, k, v, gc, gf = (tiled(getattr(inp, n)) for n in ("q", "k", "v", "gc", "gf"))
    ws = torch.empty(vsa.workspace_bytes(cfg, False), dtype=torch.uint8, device="cuda")
    vsa.lib().vsa_reset_device_status(vsa._ptr(ws), vsa._stream())
    q, k, v = (vsa.stage(cfg, x, ws) for x in (q, k, v))
    o, of, lse = vsa.fine_fwd(cfg, q, k, v, torch.from_numpy(idx).int().cuda(),
                              torch.from_numpy(cnt).int().cuda(), gc, gf,
                              torch.from_numpy(oc).float().cuda(), ws)
    torch.cuda.synchronize()
    assert vsa.lib().vsa_check_device_status(vsa._ptr(ws), vsa._stream()) == vsa.OK
    for (b, h), hd in heads.items():
        for c in cubes_of(wl, name == "tiny", seed=h):
            _, of_r, lse_r = hd.rows(c)
            sl = slice(c * 64, (c + 1) * 64)
            assert_close("O_f", to_np(of[b, h, sl]), of_r)
            assert_close("lse_f", to_np(lse[b, h, sl]), lse_r)
            assert_close("O", to_np(o[b, h, sl]), hd.output_tiled(c))


# ------------------------------------------------------------------ edge cases

def _custom(T, H, W, D, topk, seed, select="topk", heads=2, batch=1):
    wl = synth.Workload(f"edge_{T}x{H}x{W}_d{D}_k{topk}", batch, heads, D, T, H, W, select,
                        topk=topk, seed=seed)
    inp = synth.Inputs(wl, with_grad=True)
    enforce_gaps(inp)
    return inp


@pytest.mark.parametrize("thw,D,topk", [
    ((4, 4, 12), 64, 2),    # odd number of cubes: the last pair has one cube
    ((4, 4, 4), 128, 1),    # a single cube
    ((8, 4, 12), 128, 5),   # odd K, tail step with one key cube
    ((4, 8, 8), 64, 4),     # K = all cubes
])
def test_forward_edge_shapes(thw, D, topk):
    check_forward(_custom(*thw, D, topk, seed=7 + topk), full=True)


@pytest.mark.parametrize("thw,select,k", [
    ((16, 32, 32), "mass", 100),   # mass rule with kmax > 64: the shared-memory selection
    ((16, 32, 192), "topk", 32),   # 1,536 cubes: rows of 48 values per lane
    ((16, 32, 288), "topk", 32),   # 2,304 cubes: beyond the register rows
])
def test_selection_paths(thw, select, k):
    """Lists, counts, lse_c and O_c against the oracle on the selection's
    less common paths (row lengths and list capacities)."""
    T, H, W = thw
    wl = synth.Workload(f"sel_{T}x{H}x{W}_{select}{k}", 1, 1, 64, T, H, W, select,
                        topk=k, kmin=8, kmax=k, amplitude=1.3 if select == "mass" else 1.0,
                        seed=41 + k)
    inp = synth.Inputs(wl, with_grad=False)
    enforce_gaps(inp)
    _, _, _, _, v = run_forward(inp)
    hd = O.head_of(inp, 0, 0)
    assert np.array_equal(v["cnt"][0, 0].cpu().numpy(), hd.cnt)
    assert np.array_equal(v["idx"][0, 0].cpu().numpy(), hd.idx)
    assert_close("lse_c", to_np(v["lse_c"][0, 0]), hd.coarse["lse"])
    assert_close("O_c", to_np(v["oc"][0, 0]), hd.coarse["out"])


def test_full_selection_with_fine_only_gates_is_dense_attention():
    """K = all cubes, G_c = 0, G_f = 1: the output is dense softmax attention."""
    inp = _custom(4, 8, 8, 64, 4, seed=11)
    inp.gc = torch.zeros_like(inp.gc)
    inp.gf = torch.ones_like(inp.gf)
    wl = inp.wl
    _, t, _, o, _ = run_forward(inp)
    for h in range(wl.heads):
        q, k, v = (O.f64(getattr(inp, n)[0, h]) for n in ("q", "k", "v"))
        s = q @ k.T / np.sqrt(wl.head_dim)
        p = np.exp(s - s.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        assert_close("dense", to_np(o[0, h]), p @ v)


def test_fine_gates_zero_gives_repeated_coarse_output():
    inp = _custom(8, 8, 8, 64, 2, seed=12)
    inp.gf = torch.zeros_like(inp.gf)
    inp.gc = torch.ones_like(inp.gc)
    wl = inp.wl
    _, _, _, o, v = run_forward(inp)
    oc = to_np(v["oc"])
    for h in range(wl.heads):
        for c in range(wl.cubes):
            rows = synth.raster_rows_of_cube(wl, c)
            ref = np.broadcast_to(oc[0, h, c], (64, wl.head_dim))
            # O is bf16: equal to the bf16 rounding of O_c
            want = torch.from_numpy(np.ascontiguousarray(ref)).float().to(torch.bfloat16).double().numpy()
            assert np.array_equal(to_np(o[0, h])[rows], want)


def test_bad_index_lists_are_reported_not_faulted():
    """Out-of-range ids, unsorted lists and bad counts: flagged, dropped, no fault."""
    inp = _custom(8, 8, 8, 64, 2, seed=13)
    wl = inp.wl
    cfg = vsa.config_for(wl, layout="cube")
    t = cuda_inputs(inp)
    ws = torch.empty(vsa.workspace_bytes(cfg, False), dtype=torch.uint8, device="cuda")
    vsa.lib().vsa_reset_device_status(vsa._ptr(ws), vsa._stream())
    q, k, v = (vsa.stage(cfg, vsa.permute(cfg, t[n]), ws) for n in ("q", "k", "v"))
    idx = torch.tensor([[[[0, 1]] * wl.cubes] * wl.heads], dtype=torch.int32)
    idx[0, 0, 1] = torch.tensor([5, 99])       # id out of range
    idx[0, 0, 2] = torch.tensor([-3, 1])       # negative id
    idx[0, 1, 3] = torch.tensor([4, 2])        # not ascending
    cnt = torch.full((1, wl.heads, wl.cubes), 2, dtype=torch.int32)
    cnt[0, 1, 5] = 7                           # count above capacity
    oc = torch.zeros(1, wl.heads, wl.cubes, wl.head_dim, device="cuda")
    vsa.fine_fwd(cfg, q, k, v, idx.cuda(), cnt.cuda(), t["gc"], t["gf"], oc, ws)
    torch.cuda.synchronize()
    st = vsa.lib().vsa_check_device_status(vsa._ptr(ws), vsa._stream())
    assert st == vsa.ERR_DEVICE_CHECK
    # the context is still usable
    assert torch.cuda.is_available() and (torch.ones(4, device="cuda") * 2).sum().item() == 8


def test_values_outside_fp16_range_are_reported():
    inp = _custom(4, 4, 8, 64, 1, seed=15)
    wl = inp.wl
    cfg = vsa.config_for(wl)
    q = inp.q.clone()
    q[0, 1, 77, 5] = 1.0e5
    ws = torch.empty(vsa.workspace_bytes(cfg, False), dtype=torch.uint8, device="cuda")
    vsa.lib().vsa_reset_device_status(vsa._ptr(ws), vsa._stream())
    vsa.stage(cfg, inp.k.cuda(), ws)
    assert vsa.lib().vsa_check_device_status(vsa._ptr(ws), vsa._stream()) == vsa.OK
    vsa.stage(cfg, q.cuda(), ws)
    assert vsa.lib().vsa_check_device_status(vsa._ptr(ws), vsa._stream()) == vsa.ERR_DEVICE_CHECK


def test_worked_example_ties_keep_lower_ids():
    """Q = 0: all logits tie; top-1 keeps cube 0 and O_f is cube 0's mean of V."""
    inp = _custom(4, 4, 8, 64, 1, seed=14)
    inp.q = torch.zeros_like(inp.q)
    wl = inp.wl
    _, _, _, o, v = run_forward(inp)
    assert v["idx"].cpu().flatten().tolist() == [0] * (wl.heads * wl.cubes)
    vt = O.tile(O.f64(inp.v[0, 0]), wl.T, wl.H, wl.W)
    assert_close("O_f", to_np(v["o_f"][0, 0]), np.broadcast_to(vt[:64].mean(0), (128, 64)))


@pytest.mark.parametrize("thw,D,layout", [((8, 8, 8), 64, "raster"), ((8, 4, 12), 128, "raster"),
                                          ((8, 4, 12), 128, "cube")])
def test_inference_forward_in_its_smaller_saved_buffer(thw, D, layout):
    """vsa_forward(with_backward=0) into a saved buffer of vsa_saved_bytes_for(cfg, 0)
    (no O_f; staged copies only where inference stages) gives the output and
    the saved coarse results of the training-sized buffer, bit for bit."""
    inp = _custom(*thw, D, 2, seed=5)
    cfg = vsa.config_for(inp.wl, layout)
    t = cuda_inputs(inp)
    if layout == "cube":
        for n in ("q", "k", "v", "gc", "gf"):
            t[n] = vsa.permute(cfg, t[n])
    outs = []
    for small in (False, True):
        bufs = vsa.Buffers(cfg, "cuda", with_backward=False, inference_only=small)
        if small:
            assert bufs.saved.numel() < vsa.saved_layout(cfg).total
        o = vsa.forward(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs, with_backward=False)
        torch.cuda.synchronize()
        assert bufs.device_status() == vsa.OK
        wl = inp.wl
        B, H, N, nc, cap = wl.batch, wl.heads, wl.tokens, wl.cubes, wl.list_capacity
        outs.append([o.clone(), bufs.view("idx", torch.int32, (B, H, nc, cap)).clone(),
                     bufs.view("oc", torch.float32, (B, H, nc, D)).clone(),
                     bufs.view("lse_f", torch.float32, (B, H, N)).clone()])
    for a, b in zip(*outs):
        assert torch.equal(a, b)
