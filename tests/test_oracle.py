"""Pins for the fp64 oracle, against things other than the oracle itself.

Each test pins one part of the oracle to the pages or to mathematics:
brute-force loops in plain Python, exact rational arithmetic, closed forms,
invariants, finite differences, hand-derived worked examples.  A plausible
mistake in the oracle (a dropped term, a wrong sign or index, a transposed
operand, a wrong tie-break) fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import vsa_oracle as O
from trainable_block_sparse_gb300 import synth


def _rng(seed=0):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- tile / untile

@pytest.mark.parametrize("thw", [(8, 8, 8), (4, 8, 12), (12, 4, 8)])
def test_tile_matches_index_formula(thw):
    T, H, W = thw
    N = T * H * W
    x = np.arange(N, dtype=np.float64)[:, None] * np.ones((1, 3))
    xt = O.tile(x, T, H, W)
    # brute force: raster (t,h,w) goes to row c*64 + o
    for t in range(T):
        for h in range(H):
            for w in range(W):
                r = (t * H + h) * W + w
                c = ((t // 4) * (H // 4) + h // 4) * (W // 4) + w // 4
                o = (t % 4) * 16 + (h % 4) * 4 + (w % 4)
                assert xt[c * 64 + o, 0] == r
    # bijection and exact inverse
    assert sorted(xt[:, 0].tolist()) == list(range(N))
    assert np.array_equal(O.untile(xt, T, H, W), x)


def test_tile_keeps_cubes_spatially_contiguous():
    T, H, W = 8, 8, 12
    N = T * H * W
    coords = np.array([(t, h, w) for t in range(T) for h in range(H) for w in range(W)], float)
    ct = O.tile(coords, T, H, W).reshape(N // 64, 64, 3)
    # every tile spans exactly a 4x4x4 box aligned to multiples of 4
    span = ct.max(axis=1) - ct.min(axis=1)
    assert np.all(span == 3)
    assert np.all(ct.min(axis=1) % 4 == 0)


# ---------------------------------------------------------------- cube means

def test_cube_means_are_exact_rational_means():
    wl = synth.WORKLOADS["tiny"]
    inp = synth.Inputs(wl, with_grad=False)
    q = O.f64(inp.q[0, 1])
    qt = O.tile(q, wl.T, wl.H, wl.W)
    qc = O.cube_means(qt)
    rows = synth.raster_rows_of_cube(wl, 5)
    for d in (0, 17, 63):
        exact = sum(Fraction(float(q[r, d])) for r in rows) / 64
        assert Fraction(float(qc[5, d])) == exact


# ---------------------------------------------------------------- coarse stage

def _py_softmax_attention(q, k, v, scale):
    """Plain-Python loops: logits, probabilities, output, lse."""
    n, m, dv = len(q), len(k), len(v[0])
    logits = [[scale * sum(q[i][d] * k[j][d] for d in range(len(q[0]))) for j in range(m)]
              for i in range(n)]
    probs, out, lse = [], [], []
    for i in range(n):
        mx = max(logits[i])
        e = [math.exp(s - mx) for s in logits[i]]
        z = sum(e)
        probs.append([x / z for x in e])
        out.append([sum(probs[i][j] * v[j][d] for j in range(m)) for d in range(dv)])
        lse.append(mx + math.log(z))
    return logits, probs, out, lse


def test_coarse_attention_bruteforce():
    r = _rng(1)
    qc, kc, vc = r.normal(size=(6, 5)), r.normal(size=(6, 5)), r.normal(size=(6, 3))
    res = O.coarse_attention(qc, kc, vc, 0.7)
    lg, pr, out, lse = _py_softmax_attention(qc.tolist(), kc.tolist(), vc.tolist(), 0.7)
    np.testing.assert_allclose(res["logits"], lg, rtol=0, atol=1e-13)
    np.testing.assert_allclose(res["probs"], pr, rtol=0, atol=1e-13)
    np.testing.assert_allclose(res["out"], out, rtol=0, atol=1e-13)
    np.testing.assert_allclose(res["lse"], lse, rtol=0, atol=1e-13)


def test_coarse_identical_keys_give_uniform_attention():
    r = _rng(2)
    qc = r.normal(size=(4, 8))
    kc = np.tile(r.normal(size=(1, 8)), (5, 1))
    vc = r.normal(size=(5, 8))
    res = O.coarse_attention(qc, kc, vc, 0.3)
    np.testing.assert_allclose(res["probs"], 0.2, atol=1e-15)
    np.testing.assert_allclose(res["out"], np.tile(vc.mean(0), (4, 1)), atol=1e-14)


# ---------------------------------------------------------------- selection

def test_topk_properties_and_full_sort():
    r = _rng(3)
    logits = r.normal(size=(2, 9, 40))
    idx, cnt = O.select_topk(logits, 7)
    assert idx.shape == (2, 9, 7) and np.all(cnt == 7)
    for b in range(2):
        for i in range(9):
            row = logits[b, i]
            sel = idx[b, i]
            assert list(sel) == sorted(sel)
            assert len(set(sel.tolist())) == 7
            assert int(np.argmax(row)) in sel
            unsel = np.setdiff1d(np.arange(40), sel)
            assert row[sel].min() >= row[unsel].max()
            by_sort = sorted(range(40), key=lambda j: (-row[j], j))[:7]
            assert sorted(by_sort) == sel.tolist()


def test_topk_ties_keep_lower_ids():
    logits = np.array([[1.0, 3.0, 3.0, 0.0, 3.0]])
    idx, _ = O.select_topk(logits, 2)
    assert idx.tolist() == [[1, 2]]
    idx, _ = O.select_topk(np.zeros((1, 6)), 3)
    assert idx.tolist() == [[0, 1, 2]]
    # many equal scores: the kept ones are the lowest ids among the ties
    row = np.zeros((1, 300))
    row[0, ::7] = 1.0
    idx, _ = O.select_topk(row, 60)
    top = list(range(0, 300, 7))
    rest = [j for j in range(300) if j % 7][: 60 - len(top)]
    assert idx.tolist() == [sorted(top + rest)]


def test_topk_rejects_bad_k():
    with pytest.raises(ValueError):
        O.select_topk(np.zeros((2, 4)), 5)
    with pytest.raises(ValueError):
        O.select_topk(np.zeros((2, 4)), 0)


@pytest.mark.parametrize("temp", [0.3, 1.0, 4.0])
def test_mass_selection_properties(temp):
    r = _rng(4)
    logits = r.normal(size=(30, 100)) * temp
    probs, _ = O.softmax_rows(logits)
    idx, cnt = O.select_mass(logits, probs, 0.9, 8, 64)
    for i in range(30):
        n = cnt[i]
        assert 8 <= n <= 64
        sel = idx[i, :n]
        assert np.all(idx[i, n:] == -1)
        assert list(sel) == sorted(sel)
        order = sorted(range(100), key=lambda j: (-logits[i, j], j))
        assert sorted(order[:n]) == sel.tolist()
        top = [probs[i, j] for j in order]
        if n < 64:
            assert sum(top[:n]) >= 0.9
        if n > 8:
            assert sum(top[: n - 1]) < 0.9


def test_mass_selection_clamps():
    # one dominant cube: raw count 1, clamped up to kmin
    logits = np.array([[20.0] + [0.0] * 15])
    probs, _ = O.softmax_rows(logits)
    idx, cnt = O.select_mass(logits, probs, 0.9, 4, 8)
    assert cnt.tolist() == [4] and idx[0, :4].tolist() == [0, 1, 2, 3]
    # uniform row: raw count ceil(0.9*16) = 15, clamped down to kmax
    logits = np.zeros((1, 16))
    probs, _ = O.softmax_rows(logits)
    _, cnt = O.select_mass(logits, probs, 0.9, 4, 8)
    assert cnt.tolist() == [8]
    _, cnt = O.select_mass(logits, probs, 0.9, 4, 16)
    assert cnt.tolist() == [15]


# ---------------------------------------------------------------- fine stage

def _small_head(seed, T=4, H=4, W=8, D=8, gc=None, gf=None, sel=None, fixed=None):
    r = _rng(seed)
    N = T * H * W
    q, k, v = (r.normal(size=(N, D)) for _ in range(3))
    gc = r.uniform(size=(N, D)) if gc is None else gc
    gf = r.uniform(size=(N, D)) if gf is None else gf
    sel = sel or {"mode": "topk", "topk": 1, "mass": 0.9, "kmin": 1, "kmax": 2}
    return O.Head(q, k, v, gc, gf, T, H, W, sel, fixed=fixed), (q, k, v, gc, gf)


def test_full_selection_is_dense_softmax_attention():
    """K = all cubes, G_c = 0, G_f = 1 starts 'equivalent to full attention'."""
    T, H, W, D = 4, 4, 8, 8
    N = T * H * W
    zeros, ones = np.zeros((N, D)), np.ones((N, D))
    hd, (q, k, v, _, _) = _small_head(5, T, H, W, D, gc=zeros, gf=ones,
                                      sel={"mode": "topk", "topk": 2})
    o, _, lse_t = hd.forward_all()
    scale = 1.0 / math.sqrt(D)
    _, _, out, lse = _py_softmax_attention(q.tolist(), k.tolist(), v.tolist(), scale)
    np.testing.assert_allclose(o, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(O.untile(lse_t[:, None], T, H, W)[:, 0], lse, atol=1e-12)


def test_masked_equals_attention_over_gathered_keys():
    """Masked dense softmax == softmax over only the selected tiles' keys."""
    T, H, W, D = 8, 4, 8, 16
    r = _rng(6)
    N = T * H * W
    q, k, v = (r.normal(size=(N, D)) for _ in range(3))
    qt, kt, vt = (O.tile(x, T, H, W) for x in (q, k, v))
    nc = N // 64
    scale = 0.25
    for c in range(nc):
        sel = np.sort(r.choice(nc, size=2, replace=False))
        p, of, lse = O.fine_rows(qt[c * 64:(c + 1) * 64], kt, vt, sel, 2, scale)
        keys = np.concatenate([np.arange(j * 64, (j + 1) * 64) for j in sel])
        s = scale * qt[c * 64:(c + 1) * 64] @ kt[keys].T
        w = np.exp(s - s.max(1, keepdims=True))
        w /= w.sum(1, keepdims=True)
        np.testing.assert_allclose(of, w @ vt[keys], atol=1e-13)
        assert np.all(p[:, np.setdiff1d(np.arange(N), keys)] == 0)
        np.testing.assert_allclose(p.sum(1), 1.0, atol=1e-14)


def test_combine_special_cases():
    T, H, W, D = 4, 4, 8, 8
    N = T * H * W
    r = _rng(7)
    gc = r.uniform(size=(N, D))
    hd0, _ = _small_head(8, gc=gc, gf=np.zeros((N, D)))
    o0, _, _ = hd0.forward_all()
    rep = np.repeat(hd0.coarse["out"], 64, axis=0)
    assert np.array_equal(O.tile(o0, T, H, W), rep * O.tile(gc, T, H, W))
    gf = r.uniform(size=(N, D))
    hd1, _ = _small_head(8, gc=np.zeros((N, D)), gf=gf)
    o1, of1, _ = hd1.forward_all()
    assert np.array_equal(O.tile(o1, T, H, W), of1 * O.tile(gf, T, H, W))


# ---------------------------------------------------------------- worked example

def _uniform_two_cubes(golden_dir, topk):
    g = json.load(open(os.path.join(golden_dir, "uniform_two_cubes.json")))
    T, H, W, D = g["T"], g["H"], g["W"], g["head_dim"]
    N = T * H * W
    r = np.arange(N)
    v = np.stack([r, r % W], axis=1).astype(np.float64)
    q = np.zeros((N, D))
    k = _rng(9).normal(size=(N, D))
    ones = np.ones((N, D))
    hd = O.Head(q, k, v, ones, ones, T, H, W, {"mode": "topk", "topk": topk})
    hd.set_grad(ones)
    return g, hd


def test_worked_example_top1(golden_dir):
    g, hd = _uniform_two_cubes(golden_dir, 1)
    e = g["topk1"]
    assert hd.idx.tolist() == e["idx"]
    np.testing.assert_allclose(hd.coarse["out"], e["coarse_out"], atol=1e-12)
    np.testing.assert_allclose(hd.coarse["lse"], e["coarse_lse"], atol=1e-12)
    o, of, lse = hd.forward_all()
    np.testing.assert_allclose(of, np.tile(e["fine_out_every_token"], (128, 1)), atol=1e-12)
    np.testing.assert_allclose(lse, e["fine_lse_every_token"], atol=1e-12)
    np.testing.assert_allclose(o, np.tile(e["out_every_token"], (128, 1)), atol=1e-12)
    dq, dk, dv, dgc, dgf = hd.backward_all()
    dvt = O.tile(dv, 4, 4, 8)
    np.testing.assert_allclose(dvt[:64], np.tile(e["dv_cube0_token"], (64, 1)), atol=1e-12)
    np.testing.assert_allclose(dvt[64:], np.tile(e["dv_cube1_token"], (64, 1)), atol=1e-12)
    np.testing.assert_allclose(dgc, np.tile(e["dgc_every_token"], (128, 1)), atol=1e-12)
    np.testing.assert_allclose(dgf, np.tile(e["dgf_every_token"], (128, 1)), atol=1e-12)


def test_worked_example_top2(golden_dir):
    g, hd = _uniform_two_cubes(golden_dir, 2)
    e = g["topk2"]
    assert hd.idx.tolist() == e["idx"]
    o, of, _ = hd.forward_all()
    np.testing.assert_allclose(of, np.tile(e["fine_out_every_token"], (128, 1)), atol=1e-12)
    np.testing.assert_allclose(o, np.tile(e["out_every_token"], (128, 1)), atol=1e-12)


# ---------------------------------------------------------------- gradients

def _loss(q, k, v, gc, gf, do, T, H, W, sel, fixed):
    hd = O.Head(q, k, v, gc, gf, T, H, W, sel, fixed=fixed)
    return float(np.sum(hd.forward_all()[0] * do))


@pytest.mark.parametrize("mode", ["topk", "mass"])
def test_gradients_match_central_differences(mode):
    T, H, W, D = 8, 4, 8, 8
    N = T * H * W
    r = _rng(10)
    q, k, v = (r.normal(size=(N, D)) for _ in range(3))
    gc, gf = r.uniform(size=(N, D)), r.uniform(size=(N, D))
    do = r.normal(size=(N, D))
    sel = {"mode": mode, "topk": 2, "mass": 0.6, "kmin": 1, "kmax": 3}
    hd = O.Head(q, k, v, gc, gf, T, H, W, sel)
    fixed = (hd.idx.copy(), hd.cnt.copy())
    hd.set_grad(do)
    grads = hd.backward_all()
    tensors = [q, k, v, gc, gf]
    h = 1e-6
    for ti, g in enumerate(grads):
        for _ in range(40):
            i, d = int(r.integers(N)), int(r.integers(D))
            xs_p = [x.copy() for x in tensors]
            xs_m = [x.copy() for x in tensors]
            xs_p[ti][i, d] += h
            xs_m[ti][i, d] -= h
            fd = (_loss(*xs_p, do, T, H, W, sel, fixed) - _loss(*xs_m, do, T, H, W, sel, fixed)) / (2 * h)
            assert abs(fd - g[i, d]) <= 1e-6 * max(1.0, abs(fd)), (ti, i, d, fd, g[i, d])


def test_gradient_invariants():
    """Shift invariance of keys and the closed form of sum(dV)."""
    T, H, W, D = 8, 8, 8, 8
    hd, (q, k, v, gc, gf) = _small_head(11, T, H, W, D,
                                        sel={"mode": "topk", "topk": 3})
    do = _rng(12).normal(size=(T * H * W, D))
    hd.set_grad(do)
    dq, dk, dv, dgc, dgf = hd.backward_all()
    # adding one vector to every key shifts each logit row by a constant
    np.testing.assert_allclose(dk.sum(0), 0.0, atol=1e-11)
    # adding c to every value adds c*(G_c+G_f) to the output
    np.testing.assert_allclose(dv.sum(0), (do * (gc + gf)).sum(0), atol=1e-11)
    # gates enter linearly
    o, of, _ = hd.forward_all()
    np.testing.assert_allclose(dgf, do * O.untile(of, T, H, W), atol=1e-14)


@pytest.mark.parametrize("mode", ["topk", "mass"])
def test_key_partials_sum_to_key_gradients(mode):
    """fine_key_partials over all query cubes (in any split) plus the pooled
    part equals grad_key_cube of every key cube, which the finite-difference
    test pins; forget() leaves results unchanged."""
    T, H, W, D = 8, 8, 12, 8
    sel = {"mode": mode, "topk": 4, "mass": 0.7, "kmin": 2, "kmax": 6}
    hd, _ = _small_head(13, T, H, W, D, sel=sel)
    hd.set_grad(_rng(14).normal(size=(T * H * W, D)))
    split = [list(range(0, 7)), list(range(7, hd.nc))]
    parts = [hd.fine_key_partials(cs) for cs in split]
    for c in range(hd.nc):
        hd.forget(c)
    dk = sum(p[0] for p in parts) + np.repeat(hd.dkc / 64, 64, axis=0)
    dv = sum(p[1] for p in parts) + np.repeat(hd.dvc / 64, 64, axis=0)
    for j in range(hd.nc):
        rk, rv = hd.grad_key_cube(j)
        np.testing.assert_allclose(dk[j * 64:(j + 1) * 64], rk, rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv[j * 64:(j + 1) * 64], rv, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- pages' facts

def test_workloads_match_pages_facts(golden_dir):
    f = json.load(open(os.path.join(golden_dir, "pages_facts.json")))
    assert synth.TILE == f["tile_tokens"]["value"] == 64
    assert [synth.CUBE_T, synth.CUBE_H, synth.CUBE_W] == f["cube_shape"]["value"]
    wl = synth.WORKLOADS["pretrain"]
    assert [wl.T, wl.H, wl.W] == f["pseudocode_video"]["value"]
    assert wl.topk == f["pseudocode_topk"]["value"] == f["default_topk"]["value"]
    assert 1 - wl.topk / wl.cubes == f["sparsity_tile64_pretrain"]["value"]


def test_coarse_flop_share_matches_pages(golden_dir):
    from trainable_block_sparse_gb300 import flops
    f = json.load(open(os.path.join(golden_dir, "pages_facts.json")))
    wl = synth.WORKLOADS["pretrain"]
    share = flops.coarse_fwd(wl) / flops.fine_fwd_topk(wl)
    assert share < f["coarse_flop_share_upper_16k"]["value"]
    for name in ("pretrain", "wan13b", "p720"):
        w = synth.WORKLOADS[name]
        assert flops.coarse_fwd(w) / flops.fine_fwd_topk(w) < f["coarse_flop_share_upper"]["value"]


# ---------------------------------------------------------------- generator

def test_generator_is_deterministic_and_redraw_is_local():
    wl = synth.WORKLOADS["tiny"]
    a = synth.Inputs(wl)
    b = synth.Inputs(wl)
    for n in ("q", "k", "v", "gc", "gf", "do"):
        assert torch.equal(getattr(a, n), getattr(b, n))
    before = a.q.clone()
    a.redraw_query_cube(0, 1, 3, attempt=1)
    changed = (a.q != before).any(-1)
    rows = set(synth.raster_rows_of_cube(wl, 3).tolist())
    assert set(torch.nonzero(changed[0, 1]).flatten().tolist()) <= rows
    assert not changed[0, 0].any()
    assert a.gc.min() > 0 and a.gc.max() < 1
