"""fp64 CPU oracle for VSA coarse-to-fine video sparse attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module: it
is used by tests/, by the smoke check in __graft_entry__.py and by the CPU
baseline leg of bench.py.  It shares no code with the CUDA library.

It restates, in plain numpy fp64 on the exact bf16 input values, what the
method computes ("VSA: Faster Video Diffusion with Trainable Sparse
Attention"; the section numbers below are those of that page's summary):

1. tile: raster (T,H,W) tokens -> cube-major order, cube (4,4,4) = 64 tokens
   (§1 "VSA", §2 "VSA design", App. B "Pseudocode of VSA").
2. coarse inputs: per-cube means of Q, K, V (§2 "Coarse stage"; App. B).
3. coarse attention: A_c = softmax(Q_c K_c^T * scale), O_c = A_c V_c, dense over
   all cubes (§2 "Coarse stage"; the Chinese notes' 关键设计 1).
4. selection: the K largest entries of each A_c row (App. B: keep top-k blocks),
   or, for the dynamic-compute variant, the smallest top-ranked set whose
   coarse mass reaches a threshold, clamped to [kmin, kmax] (the variable
   per-query count of "Improving Video Sparse Attention with Fine-grained
   Router and Sparse Rebasing", abstract).
5. fine attention: token-level Q K^T over all keys, unselected blocks masked,
   softmax, times V (App. B "fine stage"; §2 "Fine stage").
6. combine: O = repeat(O_c over its cube) * G_c + O_f * G_f (App. B: coarse
   output repeated across each block; the notes' 关键设计 3 gating formula).
7. untile back to raster order (App. B).
8. gradients: the analytic derivatives of 2-6 with the selection held fixed
   (the method trains end to end, abstract; selection is piecewise constant).

Readings where the pages are silent: row-major token order inside and across
cubes; the coarse stage uses the same scale 1/sqrt(D) as the fine stage; ties
in selection go to the lower cube id; index lists are stored ascending and
padded with -1; the selection ranks logits (softmax is monotone, so this is
the same set as ranking A_c).
"""
from __future__ import annotations

import numpy as np
import torch

CUBE = 4
TILE = 64


# ---------------------------------------------------------------------------
# conversions
# ---------------------------------------------------------------------------

def f64(x) -> np.ndarray:
    """Exact fp64 copy of a CPU tensor (bf16/fp32) or array."""
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# 1. tile / untile  (App. B: tiling and untiling rearrange tokens)
# ---------------------------------------------------------------------------

def tile(x: np.ndarray, T: int, H: int, W: int) -> np.ndarray:
    """[..., T*H*W, D] raster -> [..., T*H*W, D] cube-major.

    Output row c*64 + o holds raster token (t, h, w) with
    c = ((t//4)*(H//4) + h//4)*(W//4) + w//4 and o = (t%4)*16 + (h%4)*4 + w%4.
    """
    lead = x.shape[:-2]
    D = x.shape[-1]
    y = x.reshape(*lead, T // CUBE, CUBE, H // CUBE, CUBE, W // CUBE, CUBE, D)
    n = len(lead)
    order = list(range(n)) + [n + 0, n + 2, n + 4, n + 1, n + 3, n + 5, n + 6]
    return y.transpose(order).reshape(*lead, T * H * W, D)


def untile(x: np.ndarray, T: int, H: int, W: int) -> np.ndarray:
    """Inverse of tile()."""
    lead = x.shape[:-2]
    D = x.shape[-1]
    y = x.reshape(*lead, T // CUBE, H // CUBE, W // CUBE, CUBE, CUBE, CUBE, D)
    n = len(lead)
    order = list(range(n)) + [n + 0, n + 3, n + 1, n + 4, n + 2, n + 5, n + 6]
    return y.transpose(order).reshape(*lead, T * H * W, D)


# ---------------------------------------------------------------------------
# 2. cube means  (§2 Coarse stage: mean-pool each cube)
# ---------------------------------------------------------------------------

def cube_means(xt: np.ndarray) -> np.ndarray:
    """[..., Nc*64, D] cube-major -> [..., Nc, D]: mean of each cube's 64 tokens."""
    lead = xt.shape[:-2]
    N, D = xt.shape[-2:]
    return xt.reshape(*lead, N // TILE, TILE, D).mean(axis=-2)


# ---------------------------------------------------------------------------
# 3. coarse attention  (§2 Coarse stage; 关键设计 1: A_c and O_c)
# ---------------------------------------------------------------------------

def softmax_rows(s: np.ndarray):
    """Row softmax with its log-sum-exp.  Rows of -inf only are not allowed."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    z = np.sum(e, axis=-1, keepdims=True)
    return e / z, (m + np.log(z))[..., 0]


def coarse_attention(qc, kc, vc, scale):
    """Dense attention on the pooled sequence.  Returns logits, A_c, O_c, lse_c."""
    logits = scale * (qc @ np.swapaxes(kc, -1, -2))
    a, lse = softmax_rows(logits)
    return {"logits": logits, "probs": a, "out": a @ vc, "lse": lse}


# ---------------------------------------------------------------------------
# 4. selection  (App. B: keep the top-k blocks; VSA2 abstract: variable count)
# ---------------------------------------------------------------------------

def rank_desc(row: np.ndarray) -> np.ndarray:
    """Cube ids ordered by descending score; equal scores keep the lower id first."""
    return np.argsort(-row, kind="stable")


def select_topk(logits: np.ndarray, k: int):
    """Per row: the k highest-scoring cubes, ascending ids.  Returns (idx, cnt)."""
    nc = logits.shape[-1]
    if not 1 <= k <= nc:
        raise ValueError("top-k must lie in [1, number of cubes]")
    flat = logits.reshape(-1, nc)
    idx = np.empty((flat.shape[0], k), np.int32)
    for r in range(flat.shape[0]):
        idx[r] = np.sort(rank_desc(flat[r])[:k])
    cnt = np.full(flat.shape[0], k, np.int32)
    return idx.reshape(*logits.shape[:-1], k), cnt.reshape(logits.shape[:-1])


def select_mass(logits: np.ndarray, probs: np.ndarray, mass: float, kmin: int, kmax: int):
    """Per row: smallest top-ranked set with sum of A_c >= mass, count clamped.

    The count is clamped to [kmin, kmax] (and to the number of cubes).  Lists
    are ascending and padded with -1 up to kmax.
    """
    nc = logits.shape[-1]
    kmax_eff = min(kmax, nc)
    kmin_eff = min(kmin, kmax_eff)
    fl = logits.reshape(-1, nc)
    fp = probs.reshape(-1, nc)
    idx = np.full((fl.shape[0], kmax), -1, np.int32)
    cnt = np.empty(fl.shape[0], np.int32)
    for r in range(fl.shape[0]):
        order = rank_desc(fl[r])
        csum = np.cumsum(fp[r][order])
        hit = np.nonzero(csum >= mass)[0]
        n_raw = int(hit[0]) + 1 if hit.size else nc
        n = min(max(n_raw, kmin_eff), kmax_eff)
        cnt[r] = n
        idx[r, :n] = np.sort(order[:n])
    return idx.reshape(*logits.shape[:-1], kmax), cnt.reshape(logits.shape[:-1])


def selection_mask(idx_row: np.ndarray, cnt: int, nc: int) -> np.ndarray:
    """Token-level key mask [Nc*64] for one query cube: True where the key's cube is selected."""
    sel = np.zeros(nc, bool)
    sel[idx_row[:cnt]] = True
    return np.repeat(sel, TILE)


# ---------------------------------------------------------------------------
# 5. fine attention  (App. B: QK^T, mask unselected, softmax, times V)
# ---------------------------------------------------------------------------

def fine_rows(qt, kt, vt, idx_row, cnt, scale):
    """Masked dense attention for the 64 query rows of one cube (one head).

    qt: [64, D] rows of this cube; kt, vt: [N, D] all keys/values (cube-major).
    Returns (P [64, N] with zeros at masked keys, O_f [64, D], lse_f [64]).
    """
    nc = kt.shape[0] // TILE
    s = scale * (qt @ kt.T)
    s = np.where(selection_mask(idx_row, cnt, nc)[None, :], s, -np.inf)
    p, lse = softmax_rows(s)
    return p, p @ vt, lse


# ---------------------------------------------------------------------------
# one (batch, head) slice, forward and backward
# ---------------------------------------------------------------------------

class Head:
    """Forward and backward of one (batch, head) slice.

    q, k, v, gc, gf, do: fp64 [N, D] in raster order.  sel: dict with
    mode ("topk"/"mass"), topk, mass, kmin, kmax.  Fine-stage work is done
    only for the query cubes asked for, so large layers can be sampled.
    """

    def __init__(self, q, k, v, gc, gf, T, H, W, sel, scale=None, fixed=None):
        self.T, self.H, self.W = T, H, W
        self.N, self.D = q.shape
        self.nc = self.N // TILE
        self.scale = 1.0 / np.sqrt(self.D) if scale is None else scale
        self.qt, self.kt, self.vt = (tile(x, T, H, W) for x in (q, k, v))
        self.gct, self.gft = tile(gc, T, H, W), tile(gf, T, H, W)
        self.qc, self.kc, self.vc = (cube_means(x) for x in (self.qt, self.kt, self.vt))
        self.coarse = coarse_attention(self.qc, self.kc, self.vc, self.scale)
        if fixed is not None:
            # selection held constant (gradients treat it as piecewise constant)
            self.idx, self.cnt = fixed
        elif sel["mode"] == "topk":
            self.idx, self.cnt = select_topk(self.coarse["logits"], sel["topk"])
        else:
            self.idx, self.cnt = select_mass(self.coarse["logits"], self.coarse["probs"],
                                             sel["mass"], sel["kmin"], sel["kmax"])
        self._rows = {}
        self._grad_rows = {}

    def rows(self, c):
        """P, O_f, lse_f of query cube c (cached)."""
        if c not in self._rows:
            r = slice(c * TILE, (c + 1) * TILE)
            self._rows[c] = fine_rows(self.qt[r], self.kt, self.vt, self.idx[c],
                                      self.cnt[c], self.scale)
        return self._rows[c]

    def output_tiled(self, c):
        """Combined output O (cube-major rows) of query cube c."""
        r = slice(c * TILE, (c + 1) * TILE)
        of = self.rows(c)[1]
        return self.coarse["out"][c][None, :] * self.gct[r] + of * self.gft[r]

    def forward_all(self):
        """O, O_f, lse_f for every cube; O in raster order, O_f/lse_f cube-major."""
        of = np.concatenate([self.rows(c)[1] for c in range(self.nc)])
        lse = np.concatenate([self.rows(c)[2] for c in range(self.nc)])
        o_t = np.concatenate([self.output_tiled(c) for c in range(self.nc)])
        return untile(o_t, self.T, self.H, self.W), of, lse

    # -- backward ------------------------------------------------------------

    def set_grad(self, do):
        """Upstream dO (raster, fp64).  Computes the coarse-branch gradients."""
        self.dot = tile(do, self.T, self.H, self.W)
        # dO_c: the coarse output is repeated over its cube, so its gradient sums
        dOc = (self.dot * self.gct).reshape(self.nc, TILE, self.D).sum(axis=1)
        a = self.coarse["probs"]
        # softmax backward, written as the Jacobian-vector product per row
        dA = dOc @ self.vc.T
        dL = a * (dA - np.sum(a * dA, axis=1, keepdims=True))
        self.dqc = self.scale * dL @ self.kc
        self.dkc = self.scale * dL.T @ self.qc
        self.dvc = a.T @ dOc
        self.dOc = dOc

    def _fine_grad_rows(self, c):
        """P, dS and dO_f of query cube c (fine branch; cached like rows())."""
        if c not in self._grad_rows:
            r = slice(c * TILE, (c + 1) * TILE)
            p = self.rows(c)[0]
            dof = self.dot[r] * self.gft[r]
            dp = dof @ self.vt.T
            ds = p * (dp - np.sum(p * dp, axis=1, keepdims=True))
            self._grad_rows[c] = (p, ds, dof)
        return self._grad_rows[c]

    def forget(self, c):
        """Drops the cached rows of query cube c (a [64, N] P per cube adds up
        to gigabytes on large slices).  Results do not change."""
        self._rows.pop(c, None)
        self._grad_rows.pop(c, None)

    def grad_query_cube(self, c):
        """dQ, dG_c, dG_f for the 64 tokens of query cube c (cube-major rows)."""
        r = slice(c * TILE, (c + 1) * TILE)
        _, ds, _ = self._fine_grad_rows(c)
        dq = self.scale * ds @ self.kt + self.dqc[c][None, :] / TILE
        dgc = self.dot[r] * self.coarse["out"][c][None, :]
        dgf = self.dot[r] * self.rows(c)[1]
        return dq, dgc, dgf

    def grad_key_cube(self, j):
        """dK, dV for the 64 tokens of key/value cube j (cube-major rows)."""
        cols = slice(j * TILE, (j + 1) * TILE)
        dk = np.repeat(self.dkc[j][None, :] / TILE, TILE, axis=0)
        dv = np.repeat(self.dvc[j][None, :] / TILE, TILE, axis=0)
        for c in range(self.nc):
            if j not in self.idx[c][: self.cnt[c]]:
                continue
            r = slice(c * TILE, (c + 1) * TILE)
            p, ds, dof = self._fine_grad_rows(c)
            dk = dk + self.scale * ds[:, cols].T @ self.qt[r]
            dv = dv + p[:, cols].T @ dof
        return dk, dv

    def fine_key_partials(self, cubes):
        """Fine-branch dK, dV [N, D] (cube-major rows) from the given query cubes.

        For every query cube c in `cubes` and every key cube j it selected, the
        two terms that grad_key_cube(j) adds for c: scale * dS[:, j]^T Q_c and
        P[:, j]^T dO_f,c; summed over `cubes`.  The pooled part is left out.
        Over all query cubes, plus repeat(dK_c)/64 and repeat(dV_c)/64, this is
        grad_key_cube for every key cube at once (each query cube's P and dS
        computed once instead of once per key cube it selected).
        """
        dk = np.zeros((self.N, self.D))
        dv = np.zeros((self.N, self.D))
        for c in cubes:
            r = slice(c * TILE, (c + 1) * TILE)
            p, ds, dof = self._fine_grad_rows(c)
            for j in self.idx[c][: self.cnt[c]]:
                cols = slice(j * TILE, (j + 1) * TILE)
                dk[cols] += self.scale * ds[:, cols].T @ self.qt[r]
                dv[cols] += p[:, cols].T @ dof
        return dk, dv

    def backward_all(self):
        """dQ, dK, dV, dG_c, dG_f for the whole slice, raster order."""
        parts = [self.grad_query_cube(c) for c in range(self.nc)]
        dq, dgc, dgf = (np.concatenate([p[i] for p in parts]) for i in range(3))
        kv = [self.grad_key_cube(j) for j in range(self.nc)]
        dk = np.concatenate([x[0] for x in kv])
        dv = np.concatenate([x[1] for x in kv])
        u = lambda x: untile(x, self.T, self.H, self.W)  # noqa: E731
        return u(dq), u(dk), u(dv), u(dgc), u(dgf)


def selection_of(wl) -> dict:
    return {"mode": wl.select, "topk": wl.topk, "mass": wl.mass,
            "kmin": wl.kmin, "kmax": wl.kmax}


def head_of(inputs, b: int, h: int, scale=None) -> Head:
    """Build the oracle's Head for one (batch, head) slice of a synth.Inputs."""
    wl = inputs.wl
    t = lambda x: f64(x[b, h])  # noqa: E731
    hd = Head(t(inputs.q), t(inputs.k), t(inputs.v), t(inputs.gc), t(inputs.gf),
              wl.T, wl.H, wl.W, selection_of(wl), scale)
    if inputs.do is not None:
        hd.set_grad(t(inputs.do))
    return hd


def forward(inputs, scale=None):
    """Whole-layer forward (small layers only): O raster, plus per-slice data."""
    wl = inputs.wl
    B, Hd = wl.batch, wl.heads
    o = np.empty((B, Hd, wl.tokens, wl.head_dim))
    heads = {}
    for b in range(B):
        for h in range(Hd):
            hd = head_of(inputs, b, h, scale)
            o[b, h] = hd.forward_all()[0]
            heads[(b, h)] = hd
    return o, heads


def backward(heads, wl):
    """Whole-layer gradients (small layers only), raster order, fp64."""
    shape = (wl.batch, wl.heads, wl.tokens, wl.head_dim)
    out = [np.empty(shape) for _ in range(5)]
    for (b, h), hd in heads.items():
        for arr, g in zip(out, hd.backward_all()):
            arr[b, h] = g
    return tuple(out)
