"""Test-side helpers: gap enforcement on the synthetic inputs (oracle logits),
and the parity check against the oracle's fp64 values."""
import numpy as np
import torch

from oracle import vsa_oracle as O

GAP = 1e-3       # smallest accepted logit gap at a selection boundary
MASS_MARGIN = 1e-4
ATOL = 2e-2      # max-abs error bound against the fp64 oracle
RTOL_L2 = 1e-2   # relative L2 error bound against the fp64 oracle


def _row_ok(logits_row, wl):
    """True when this row's selection cannot flip under ~1e-5 logit noise."""
    s = np.sort(logits_row)[::-1]
    nc = s.size
    if wl.select == "topk":
        k = wl.topk
        return k >= nc or s[k - 1] - s[k] >= GAP
    p = np.exp(s - s[0])
    p /= p.sum()
    csum = np.cumsum(p)
    hit = np.nonzero(csum >= wl.mass)[0]
    n_raw = int(hit[0]) + 1 if hit.size else nc
    kmax = min(wl.kmax, nc)
    cnt = min(max(n_raw, min(wl.kmin, kmax)), kmax)
    if cnt < nc and s[cnt - 1] - s[cnt] < GAP:
        return False
    if cnt >= 2 and s[cnt - 2] - s[cnt - 1] < GAP:
        return False
    for n in (cnt - 1, cnt):
        if n >= 1 and abs(csum[n - 1] - wl.mass) < MASS_MARGIN:
            return False
    return True


def enforce_gaps(inputs, max_attempts=200):
    """Redraws query cubes of `inputs` until every row's selection is unambiguous.

    Uses the oracle's fp64 logits of the bf16-rounded tensors.  Returns the
    number of redraws.
    """
    wl = inputs.wl
    scale = 1.0 / np.sqrt(wl.head_dim)
    redraws = 0
    for b in range(wl.batch):
        for h in range(wl.heads):
            kc = O.cube_means(O.tile(O.f64(inputs.k[b, h]), wl.T, wl.H, wl.W))
            qc = O.cube_means(O.tile(O.f64(inputs.q[b, h]), wl.T, wl.H, wl.W))
            logits = scale * qc @ kc.T
            for c in range(wl.cubes):
                attempt = 0
                while not _row_ok(logits[c], wl):
                    attempt += 1
                    if attempt > max_attempts:
                        raise RuntimeError(f"could not separate row {(b, h, c)}")
                    inputs.redraw_query_cube(b, h, c, attempt)
                    redraws += 1
                    rows = torch.from_numpy(_rows(wl, c))
                    qrow = O.f64(inputs.q[b, h, rows]).mean(axis=0)
                    logits[c] = scale * kc @ qrow
    return redraws


def _rows(wl, c):
    from trainable_block_sparse_gb300 import synth
    return synth.raster_rows_of_cube(wl, c)


def cuda_inputs(inputs):
    names = ("q", "k", "v", "gc", "gf", "do")
    return {n: (getattr(inputs, n).cuda() if getattr(inputs, n) is not None else None)
            for n in names}


def errors(gpu, ref):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    max_abs = float(np.max(np.abs(g - r))) if g.size else 0.0
    denom = float(np.linalg.norm(r))
    rel = float(np.linalg.norm(g - r) / denom) if denom > 0 else float(np.linalg.norm(g - r))
    return max_abs, rel


def assert_close(name, gpu, ref, atol=ATOL, rtol_l2=RTOL_L2):
    max_abs, rel = errors(gpu, ref)
    assert np.all(np.isfinite(np.asarray(gpu, dtype=np.float64))), f"{name}: non-finite values"
    assert max_abs <= atol and rel <= rtol_l2, \
        f"{name}: max-abs {max_abs:.3e} (bound {atol}), rel-L2 {rel:.3e} (bound {rtol_l2})"
    return max_abs, rel


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()
