"""Work distribution of the persistent fine-stage kernels: a host-side report.

The fine forward kernel and both fine backward passes launch one CTA per SM
(grid = min(items, SMs); the head_dim-64 forward two per SM, grid =
min(items, 2 SMs)).  A CTA takes the next schedule position from a counter
shared by the launch whenever it has room for another item, so positions are
handed out in schedule order to whichever CTA frees up first.  The schedule
is the item order, or (when the K and V of all slices fit in twice the L2)
the items sorted by step count, largest first: the longest-processing-time
rule.  An item is a pair of neighbouring cubes (2p, 2p + 1) of one (batch,
head), item index = bh * ceil(Nc / 2) + p:

  * forward and dQ pass: two query cubes walking the union of their index
    lists;
  * key-major pass: two key cubes walking the union of their transposed
    lists (the query cubes that selected them).

Each step of an item covers two key (or query) tiles, so an item costs
ceil(|union| / 2) steps (the schedule's cost); a step of the head_dim-64
forward covers one key tile, so there an item takes |union| steps.  This
module recomputes those costs from the index lists that the coarse stage
emitted and reports how evenly the assignment spreads them over the CTAs,
modelling a step as the unit of time ("VSA: Faster Video Diffusion with
Trainable Sparse Attention", §2: the fine stage attends only within the
selected blocks, so per-cube work varies with the selection, most of all
with the coarse-mass rule of the dynamic variant).  For comparison it also
gives the static assignment (CTA c taking positions c, c + grid, ...).
"""
from __future__ import annotations

import heapq

import numpy as np


def selection_matrix(idx: np.ndarray, cnt: np.ndarray) -> np.ndarray:
    """Boolean [BH, Nc, Nc]: row i has column j set when key cube j is in the
    first cnt[i] entries of query cube i's list."""
    idx = np.asarray(idx).reshape(-1, idx.shape[-2], idx.shape[-1])
    cnt = np.asarray(cnt).reshape(idx.shape[0], idx.shape[1])
    bh, nc, cap = idx.shape
    live = np.arange(cap)[None, None, :] < cnt[:, :, None]
    sel = np.zeros((bh, nc, nc), dtype=bool)
    b, i, e = np.nonzero(live)
    sel[b, i, idx[b, i, e]] = True
    return sel


def pair_union_sizes(sel: np.ndarray) -> np.ndarray:
    """|list(2p) U list(2p+1)| per pair, [BH, ceil(Nc/2)]; a lone last cube
    pairs with nothing."""
    bh, nc, _ = sel.shape
    even = sel[:, 0::2]
    odd = np.zeros_like(even)
    odd[:, : nc // 2] = sel[:, 1::2]
    return (even | odd).sum(-1)


def item_steps(sel: np.ndarray, head_dim: int = 128) -> dict[str, np.ndarray]:
    """Steps per work item, flattened in item order, for each fine kernel."""
    union = pair_union_sizes(sel)
    fwd = (union + 1) // 2
    key = (pair_union_sizes(np.swapaxes(sel, 1, 2)) + 1) // 2
    return {"fine_fwd": (union if head_dim == 64 else fwd).ravel(), "fine_bwd_dq": fwd.ravel(),
            "fine_bwd_dkdv": key.ravel()}


def kernel_grid(name: str, items: int, sms: int, head_dim: int) -> int:
    """CTAs a fine kernel launches for `items` work items."""
    per_sm = 2 if (name == "fine_fwd" and head_dim == 64) else 1
    return min(items, per_sm * sms)


def schedule_order(cost: np.ndarray) -> np.ndarray:
    """Item index at each schedule position when the items are cost-sorted:
    largest first, ties in item order."""
    return np.argsort(-np.asarray(cost), kind="stable")


def cta_work(steps: np.ndarray, grid: int, order: np.ndarray | None = None) -> np.ndarray:
    """Total steps of each of `grid` CTAs when positions are handed out, in
    schedule order (`order`, default item order), to the CTA with the least
    work so far (the lowest index on ties): the counter the kernels share."""
    steps = np.asarray(steps)
    seq = steps if order is None else steps[np.asarray(order)]
    grid = min(int(grid), seq.size)
    if grid <= 0:
        return np.zeros(0, dtype=np.int64)
    heap = [(0, c) for c in range(grid)]
    work = np.zeros(grid, dtype=np.int64)
    for w in seq.tolist():
        t, c = heapq.heappop(heap)
        work[c] = t + w
        heapq.heappush(heap, (t + w, c))
    return work


def cta_work_static(steps: np.ndarray, grid: int, order: np.ndarray | None = None) -> np.ndarray:
    """Total steps of each CTA under the static assignment: CTA c takes
    positions c, c + grid, ... of the schedule."""
    steps = np.asarray(steps)
    seq = steps if order is None else steps[np.asarray(order)]
    n = seq.size
    grid = min(int(grid), n)
    if grid <= 0:
        return np.zeros(0, dtype=np.int64)
    padded = np.zeros(-(-n // grid) * grid, dtype=np.int64)
    padded[:n] = seq
    return padded.reshape(-1, grid).sum(0)


def sm_work(cta: np.ndarray, sms: int) -> np.ndarray:
    """Per-SM totals of a kernel whose CTAs s, s + sms, s + 2 sms, ... share
    SM s."""
    cta = np.asarray(cta)
    n = -(-cta.size // sms) * sms
    padded = np.zeros(n, dtype=cta.dtype)
    padded[:cta.size] = cta
    return padded.reshape(-1, sms).sum(0)


def uses_cost_order(batch_heads: int, tokens: int, head_dim: int) -> bool:
    """The library sorts the items by cost only when the fp16 K and V of all
    slices fit in 256 MB (twice the L2); otherwise it keeps item order, whose
    concurrently running items share K/V tiles in L2."""
    return 4.0 * batch_heads * tokens * head_dim <= 256.0 * 1024 * 1024


def load_balance(idx: np.ndarray, cnt: np.ndarray, sms: int, ordered: bool = True,
                 head_dim: int = 128) -> dict:
    """max/mean per-CTA steps of each fine kernel (positions handed out from
    the shared counter in the cost-sorted schedule when `ordered`, else in
    item order), the same for the static assignment, the step count of the
    biggest item, and the histogram of per-cube list lengths."""
    sel = selection_matrix(idx, cnt)
    out = {"schedule": "cost-sorted, largest first" if ordered else "item order",
           "assignment": "shared counter: next position to the first free CTA"}
    all_steps = item_steps(sel, head_dim)
    cost = item_steps(sel)["fine_fwd"]  # the schedule's cost: two key tiles per step
    for name, steps in all_steps.items():
        grid = kernel_grid(name, steps.size, sms, head_dim)
        c = cost if name != "fine_bwd_dkdv" else steps
        order = schedule_order(c) if ordered else None
        w = cta_work(steps, grid, order)
        w_static = cta_work_static(steps, grid, order)
        mean = float(w.mean()) if w.size else 0.0
        out[name] = {"items": int(steps.size), "ctas": int(w.size),
                     "steps_total": int(steps.sum()),
                     "cta_steps_max": int(w.max()) if w.size else 0,
                     "cta_steps_mean": mean,
                     "max_over_mean": float(w.max() / mean) if mean > 0 else 1.0,
                     "max_over_mean_static": float(w_static.max() / mean) if mean > 0 else 1.0,
                     "item_steps_max": int(steps.max()) if steps.size else 0}
        if grid > sms:
            # two CTAs per SM: CTAs s and s + sms share SM s (the block
            # scheduler places a grid round-robin), so the SMs' loads are the pairs
            sm = sm_work(w, sms)
            out[name]["sm_max_over_mean"] = float(sm.max() / sm.mean()) if sm.size else 1.0
    counts = np.bincount(np.asarray(cnt).ravel(), minlength=1)
    out["count_histogram"] = {int(c): int(n) for c, n in enumerate(counts) if n}
    return out
