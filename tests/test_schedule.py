"""Host-side work-distribution report of the persistent fine kernels, checked
against a plain set-based recomputation on small random selections."""
import math
import random

import numpy as np

from trainable_block_sparse_gb300 import schedule


def _random_lists(rng, bh, nc, cap):
    idx = np.full((bh, nc, cap), -1, dtype=np.int32)
    cnt = np.zeros((bh, nc), dtype=np.int32)
    for b in range(bh):
        for i in range(nc):
            c = rng.randint(1, cap)
            sel = sorted(rng.sample(range(nc), c))
            idx[b, i, :c] = sel
            cnt[b, i] = c
    return idx, cnt


def _hand_out(seq, grid):
    """Positions in order, each to the CTA with the least work so far (lowest
    index on ties), by a linear scan."""
    work = [0] * grid
    for w in seq:
        c = min(range(grid), key=lambda k: (work[k], k))
        work[c] += w
    return work


def _brute(idx, cnt, sms):
    bh, nc, _ = idx.shape
    lists = [[set(idx[b, i, : cnt[b, i]].tolist()) for i in range(nc)] for b in range(bh)]
    tlists = [[{i for i in range(nc) if j in lists[b][i]} for j in range(nc)] for b in range(bh)]
    res = {}
    for name, L in (("fine_fwd", lists), ("fine_bwd_dkdv", tlists)):
        steps = []
        for b in range(bh):
            for p in range((nc + 1) // 2):
                u = set(L[b][2 * p])
                if 2 * p + 1 < nc:
                    u |= L[b][2 * p + 1]
                steps.append(math.ceil(len(u) / 2))
        grid = min(len(steps), sms)
        # schedule: largest first (item order on ties), handed out to free CTAs
        order = sorted(range(len(steps)), key=lambda i: (-steps[i], i))
        res[name] = (steps, _hand_out([steps[i] for i in order], grid))
    return res


def test_item_steps_and_cta_work_match_set_recomputation():
    rng = random.Random(7)
    for bh, nc, cap, sms in ((1, 8, 3, 3), (3, 9, 5, 4), (2, 17, 6, 152)):
        idx, cnt = _random_lists(rng, bh, nc, cap)
        sel = schedule.selection_matrix(idx, cnt)
        steps = schedule.item_steps(sel)
        ref = _brute(idx, cnt, sms)
        for name in ("fine_fwd", "fine_bwd_dkdv"):
            assert steps[name].tolist() == ref[name][0]
            grid = min(steps[name].size, sms)
            order = schedule.schedule_order(steps[name])
            assert schedule.cta_work(steps[name], grid, order).tolist() == ref[name][1]
        assert steps["fine_bwd_dq"].tolist() == ref["fine_fwd"][0]


def test_load_balance_report():
    # 1 head, 4 cubes; cube i selects {i} except cube 0 selects everything
    idx = np.array([[[0, 1, 2, 3], [1, -1, -1, -1], [2, -1, -1, -1], [3, -1, -1, -1]]],
                   dtype=np.int32)
    cnt = np.array([[4, 1, 1, 1]], dtype=np.int32)
    r = schedule.load_balance(idx, cnt, sms=2)
    # query pairs (0,1): union 4 -> 2 steps; (2,3): union 2 -> 1 step; one per CTA
    assert r["fine_fwd"]["cta_steps_max"] == 2
    assert r["fine_fwd"]["max_over_mean"] == 2 / 1.5
    # transposed: key cubes 0..3 are selected by {0},{0,1},{0,2},{0,3}
    # pairs (0,1): union {0,1} -> 1 step; (2,3): {0,2,3} -> 2 steps
    assert r["fine_bwd_dkdv"]["steps_total"] == 3
    assert r["count_histogram"] == {1: 3, 4: 1}


def test_counter_hands_positions_to_the_first_free_cta():
    # 8 items on 4 CTAs, largest first: 8,7,6,5 then 4 -> the CTA at 5, 3 -> at 6,
    # 2 -> at 7, 1 -> at 8: totals 9,9,9,9
    steps = np.array([1, 8, 2, 7, 3, 6, 4, 5])
    order = schedule.schedule_order(steps)
    assert steps[order].tolist() == [8, 7, 6, 5, 4, 3, 2, 1]
    assert schedule.cta_work(steps, 4, order).tolist() == [9, 9, 9, 9]
    # item order: 1,8,2,7 start; 3 -> CTA 0 (at 1), 6 -> CTA 2 (at 2), 4 -> CTA 0
    # (at 4), 5 -> CTA 3 (at 7)
    assert schedule.cta_work(steps, 4).tolist() == [8, 8, 8, 12]
    # the static assignment: CTA c takes positions c and c + 4
    assert schedule.cta_work_static(steps, 4).tolist() == [4, 14, 6, 12]
    assert schedule.cta_work_static(steps, 4, order).tolist() == [12, 10, 8, 6]
    # list scheduling: no CTA ends later than the mean plus the largest item
    rng = np.random.default_rng(3)
    for _ in range(20):
        st = rng.integers(1, 40, size=int(rng.integers(1, 400)))
        for grid in (1, 7, 152):
            w = schedule.cta_work(st, grid)
            g = min(grid, st.size)
            assert w.sum() == st.sum() and w.size == g
            assert w.max() <= st.sum() / g + st.max()


def test_head_dim_64_forward_runs_two_ctas_per_sm_with_one_key_tile_per_step():
    # the same 4-cube selection as above; the head_dim-64 forward takes one key
    # tile per step (pair (0,1): 4 steps, pair (2,3): 2) on up to 2 x sms CTAs,
    # in the schedule built from the two-tile costs
    idx = np.array([[[0, 1, 2, 3], [1, -1, -1, -1], [2, -1, -1, -1], [3, -1, -1, -1]]],
                   dtype=np.int32)
    cnt = np.array([[4, 1, 1, 1]], dtype=np.int32)
    r = schedule.load_balance(idx, cnt, sms=1, head_dim=64)
    assert r["fine_fwd"]["ctas"] == 2 and r["fine_fwd"]["steps_total"] == 6
    assert r["fine_fwd"]["cta_steps_max"] == 4
    assert r["fine_bwd_dq"]["ctas"] == 1 and r["fine_bwd_dq"]["steps_total"] == 3
    assert schedule.kernel_grid("fine_fwd", 1000, 152, 64) == 304
    assert schedule.kernel_grid("fine_fwd", 1000, 152, 128) == 152
    # 8 items, 2 SMs: the kernel's 4 CTAs take positions from the counter
    steps = np.array([1, 8, 2, 7, 3, 6, 4, 5])
    order = schedule.schedule_order(steps)
    grid = schedule.kernel_grid("fine_fwd", steps.size, 2, 64)
    assert grid == 4
    assert schedule.cta_work(steps, grid, order).tolist() == _hand_out(steps[order].tolist(), 4)


def test_two_ctas_per_sm_report_the_pairs_of_ctas_that_share_an_sm():
    # CTAs s and s + sms share SM s
    assert schedule.sm_work(np.array([5, 1, 2, 7]), 2).tolist() == [7, 8]
    assert schedule.sm_work(np.array([5, 1, 2]), 2).tolist() == [7, 1]
    idx = np.array([[[0, 1, 2, 3], [1, -1, -1, -1], [2, -1, -1, -1], [3, -1, -1, -1]]],
                   dtype=np.int32)
    cnt = np.array([[4, 1, 1, 1]], dtype=np.int32)
    r = schedule.load_balance(idx, cnt, sms=1, head_dim=64)
    # both items on the one SM: its load is all 6 steps, the mean is 6
    assert r["fine_fwd"]["sm_max_over_mean"] == 1.0
