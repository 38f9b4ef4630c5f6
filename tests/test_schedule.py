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
        # schedule: largest first; full rounds of `grid` positions alternate direction
        order = sorted(range(len(steps)), key=lambda i: (-steps[i], i))
        rounds = [order[r:r + grid] for r in range(0, len(order), grid)]
        seq = []
        for r, chunk in enumerate(rounds):
            seq += chunk[::-1] if (r % 2 and len(chunk) == grid) else chunk
        work = [sum(steps[seq[k]] for k in range(c, len(seq), grid)) for c in range(grid)]
        res[name] = (steps, work)
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
            assert schedule.cta_work(steps[name], sms).tolist() == ref[name][1]
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


def test_snake_schedule_balances_sorted_items():
    # 8 items on 4 CTAs: sorted 8,7,6,5 | 4,3,2,1 -> CTA totals 9,9,9,9
    steps = np.array([1, 8, 2, 7, 3, 6, 4, 5])
    assert schedule.cta_work(steps, 4).tolist() == [9, 9, 9, 9]
    order = schedule.schedule_order(steps, 4)
    assert sorted(order.tolist()) == list(range(8))
    assert steps[order].tolist() == [8, 7, 6, 5, 1, 2, 3, 4]
    # plain item order: CTA c takes items c and c + 4
    assert schedule.cta_work(steps, 4, scheduled=False).tolist() == [4, 14, 6, 12]


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
    # 8 items, 2 SMs: the schedule deals rounds of 2 positions by the two-tile cost,
    # the kernel's 4 CTAs take positions c, c + 4
    steps = np.array([1, 8, 2, 7, 3, 6, 4, 5])
    order = schedule.schedule_order(steps, 2)
    seq = steps[order]
    want = [int(seq[c::4].sum()) for c in range(4)]
    assert schedule.cta_work(steps, 2, grid=4).tolist() == want


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
