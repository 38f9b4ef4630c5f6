"""The oracle's process pool moves inputs to oracle Heads and results back: a
whole layer through it (split into many small tasks over two processes) equals
the oracle called directly, bit for bit."""
import numpy as np
import pytest

from oracle import vsa_oracle as O
from trainable_block_sparse_gb300 import synth


@pytest.fixture(scope="module")
def pool():
    from oracle.pool import OraclePool
    p = OraclePool(processes=2)
    yield p
    p.close()


@pytest.mark.parametrize("name", ["tiny", "tiny_mass"])
def test_pool_layer_equals_direct_oracle(pool, name):
    if name == "tiny":
        wl = synth.WORKLOADS["tiny"]
    else:
        wl = synth.Workload("tiny_mass", 1, 2, 64, 8, 8, 8, "mass", mass=0.5, kmin=2, kmax=6,
                            seed=5)
    inp = synth.Inputs(wl, with_grad=True)
    slices = [(0, h) for h in range(wl.heads)]
    got = pool.layer(inp, slices, "pool_test", backward=True, chunk=3)
    for b, h in slices:
        r = got[(b, h)]
        hd = O.head_of(inp, b, h)
        assert r["cubes"] == list(range(wl.cubes))
        np.testing.assert_array_equal(r["idx"], hd.idx)
        np.testing.assert_array_equal(r["cnt"], hd.cnt)
        np.testing.assert_array_equal(r["oc"], hd.coarse["out"])
        for i, c in enumerate(range(wl.cubes)):
            _, of, lse = hd.rows(c)
            np.testing.assert_array_equal(r["o_f"][i], of)
            np.testing.assert_array_equal(r["lse_f"][i], lse)
            np.testing.assert_array_equal(r["o"][i], hd.output_tiled(c))
            rq, rgc, rgf = hd.grad_query_cube(c)
            np.testing.assert_array_equal(r["dq"][i], rq)
            np.testing.assert_array_equal(r["dgc"][i], rgc)
            np.testing.assert_array_equal(r["dgf"][i], rgf)
        for j in range(wl.cubes):
            rk, rv = hd.grad_key_cube(j)
            # the pool sums per-task partials: same terms, another summation order
            np.testing.assert_allclose(r["dk"][j * 64:(j + 1) * 64], rk, rtol=0, atol=1e-12)
            np.testing.assert_allclose(r["dv"][j * 64:(j + 1) * 64], rv, rtol=0, atol=1e-12)
