"""Backward parity at the magnitudes training produces, not only at N(0,1).

* Small upstream gradients: bf16 training without loss scaling hands the
  attention backward dO of 1e-5 to 1e-8.  The fp16 operand dO (.) G_f of the
  fine backward is staged times a power of two per (batch, head) slice, so dO
  scaled by 2^-16 and 2^-26 must give the same gradients scaled by the same
  factor.  The oracle is linear in dO and a power-of-two factor is exact in
  fp64, so the GPU's gradients times 2^16 (2^26) are compared with the
  oracle's gradients for the unscaled dO, at the usual bounds: that is the
  comparison with the oracle at dO * 2^-k under bounds scaled by 2^-k.
* Large logits: Q and K times 8 (logits times 64, softmax rows close to one
  hot); the oracle is recomputed for these inputs.  The gradients grow with
  them (dQ = scale * dS K and dK = scale * dS^T Q carry the factor 8 of K and
  Q; sharper rows of P concentrate dV on fewer keys), and fp16 rounding errors
  grow in proportion.  So each tensor's max-abs bound, 2e-2 at the N(0,1)
  inputs the bound was set for, is scaled by how much that tensor's largest
  oracle value grows over the same slice at those inputs (at least 1);
  rel-L2 1e-2 stays as it is.

Layers: the tiny one (every element), two whole slices of the pretraining
layer and one whole slice of the 720p layer.
"""
import dataclasses

import numpy as np
import pytest
import torch

from tests.helpers import ATOL, assert_close
from tests.test_gpu_forward import gapped
from tests.test_gpu_full_parity import P720_SLICE, all_slices, compare_slice, gpu_layer
from trainable_block_sparse_gb300 import build

pytestmark = pytest.mark.gpu

CASES = {"tiny": None, "pretrain": [(0, 0), (1, 11)], "p720": [P720_SLICE]}
GRADS = ("dq", "dk", "dv", "dgc", "dgf")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@dataclasses.dataclass
class Scaled:
    """The tensors of a synth.Inputs with some of them multiplied by a power of two."""
    wl: object
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    gc: torch.Tensor
    gf: torch.Tensor
    do: torch.Tensor


def scaled(inp, **factors):
    t = {n: getattr(inp, n) for n in ("q", "k", "v", "gc", "gf", "do")}
    for n, f in factors.items():
        y = (t[n].float() * f).to(torch.bfloat16)
        assert torch.equal(y.float(), t[n].float() * f), "a power-of-two factor must be exact"
        t[n] = y
    return Scaled(inp.wl, **t)


def _slices(name, wl):
    return CASES[name] if CASES[name] is not None else all_slices(wl)


def _oracle(pool, name, inp, slices):
    # the same oracle results the full-coverage tests compare against
    if name == "pretrain":
        return pool.layer_memo(("full", "pretrain"), inp, all_slices(inp.wl), name, backward=True)
    if name == "p720":
        return pool.layer_memo(("full", "p720", P720_SLICE), inp, slices, name, backward=True)
    return pool.layer_memo(("full", name), inp, slices, name, backward=True)


@pytest.mark.parametrize("name", list(CASES))
def test_small_upstream_gradients(name, oracle_pool):
    inp = gapped(name)
    slices = _slices(name, inp.wl)
    ref = _oracle(oracle_pool, name, inp, slices)
    for k in (16, 26):
        got = gpu_layer(scaled(inp, do=2.0 ** -k), slices, backward=True)
        for key in slices:
            for n in GRADS:
                g = got[key][n] * 2.0 ** k
                r = ref[key][n].reshape(g.shape)
                assert_close(f"{n} {key} dO*2^-{k} (times 2^{k})", g, r)


@pytest.mark.parametrize("name", list(CASES))
def test_large_logits(name, oracle_pool):
    base_inp = gapped(name)
    inp = scaled(base_inp, q=8.0, k=8.0)
    slices = _slices(name, inp.wl)
    base = _oracle(oracle_pool, name, base_inp, slices)
    got = gpu_layer(inp, slices, backward=True)
    ref = oracle_pool.layer(inp, slices, f"{name}_qk8", backward=True)
    for key in slices:
        growth = {n: max(1.0, float(np.max(np.abs(ref[key][n])) / np.max(np.abs(base[key][n]))))
                  for n in ("o", "o_f") + GRADS}
        compare_slice(inp.wl, key, got[key], ref[key], backward=True,
                      atol={n: ATOL * g for n, g in growth.items()})
