"""vsa_fine_fwd_noalloc: the fine stage for callers that cannot allocate.

A caller with no device allocator of its own (a plugin handed only its input
and output buffers by a host engine that owns all device memory) cannot supply
the scratch buffer vsa_fine_fwd takes.  vsa_fine_fwd_noalloc keeps that scratch
in a fixed array inside the library.  These tests call it through the C ABI and
check it against vsa_fine_fwd on the same inputs, on two calls in a row (the
array keeps the previous call's contents; the results must be bitwise equal:
same kernel, same inputs, no atomics), and that a configuration needing
more scratch than the array holds is refused before anything runs.

This file is collected last on purpose: the array stays resident on the GPU
for the rest of the process.
"""
import ctypes

import pytest
import torch

from trainable_block_sparse_gb300 import build, synth, vsa

_ARGS = [ctypes.POINTER(vsa.Config)] + [ctypes.c_void_p] * 13


def _lib():
    build.build()
    L = vsa.lib()
    fn = L.vsa_fine_fwd_noalloc
    fn.argtypes = _ARGS
    fn.restype = ctypes.c_int
    return L


def test_noalloc_refuses_configs_beyond_its_scratch():
    L = _lib()
    # 720p layer with 256-entry lists: 22,000 query pairs x (20 + 2048) bytes > 8 MiB
    cfg = vsa.make_config(1, 40, 20, 44, 80, 128, topk=256)
    assert L.vsa_validate(ctypes.byref(cfg)) == vsa.OK
    st = L.vsa_fine_fwd_noalloc(ctypes.byref(cfg), *([None] * 13))
    assert st == vsa.ERR_SHAPE


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["pretrain", "wan13b"])
def test_noalloc_matches_fine_fwd_on_two_calls(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = _lib()
    wl = synth.WORKLOADS[name]
    inp = synth.Inputs(wl, with_grad=False)
    cfg = vsa.config_for(wl)
    t = {n: getattr(inp, n).cuda() for n in ("q", "k", "v", "gc", "gf")}
    ws = torch.empty(vsa.workspace_bytes(cfg, False), dtype=torch.uint8, device="cuda")
    L.vsa_reset_device_status(vsa._ptr(ws), vsa._stream())
    q16, k16, v16 = (vsa.stage(cfg, t[n], ws) for n in ("q", "k", "v"))
    _, _, _, oc, _, idx, cnt = vsa.coarse_select(cfg, t["q"], t["k"], t["v"], ws)
    o_ref, of_ref, lse_ref = vsa.fine_fwd(cfg, q16, k16, v16, idx, cnt, t["gc"], t["gf"], oc, ws)
    torch.cuda.synchronize()
    assert L.vsa_check_device_status(vsa._ptr(ws), vsa._stream()) == vsa.OK

    P = vsa._ptr
    for call in range(2):
        o = torch.full_like(o_ref, float("nan"))
        of = torch.full_like(of_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        st = L.vsa_fine_fwd_noalloc(ctypes.byref(cfg), P(q16), P(k16), P(v16), P(idx), P(cnt),
                                    P(t["gc"]), P(t["gf"]), P(oc), P(o), P(of), P(lse),
                                    P(status), vsa._stream())
        assert st == vsa.OK, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert status.item() == 0, f"call {call}: device status bits {status.item()}"
        # the same kernel on the same inputs, each work item writing only its
        # own rows without atomics: bitwise equal, in any item order
        assert torch.equal(o, o_ref), f"O differs on call {call}"
        assert torch.equal(of, of_ref), f"O_f differs on call {call}"
        assert torch.equal(lse, lse_ref), f"lse_f differs on call {call}"
