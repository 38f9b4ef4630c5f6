"""Device-side failure reporting without a GPU fault.

Every pipelined kernel waits on mbarriers with a time limit; on expiry it
records a time-out in the status word of the workspace and returns instead of
spinning forever.  vsa_probe_wait_timeout runs that same bounded wait on a
barrier nothing completes, so the expiry path can be exercised for real: the
status word must report VSA_ERR_TIMEOUT, the wait must have lasted about the
limit, and the context must stay usable (a reset clears the word and a full
forward pass afterwards still matches the oracle)."""
import time

import pytest
import torch

from tests.test_gpu_forward import check_forward, gapped
from trainable_block_sparse_gb300 import build, vsa


@pytest.mark.gpu
def test_expired_wait_is_reported_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    L = vsa.lib()
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    s = vsa._stream()
    assert L.vsa_reset_device_status(vsa._ptr(ws), s) == vsa.OK
    assert L.vsa_check_device_status(vsa._ptr(ws), s) == vsa.OK
    limit_us = 200_000
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert L.vsa_probe_wait_timeout(vsa._ptr(ws), limit_us, s) == vsa.OK
    assert L.vsa_check_device_status(vsa._ptr(ws), s) == vsa.ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert elapsed >= 0.9 * limit_us * 1e-6, elapsed
    assert elapsed < 30.0, elapsed
    # the context is intact: clear the word, then a whole forward pass still works
    assert L.vsa_reset_device_status(vsa._ptr(ws), s) == vsa.OK
    assert L.vsa_check_device_status(vsa._ptr(ws), s) == vsa.OK
    check_forward(gapped("tiny"))


@pytest.mark.gpu
def test_device_range_flag_surfaces_through_autograd():
    """A Q value above fp16's range is flagged by the staging kernel; the
    autograd entry point reads the status word and raises VSAError."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    inp = gapped("tiny")
    wl = inp.wl
    t = {n: getattr(inp, n).cuda() for n in ("q", "k", "v", "gc", "gf")}
    q = t["q"].clone()
    q[0, 1, 77, 5] = 1.0e5
    with pytest.raises(vsa.VSAError) as e:
        vsa.video_sparse_attention(q.requires_grad_(True), t["k"], t["v"], t["gc"], t["gf"],
                                   (wl.T, wl.H, wl.W), topk=wl.topk)
    assert e.value.status == vsa.ERR_DEVICE_CHECK
    # a clean call afterwards still works (the flag lives in that call's buffers)
    o = vsa.video_sparse_attention(t["q"], t["k"], t["v"], t["gc"], t["gf"],
                                   (wl.T, wl.H, wl.W), topk=wl.topk)
    assert torch.isfinite(o.float()).all()
