"""HostPipeline: a layer's forward + backward from pinned host tensors, cut
into (batch entry, head group) units whose copies overlap the kernels, gives
exactly the results of one device-resident call (every slice is computed by
the same kernels either way)."""
import pytest
import torch

from trainable_block_sparse_gb300 import build, synth, vsa
from trainable_block_sparse_gb300.host_pipeline import IN_NAMES, OUT_NAMES, HostPipeline


@pytest.mark.gpu
@pytest.mark.parametrize("name,hpu", [("pretrain", 5), ("tiny", 1)])
def test_host_pipeline_matches_device_call(name, hpu):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    wl = synth.WORKLOADS[name]
    inp = synth.Inputs(wl, with_grad=True)
    cfg = vsa.config_for(wl)
    dev = torch.device("cuda")
    t = {n: getattr(inp, n).to(dev) for n in IN_NAMES}
    bufs = vsa.Buffers(cfg, dev, with_backward=True)
    o = vsa.forward(cfg, t["q"], t["k"], t["v"], t["gc"], t["gf"], bufs, True)
    grads = vsa.backward(cfg, t["gc"], t["gf"], t["do"], bufs)
    assert bufs.device_status() == vsa.OK
    ref = dict(zip(OUT_NAMES, (o,) + tuple(grads)))

    host_in = {n: getattr(inp, n).pin_memory() for n in IN_NAMES}
    host_out = {n: torch.full(ref[n].shape, float("nan"), dtype=ref[n].dtype).pin_memory()
                for n in OUT_NAMES}
    pipe = HostPipeline(cfg, dev, heads_per_unit=hpu)
    for _ in range(2):  # the second pass reuses every buffer set
        pipe.step(host_in, host_out)
    assert pipe.check_status() == vsa.OK
    for n in OUT_NAMES:
        assert torch.equal(host_out[n], ref[n].cpu()), n
