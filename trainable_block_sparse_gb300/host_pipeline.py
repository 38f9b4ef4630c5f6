"""One VSA layer (forward + backward) on host-resident tensors, with the
host<->device copies overlapped with the kernels.

Every (batch, head) slice of the layer is independent: the coarse and fine
stages never mix heads ("VSA: Faster Video Diffusion with Trainable Sparse
Attention", §2: each head selects its own blocks).  `HostPipeline` therefore
cuts the layer into units of one batch entry and a group of heads, and runs
them through CUDA streams for copy-in (pinned host -> device), compute
(vsa_forward + vsa_backward through the C ABI) and copy-out (device -> pinned
host).  Two sets of device buffers alternate between units, so while unit i
computes, unit i+1's inputs arrive and unit i-1's outputs leave.  Nothing
here computes: it only schedules copies and library calls.  (Spreading each
direction's copies over two streams measured no faster on the 720p layer:
the host link is the limit there.)
"""
from __future__ import annotations

import torch

from . import vsa

IN_NAMES = ("q", "k", "v", "gc", "gf", "do")
OUT_NAMES = ("o", "dq", "dk", "dv", "dgc", "dgf")


class HostPipeline:
    """Forward + backward of one layer from pinned host tensors to pinned host
    tensors.

    cfg: the layer's vsa.Config (batch, heads, video shape, selection).
    heads_per_unit: heads per pipeline unit (the last unit of a batch entry
    may hold fewer).  Inputs q, k, v, gc, gf, do: bf16 [B, heads, N, D];
    outputs: o bf16, dq, dk, dv, dgc, dgf of cfg's gradient dtype (fp32 or bf16),
    same shape; all pinned.
    """

    def __init__(self, cfg: vsa.Config, device, heads_per_unit: int, n_sets: int = 2,
                 copy_streams: int = 1):
        self.cfg = cfg
        self.device = torch.device(device)
        self.hpu = max(1, min(heads_per_unit, cfg.heads))
        self.n_sets = n_sets
        self.streams = {k: torch.cuda.Stream(self.device) for k in ("in", "comp", "out")}
        # each direction's tensors are spread over several streams, so more
        # than one copy is in flight per direction
        self.copy_in = [self.streams["in"]] + [torch.cuda.Stream(self.device)
                                               for _ in range(copy_streams - 1)]
        self.copy_out = [self.streams["out"]] + [torch.cuda.Stream(self.device)
                                                 for _ in range(copy_streams - 1)]
        N = cfg.T * cfg.H * cfg.W
        D = cfg.head_dim
        self.sets = []
        for _ in range(n_sets):
            s = {"cfg": {}, "bufs": {}}
            shape = (1, self.hpu, N, D)
            s["in"] = {n: torch.empty(shape, dtype=torch.bfloat16, device=self.device)
                       for n in IN_NAMES}
            s["out"] = {"o": torch.empty(shape, dtype=torch.bfloat16, device=self.device)}
            gdt = vsa.grad_torch_dtype(cfg)
            for n in OUT_NAMES[1:]:
                s["out"][n] = torch.empty(shape, dtype=gdt, device=self.device)
            s["events"] = {"comp": torch.cuda.Event(),
                           "in": [torch.cuda.Event() for _ in range(copy_streams)],
                           "out": [torch.cuda.Event() for _ in range(copy_streams)]}
            s["used"] = False
            self.sets.append(s)

    def _sub(self, s, heads: int):
        """Config and buffers of a unit of `heads` heads (created once per size)."""
        if heads not in s["cfg"]:
            c = self.cfg
            sub = vsa.Config(1, heads, c.T, c.H, c.W, c.head_dim, c.select_mode, c.topk, c.mass,
                             c.kmin, c.kmax, c.scale, c.layout, c.grad_dtype)
            s["cfg"][heads] = sub
            with torch.cuda.stream(self.streams["comp"]):
                s["bufs"][heads] = vsa.Buffers(sub, self.device, with_backward=True)
        return s["cfg"][heads], s["bufs"][heads]

    def units(self):
        for b in range(self.cfg.batch):
            for h0 in range(0, self.cfg.heads, self.hpu):
                yield b, h0, min(self.hpu, self.cfg.heads - h0)

    def step(self, host_in: dict, host_out: dict) -> None:
        """Enqueue the whole layer; returns before the copies finish (call
        torch.cuda.synchronize() or check_status() to wait)."""
        st = self.streams
        for i, (b, h0, hn) in enumerate(self.units()):
            s = self.sets[i % self.n_sets]
            ev = s["events"]
            sub, bufs = self._sub(s, hn)
            dev_in = {n: t[:, :hn] for n, t in s["in"].items()}
            dev_out = {n: t[:, :hn] for n, t in s["out"].items()}
            ci, co = self.copy_in, self.copy_out
            for j, cs in enumerate(ci):
                with torch.cuda.stream(cs):
                    if s["used"]:
                        cs.wait_event(ev["comp"])  # the set's previous unit has read its inputs
                    for n in IN_NAMES[j::len(ci)]:
                        dev_in[n].copy_(host_in[n][b:b + 1, h0:h0 + hn], non_blocking=True)
                    ev["in"][j].record(cs)
            with torch.cuda.stream(st["comp"]):
                for e in ev["in"]:
                    st["comp"].wait_event(e)
                if s["used"]:
                    for e in ev["out"]:
                        st["comp"].wait_event(e)  # its previous outputs have left
                vsa.forward(sub, dev_in["q"], dev_in["k"], dev_in["v"], dev_in["gc"],
                            dev_in["gf"], bufs, True, out=dev_out["o"])
                vsa.backward(sub, dev_in["gc"], dev_in["gf"], dev_in["do"], bufs,
                             tuple(dev_out[n] for n in OUT_NAMES[1:]))
                ev["comp"].record(st["comp"])
            for j, cs in enumerate(co):
                with torch.cuda.stream(cs):
                    cs.wait_event(ev["comp"])
                    for n in OUT_NAMES[j::len(co)]:
                        host_out[n][b:b + 1, h0:h0 + hn].copy_(dev_out[n], non_blocking=True)
                    ev["out"][j].record(cs)
            s["used"] = True

    def check_status(self) -> int:
        """Waits for all work; the first non-OK device status of any buffer set."""
        torch.cuda.synchronize(self.device)
        for s in self.sets:
            for bufs in s["bufs"].values():
                with torch.cuda.stream(self.streams["comp"]):
                    st = bufs.device_status()
                if st != vsa.OK:
                    return st
        return vsa.OK
