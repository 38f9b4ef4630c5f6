"""Thin Python binding of libvsa.so (include/vsa.h): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
passes device pointers, sizes and the current torch stream through ctypes,
and raises when the library is missing or a call fails.  There is no CPU path.

User entry point: `video_sparse_attention(q, k, v, gc, gf, video_shape, ...)`,
differentiable through `torch.autograd`.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libvsa.so")

OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_UNSUPPORTED, ERR_ALIGNMENT, ERR_CUDA, ERR_TIMEOUT, \
    ERR_DEVICE_CHECK = range(8)
SELECT_TOPK, SELECT_MASS = 0, 1
LAYOUT_RASTER, LAYOUT_CUBE = 0, 1
GRAD_FP32, GRAD_BF16 = 0, 1


class Config(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("T", ctypes.c_int32), ("H", ctypes.c_int32), ("W", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("select_mode", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("mass", ctypes.c_float),
                ("kmin", ctypes.c_int32), ("kmax", ctypes.c_int32),
                ("scale", ctypes.c_float), ("layout", ctypes.c_int32),
                ("grad_dtype", ctypes.c_int32)]


class SavedLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("q16", "k16", "v16", "qc", "kc", "vc", "oc", "lse_c", "idx", "cnt",
                 "o_f", "lse_f", "total")] + [("list_cap", ctypes.c_int32)]


_P = ctypes.c_void_p
_SIGS = {
    "vsa_validate": [ctypes.POINTER(Config)],
    "vsa_status_string": [ctypes.c_int],
    "vsa_saved_bytes": [ctypes.POINTER(Config), ctypes.POINTER(SavedLayout)],
    "vsa_saved_bytes_for": [ctypes.POINTER(Config), ctypes.c_int, ctypes.POINTER(SavedLayout)],
    "vsa_workspace_bytes": [ctypes.POINTER(Config), ctypes.c_int],
    "vsa_reset_device_status": [_P, _P],
    "vsa_check_device_status": [_P, _P],
    "vsa_permute": [ctypes.POINTER(Config), _P, _P, ctypes.c_int, _P],
    "vsa_stage": [ctypes.POINTER(Config)] + [_P] * 5,
    "vsa_coarse_select": [ctypes.POINTER(Config)] + [_P] * 12,
    "vsa_fine_fwd": [ctypes.POINTER(Config)] + [_P] * 13,
    "vsa_combine_bwd": [ctypes.POINTER(Config)] + [_P] * 13,
    "vsa_coarse_bwd": [ctypes.POINTER(Config)] + [_P] * 11,
    "vsa_fine_bwd": [ctypes.POINTER(Config)] + [_P] * 17,
    "vsa_forward": [ctypes.POINTER(Config)] + [_P] * 7 + [ctypes.c_int, _P, _P],
    "vsa_backward": [ctypes.POINTER(Config)] + [_P] * 11,
    "vsa_probe_wait_timeout": [_P, ctypes.c_uint32, _P],
    "vsa_fine_fwd_bf16": [ctypes.POINTER(Config)] + [_P] * 12,
    "vsa_stage_fp8": [ctypes.POINTER(Config)] + [_P] * 12,
    "vsa_fine_fwd_fp8": [ctypes.POINTER(Config)] + [_P] * 13,
    "vsa_forward_fp8": [ctypes.POINTER(Config)] + [_P] * 9,
}
_RESTYPES = {"vsa_status_string": ctypes.c_char_p, "vsa_saved_bytes": ctypes.c_size_t,
             "vsa_saved_bytes_for": ctypes.c_size_t,
             "vsa_workspace_bytes": ctypes.c_size_t}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libvsa.so not found at {LIB_PATH}; build it with "
                "`python -m trainable_block_sparse_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = _RESTYPES.get(name, ctypes.c_int)
        _lib = L
    return _lib


class VSAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().vsa_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")


def check(status: int, where: str) -> None:
    if status != OK:
        raise VSAError(status, where)


def make_config(batch, heads, T, H, W, head_dim, *, topk=32, select="topk", mass=0.9,
                kmin=8, kmax=64, scale=0.0, layout="raster", grad_dtype="fp32") -> Config:
    if grad_dtype not in ("fp32", "bf16"):
        raise ValueError(f"grad_dtype must be 'fp32' or 'bf16', got {grad_dtype!r}")
    return Config(batch, heads, T, H, W, head_dim,
                  SELECT_TOPK if select == "topk" else SELECT_MASS, topk, mass, kmin, kmax,
                  scale, LAYOUT_RASTER if layout == "raster" else LAYOUT_CUBE,
                  GRAD_FP32 if grad_dtype == "fp32" else GRAD_BF16)


def grad_torch_dtype(cfg: Config):
    """torch dtype of the gradients the library writes for cfg."""
    return torch.bfloat16 if cfg.grad_dtype == GRAD_BF16 else torch.float32


def config_for(wl, layout="raster", grad_dtype="fp32") -> Config:
    """Config of a synth.Workload."""
    return make_config(wl.batch, wl.heads, wl.T, wl.H, wl.W, wl.head_dim, topk=wl.topk,
                       select=wl.select, mass=wl.mass, kmin=wl.kmin, kmax=wl.kmax,
                       layout=layout, grad_dtype=grad_dtype)


def saved_layout(cfg: Config, with_backward: bool = True) -> SavedLayout:
    """The `saved` buffer's layout for training (every piece) or, with
    with_backward False, for an inference forward alone."""
    L = SavedLayout()
    n = lib().vsa_saved_bytes_for(ctypes.byref(cfg), int(with_backward), ctypes.byref(L))
    if n == 0:
        check(lib().vsa_validate(ctypes.byref(cfg)), "vsa_saved_bytes")
    return L


def workspace_bytes(cfg: Config, with_backward: bool) -> int:
    n = lib().vsa_workspace_bytes(ctypes.byref(cfg), int(with_backward))
    if n == 0:
        check(lib().vsa_validate(ctypes.byref(cfg)), "vsa_workspace_bytes")
    return n


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libvsa takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libvsa takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


class Buffers:
    """Caller-owned device buffers of one layer: the `saved` context and `ws` scratch.
    `inference_only` sizes `saved` for forward(with_backward=False) alone."""

    def __init__(self, cfg: Config, device, with_backward: bool, inference_only: bool = False):
        if with_backward and inference_only:
            raise ValueError("inference_only buffers cannot hold a backward's context")
        self.cfg = cfg
        self.layout = saved_layout(cfg, with_backward=not inference_only)
        self.saved = torch.empty(self.layout.total, dtype=torch.uint8, device=device)
        self.ws = torch.empty(workspace_bytes(cfg, with_backward), dtype=torch.uint8,
                              device=device)
        check(lib().vsa_reset_device_status(_ptr(self.ws), _stream()), "vsa_reset_device_status")

    def view(self, name: str, dtype, shape):
        off = getattr(self.layout, name)
        n = 1
        for s in shape:
            n *= s
        itemsize = torch.empty((), dtype=dtype).element_size()
        return self.saved[off: off + n * itemsize].view(dtype).view(*shape)

    def device_status(self) -> int:
        return lib().vsa_check_device_status(_ptr(self.ws), _stream())


# ------------------------------------------------------------------ entry points

def permute(cfg: Config, x: torch.Tensor, inverse: bool = False) -> torch.Tensor:
    out = torch.empty_like(x)
    check(lib().vsa_permute(ctypes.byref(cfg), _ptr(x), _ptr(out), int(inverse), _stream()),
          "vsa_permute")
    return out


def stage(cfg: Config, x, ws, want_pooled=False):
    """bf16 x (cfg.layout order) -> fp16 cube-order staged copy (and cube means)."""
    B, Hd, N, D = x.shape
    x16 = torch.empty(B, Hd, N, D, dtype=torch.float16, device=x.device)
    pooled = (torch.empty(B, Hd, N // 64, D, dtype=torch.float32, device=x.device)
              if want_pooled else None)
    check(lib().vsa_stage(ctypes.byref(cfg), _ptr(x), _ptr(x16), _ptr(pooled), _ptr(ws),
                          _stream()), "vsa_stage")
    return (x16, pooled) if want_pooled else x16


def coarse_select(cfg: Config, q, k, v, ws):
    """bf16 q, k, v (cfg.layout order) -> (qc, kc, vc, oc, lse_c, idx, cnt)."""
    B, Hd, N, D = q.shape
    nc = N // 64
    cap = cfg.topk if cfg.select_mode == SELECT_TOPK else cfg.kmax
    f = dict(dtype=torch.float32, device=q.device)
    qc, kc, vc, oc = (torch.empty(B, Hd, nc, D, **f) for _ in range(4))
    lse = torch.empty(B, Hd, nc, **f)
    idx = torch.empty(B, Hd, nc, cap, dtype=torch.int32, device=q.device)
    cnt = torch.empty(B, Hd, nc, dtype=torch.int32, device=q.device)
    check(lib().vsa_coarse_select(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(qc),
                                  _ptr(kc), _ptr(vc), _ptr(oc), _ptr(lse), _ptr(idx), _ptr(cnt),
                                  _ptr(ws), _stream()), "vsa_coarse_select")
    return qc, kc, vc, oc, lse, idx, cnt


def coarse_select_pooled(cfg: Config, qc, kc, vc, ws):
    """fp32 cube means qc, kc, vc [B,heads,Nc,D] (e.g. from stage) -> (oc, lse_c, idx, cnt):
    vsa_coarse_select with q, k, v NULL, so nothing is pooled again."""
    B, Hd, nc, D = qc.shape
    cap = cfg.topk if cfg.select_mode == SELECT_TOPK else cfg.kmax
    f = dict(dtype=torch.float32, device=qc.device)
    oc = torch.empty(B, Hd, nc, D, **f)
    lse = torch.empty(B, Hd, nc, **f)
    idx = torch.empty(B, Hd, nc, cap, dtype=torch.int32, device=qc.device)
    cnt = torch.empty(B, Hd, nc, dtype=torch.int32, device=qc.device)
    check(lib().vsa_coarse_select(ctypes.byref(cfg), None, None, None, _ptr(qc), _ptr(kc),
                                  _ptr(vc), _ptr(oc), _ptr(lse), _ptr(idx), _ptr(cnt), _ptr(ws),
                                  _stream()), "vsa_coarse_select")
    return oc, lse, idx, cnt


def fine_fwd(cfg: Config, q16, k16, v16, idx, cnt, gc, gf, oc, ws, want_saved=True):
    """Staged fp16 cube-order q, k, v; caller-layout bf16 gates -> (o, o_f, lse_f)."""
    q, k, v = q16, k16, v16
    B, Hd, N, D = q.shape
    o = torch.empty_like(gc)
    of = torch.empty(B, Hd, N, D, dtype=torch.float16, device=q.device) if want_saved else None
    lse = torch.empty(B, Hd, N, dtype=torch.float32, device=q.device) if want_saved else None
    check(lib().vsa_fine_fwd(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(cnt),
                             _ptr(gc), _ptr(gf), _ptr(oc), _ptr(o), _ptr(of), _ptr(lse),
                             _ptr(ws), _stream()), "vsa_fine_fwd")
    return o, of, lse


def stage_fp8(cfg: Config, q, k, v, ws, want_pooled=False):
    """bf16 q, k, v (cfg.layout order) -> e4m3 copies (q8, k8, v8t as uint8),
    scales [B, heads, 3] and, optionally, the cube means (qc, kc, vc)."""
    B, Hd, N, D = q.shape
    u8 = dict(dtype=torch.uint8, device=q.device)
    q8, k8 = torch.empty(B, Hd, N, D, **u8), torch.empty(B, Hd, N, D, **u8)
    v8t = torch.empty(B, Hd, N // 64, D, 64, **u8)
    scales = torch.empty(B, Hd, 3, dtype=torch.float32, device=q.device)
    pooled = [torch.empty(B, Hd, N // 64, D, dtype=torch.float32, device=q.device)
              if want_pooled else None for _ in range(3)]
    check(lib().vsa_stage_fp8(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(q8), _ptr(k8),
                              _ptr(v8t), _ptr(scales), *(_ptr(x) for x in pooled), _ptr(ws),
                              _stream()), "vsa_stage_fp8")
    return (q8, k8, v8t, scales) + (tuple(pooled) if want_pooled else ())


def fine_fwd_fp8(cfg: Config, q8, k8, v8t, scales, idx, cnt, gc, gf, oc, ws, want_lse=True):
    """e4m3 copies from stage_fp8 -> (o, lse_f)."""
    B, Hd, N, D = q8.shape
    o = torch.empty_like(gc)
    lse = torch.empty(B, Hd, N, dtype=torch.float32, device=q8.device) if want_lse else None
    check(lib().vsa_fine_fwd_fp8(ctypes.byref(cfg), _ptr(q8), _ptr(k8), _ptr(v8t), _ptr(scales),
                                 _ptr(idx), _ptr(cnt), _ptr(gc), _ptr(gf), _ptr(oc), _ptr(o),
                                 _ptr(lse), _ptr(ws), _stream()), "vsa_fine_fwd_fp8")
    return o, lse


def forward_fp8(cfg: Config, q, k, v, gc, gf, bufs: Buffers, out=None):
    """Whole inference forward with the e4m3 fine stage; bufs.saved receives
    the copies and coarse results (not usable by backward())."""
    o = torch.empty_like(q) if out is None else out
    check(lib().vsa_forward_fp8(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(gc), _ptr(gf),
                                _ptr(o), _ptr(bufs.saved), _ptr(bufs.ws), _stream()),
          "vsa_forward_fp8")
    return o


def fine_fwd_bf16(cfg: Config, q, k, v, idx, cnt, gc, gf, oc, ws, want_lse=True):
    """bf16 q, k, v read in place (cfg.layout order) -> (o, lse_f)."""
    B, Hd, N, D = q.shape
    o = torch.empty_like(gc)
    lse = torch.empty(B, Hd, N, dtype=torch.float32, device=q.device) if want_lse else None
    check(lib().vsa_fine_fwd_bf16(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(idx),
                                  _ptr(cnt), _ptr(gc), _ptr(gf), _ptr(oc), _ptr(o), _ptr(lse),
                                  _ptr(ws), _stream()), "vsa_fine_fwd_bf16")
    return o, lse


def combine_bwd(cfg: Config, d_o, gc, gf, o_f, oc, ws):
    """-> (dgc, dgf, dof16, doc, delta, gscale); dof16 and delta carry gscale."""
    B, Hd, N, D = d_o.shape
    f = dict(dtype=torch.float32, device=d_o.device)
    gd = dict(dtype=grad_torch_dtype(cfg), device=d_o.device)
    dgc, dgf = torch.empty(B, Hd, N, D, **gd), torch.empty(B, Hd, N, D, **gd)
    dof = torch.empty(B, Hd, N, D, dtype=torch.float16, device=d_o.device)
    doc = torch.empty(B, Hd, N // 64, D, **f)
    delta = torch.empty(B, Hd, N, **f)
    gscale = torch.empty(B, Hd, **f)
    check(lib().vsa_combine_bwd(ctypes.byref(cfg), _ptr(d_o), _ptr(gc), _ptr(gf), _ptr(o_f),
                                _ptr(oc), _ptr(dgc), _ptr(dgf), _ptr(dof), _ptr(doc),
                                _ptr(delta), _ptr(gscale), _ptr(ws), _stream()),
          "vsa_combine_bwd")
    return dgc, dgf, dof, doc, delta, gscale


def coarse_bwd(cfg: Config, qc, kc, vc, oc, lse_c, doc, ws):
    dqc, dkc, dvc = (torch.empty_like(qc) for _ in range(3))
    check(lib().vsa_coarse_bwd(ctypes.byref(cfg), _ptr(qc), _ptr(kc), _ptr(vc), _ptr(oc),
                               _ptr(lse_c), _ptr(doc), _ptr(dqc), _ptr(dkc), _ptr(dvc),
                               _ptr(ws), _stream()), "vsa_coarse_bwd")
    return dqc, dkc, dvc


def fine_bwd(cfg: Config, q16, k16, v16, idx, cnt, lse_f, dof16, delta, dqc, dkc, dvc, ws,
             gscale=None):
    """Staged fp16 operands -> dq, dk, dv (cfg.grad_dtype) in cfg.layout order.

    gscale: the per-slice factor dof16 and delta carry (combine_bwd's output),
    or None for 1."""
    q, k, v, dof = q16, k16, v16, dof16
    B, Hd, N, D = q.shape
    f = dict(dtype=grad_torch_dtype(cfg), device=q.device)
    dq, dk, dv = (torch.empty(B, Hd, N, D, **f) for _ in range(3))
    check(lib().vsa_fine_bwd(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(cnt),
                             _ptr(lse_f), _ptr(dof), _ptr(delta), _ptr(gscale), _ptr(dqc),
                             _ptr(dkc), _ptr(dvc), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                             _stream()),
          "vsa_fine_bwd")
    return dq, dk, dv


def forward(cfg: Config, q, k, v, gc, gf, bufs: Buffers, with_backward=True, out=None):
    o = torch.empty_like(q) if out is None else out
    check(lib().vsa_forward(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(gc), _ptr(gf),
                            _ptr(o), _ptr(bufs.saved), int(with_backward), _ptr(bufs.ws),
                            _stream()), "vsa_forward")
    return o


def backward(cfg: Config, gc, gf, d_o, bufs: Buffers, grads=None):
    B, Hd, N, D = gc.shape
    if grads is None:
        grads = tuple(torch.empty(B, Hd, N, D, dtype=grad_torch_dtype(cfg), device=gc.device)
                      for _ in range(5))
    dq, dk, dv, dgc, dgf = grads
    check(lib().vsa_backward(ctypes.byref(cfg), _ptr(gc), _ptr(gf), _ptr(bufs.saved), _ptr(d_o),
                             _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dgc), _ptr(dgf), _ptr(bufs.ws),
                             _stream()), "vsa_backward")
    return grads


# ------------------------------------------------------------------ autograd

class _VSAFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, gc, gf, cfg_tuple, check_status):
        cfg = Config(*cfg_tuple)
        need = any(t.requires_grad for t in (q, k, v, gc, gf))
        bufs = Buffers(cfg, q.device, with_backward=need, inference_only=not need)
        o = forward(cfg, q, k, v, gc, gf, bufs, with_backward=need)
        if check_status:
            check(bufs.device_status(), "video_sparse_attention (forward, device status)")
        ctx.cfg, ctx.bufs, ctx.check_status = cfg, bufs, check_status
        ctx.save_for_backward(gc, gf)
        return o

    @staticmethod
    def backward(ctx, d_o):
        gc, gf = ctx.saved_tensors
        if d_o.shape != gc.shape:
            raise ValueError(f"gradient of O has shape {tuple(d_o.shape)}, "
                             f"expected {tuple(gc.shape)}")
        d_o = d_o.to(torch.bfloat16).contiguous()
        # the library writes bf16 gradients directly (the config asks for them)
        dq, dk, dv, dgc, dgf = backward(ctx.cfg, gc, gf, d_o, ctx.bufs)
        if ctx.check_status:
            check(ctx.bufs.device_status(), "video_sparse_attention (backward, device status)")
        return dq, dk, dv, dgc, dgf, None, None


def _check_inputs(q, k, v, gc, gf, video_shape, layout):
    """Refuses, before any launch, what the kernels would misread."""
    named = (("q", q), ("k", k), ("v", v), ("gc", gc), ("gf", gf))
    for name, t in named:
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
        if t.dim() != 4:
            raise ValueError(f"{name} must be 4-D [batch, heads, tokens, head_dim], "
                             f"got shape {tuple(t.shape)}")
    for name, t in named[1:]:
        if t.shape != q.shape:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, q has {tuple(q.shape)}")
    if len(video_shape) != 3:
        raise ValueError(f"video_shape must be (T, H, W), got {video_shape!r}")
    T, H, W = (int(x) for x in video_shape)
    if q.shape[2] != T * H * W:
        raise ValueError(f"tokens per slice {q.shape[2]} != T*H*W = {T * H * W}")
    if layout not in ("raster", "cube"):
        raise ValueError(f"layout must be 'raster' or 'cube', got {layout!r}")
    for name, t in named:
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")


def video_sparse_attention(q, k, v, gc, gf, video_shape, *, topk=32, select="topk", mass=0.9,
                           kmin=8, kmax=64, scale=0.0, layout="raster", check_status=True):
    """VSA attention of [B, heads, T*H*W, D] bf16 CUDA tensors (raster or cube order).

    gc, gf: per-token, per-channel gates (same shape and dtype).  Returns O, bf16.
    Gradients flow to q, k, v, gc, gf as bf16 (the cube selection is held fixed).
    All five inputs must be contiguous bf16 CUDA tensors of one shape with
    T*H*W tokens; anything else raises before a kernel is launched.  With
    check_status (the default) the forward and the backward each read the
    library's device status word after their kernels (one stream
    synchronisation each) and raise VSAError if a kernel recorded a failure
    (a bounded wait that expired, a bad index list, a Q/K/V value outside the
    fp16 range or a non-finite gradient).
    """
    _check_inputs(q, k, v, gc, gf, video_shape, layout)
    T, H, W = (int(x) for x in video_shape)
    B, Hd, N, D = q.shape
    if select not in ("topk", "mass"):
        raise ValueError(f"select must be 'topk' or 'mass', got {select!r}")
    cfg = make_config(B, Hd, T, H, W, D, topk=topk, select=select, mass=mass, kmin=kmin,
                      kmax=kmax, scale=scale, layout=layout, grad_dtype="bf16")
    check(lib().vsa_validate(ctypes.byref(cfg)), "video_sparse_attention")
    cfg_tuple = tuple(getattr(cfg, n) for n, _ in Config._fields_)
    return _VSAFunction.apply(q, k, v, gc, gf, cfg_tuple, bool(check_status))
