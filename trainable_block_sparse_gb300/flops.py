"""Work counts used for reporting: executed FLOPs and algorithmic HBM bytes.

Executed FLOPs count only selected (query cube, key cube) pairs, as dense
64x64 tiles: forward 2 matmuls (QK^T, PV) = 4*64*64*D per pair; backward
5 matmuls (S recompute, dP, dV, dK, dQ) = 10*64*64*D per pair.  The coarse
stage is 2 matmuls on the pooled sequence: 4*Nc^2*D per (batch, head).
"""
from .synth import TILE


def fine_fwd_pairs(pairs: int, head_dim: int) -> float:
    return 4.0 * TILE * TILE * head_dim * pairs


def fine_bwd_pairs(pairs: int, head_dim: int) -> float:
    return 10.0 * TILE * TILE * head_dim * pairs


def fine_fwd_topk(wl) -> float:
    return fine_fwd_pairs(wl.bh * wl.cubes * wl.topk, wl.head_dim)


def coarse_fwd(wl) -> float:
    return 4.0 * wl.cubes * wl.cubes * wl.head_dim * wl.bh


def tensor_bytes(wl, elem_bytes: int = 2) -> int:
    """Bytes of one [B, heads, N, D] tensor."""
    return wl.bh * wl.tokens * wl.head_dim * elem_bytes
