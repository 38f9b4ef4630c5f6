"""The fp64 oracle over whole layers, in a pool of host processes.

TEST INFRASTRUCTURE ONLY, like the oracle itself: used by tests/ and by the
CPU-baseline legs of bench.py, never by the product path.

Full-coverage parity compares every output element of a layer with the
oracle.  One (batch, head) slice of the pretraining layer is ~0.3 TFLOP of
fp64 work in the oracle's literal masked-dense form, so the slices (and the
query cubes of one large slice) are spread over a pool of processes, each
running the oracle single-threaded.

The pool is started with the "spawn" method (a forked child of a process that
has used CUDA can hang), before or after the caller's GPU work.  Inputs reach
the workers as .npy files of the exact bf16 values (as float32) in a temporary
directory; workers map them read-only.  Nothing here computes any part of the
method: it only moves inputs to oracle.vsa_oracle.Head and results back.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import shutil
import tempfile

import numpy as np

NAMES = ("q", "k", "v", "gc", "gf", "do")
_BLAS_ENV = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def _path(d, tag, name, b, h):
    return os.path.join(d, f"{tag}_{name}_{b}_{h}.npy")


# ------------------------------------------------------------------ worker side

_cache = {}  # the worker's current slice: key -> oracle Head


def _head(task):
    from oracle import vsa_oracle as O
    key = (task["dir"], task["tag"], task["b"], task["h"])
    if key not in _cache:
        _cache.clear()
        d, tag, b, h = key
        arr = {n: np.load(_path(d, tag, n, b, h), mmap_mode="r")
               for n in NAMES if os.path.exists(_path(d, tag, n, b, h))}
        T, H, W = task["thw"]
        hd = O.Head(*(np.asarray(arr[n], dtype=np.float64) for n in NAMES[:5]), T, H, W,
                    task["sel"], task.get("scale"))
        if "do" in arr and task["backward"]:
            hd.set_grad(np.asarray(arr["do"], dtype=np.float64))
        _cache[key] = hd
    return _cache[key]


def _run(task):
    """Oracle results of one slice for the query cubes of `task` (cube-major rows)."""
    hd = _head(task)
    out = {"b": task["b"], "h": task["h"], "cubes": list(task["cubes"])}
    if task["coarse"]:
        out.update(idx=hd.idx, cnt=hd.cnt, oc=hd.coarse["out"], lse_c=hd.coarse["lse"], qc=hd.qc)
    o, of, lse, dq, dgc, dgf = [], [], [], [], [], []
    for c in task["cubes"]:
        _, f, l = hd.rows(c)
        of.append(f)
        lse.append(l)
        o.append(hd.output_tiled(c))
        if task["backward"]:
            rq, rgc, rgf = hd.grad_query_cube(c)
            dq.append(rq)
            dgc.append(rgc)
            dgf.append(rgf)
    if not task["cubes"]:
        return out
    out.update(o=np.stack(o), o_f=np.stack(of), lse_f=np.stack(lse))
    if task["backward"]:
        out.update(dq=np.stack(dq), dgc=np.stack(dgc), dgf=np.stack(dgf))
        out["dk_part"], out["dv_part"] = hd.fine_key_partials(task["cubes"])
        if task["coarse"]:
            out["dk_pool"] = np.repeat(hd.dkc / 64, 64, axis=0)
            out["dv_pool"] = np.repeat(hd.dvc / 64, 64, axis=0)
    for c in task["cubes"]:
        hd.forget(c)
    return out


# ------------------------------------------------------------------ parent side

class OraclePool:
    """A spawn-started process pool plus a directory of input slices."""

    def __init__(self, processes: int | None = None):
        n = processes or min(16, os.cpu_count() or 1)
        saved = {k: os.environ.get(k) for k in _BLAS_ENV}
        for k in _BLAS_ENV:  # one BLAS thread per worker: the pool is the parallelism
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(n)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.processes = n
        self.dir = tempfile.mkdtemp(prefix="vsa_oracle_")
        self.calls = 0  # makes every call's file names (and worker caches) its own
        self.memo = {}

    def close(self):
        self.pool.terminate()
        self.pool.join()
        shutil.rmtree(self.dir, ignore_errors=True)

    def layer_memo(self, key, inp, slices, tag, backward, **kw):
        """layer() once per key (for results that several tests compare against)."""
        if key not in self.memo:
            self.memo[key] = self.layer(inp, slices, tag, backward, **kw)
        return self.memo[key]

    def layer(self, inp, slices, tag, backward, chunk=None, cubes=None, scale=None):
        """Oracle outputs for whole slices of a synth.Inputs-like object.

        inp: has .wl and bf16 CPU tensors q, k, v, gc, gf (and do when
        backward).  slices: (b, h) pairs.  cubes: query cubes to compute (all by
        default).  Returns {(b, h): dict} with cube-major o, o_f, lse_f, the
        coarse results and, for the backward, dq, dgc, dgf over those cubes and
        dk, dv over every key cube (complete only when every query cube was
        computed).
        """
        wl = inp.wl
        cubes = list(range(wl.cubes)) if cubes is None else list(cubes)
        self.calls += 1
        tag = f"{tag}{self.calls}"
        for b, h in slices:
            for n in NAMES:
                t = getattr(inp, n, None)
                if t is None or (n == "do" and not backward):
                    continue
                np.save(_path(self.dir, tag, n, b, h), t[b, h].float().numpy())
        if chunk is None:  # about two tasks per worker
            chunk = max(1, -(-len(slices) * len(cubes) // (2 * self.processes)))
        sel = {"mode": wl.select, "topk": wl.topk, "mass": wl.mass, "kmin": wl.kmin,
               "kmax": wl.kmax}
        tasks = []
        for b, h in slices:
            for i in range(0, max(1, len(cubes)), chunk):
                tasks.append({"dir": self.dir, "tag": tag, "b": b, "h": h,
                              "thw": (wl.T, wl.H, wl.W), "sel": sel, "scale": scale,
                              "cubes": cubes[i:i + chunk], "backward": backward,
                              "coarse": i == 0})
        res = {}
        for r in self.pool.imap_unordered(_run, tasks):
            key = (r["b"], r["h"])
            acc = res.setdefault(key, {"parts": []})
            acc["parts"].append(r)
        out = {}
        for key, acc in res.items():
            parts = sorted(acc["parts"], key=lambda r: r["cubes"][0] if r["cubes"] else -1)
            d = {"cubes": [c for r in parts for c in r["cubes"]]}
            first = parts[0]
            for n in ("idx", "cnt", "oc", "lse_c", "qc"):
                d[n] = first[n]
            if not cubes:
                out[key] = d
                continue
            for n in ("o", "o_f", "lse_f") + (("dq", "dgc", "dgf") if backward else ()):
                d[n] = np.concatenate([r[n] for r in parts])
            if backward:
                d["dk"] = first["dk_pool"] + sum(r["dk_part"] for r in parts)
                d["dv"] = first["dv_pool"] + sum(r["dv_part"] for r in parts)
            out[key] = d
        for b, h in slices:
            for n in NAMES:
                p = _path(self.dir, tag, n, b, h)
                if os.path.exists(p):
                    os.remove(p)
        return out
