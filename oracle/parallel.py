"""The oracle's MoE layer spread over the host cores, one expert per process.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: used by the full-size
GPU parity tests and by the CPU-baseline / reference legs of ``bench.py``.

The oracle's cost is dominated by dequantising each active expert's two
blocks, not by the token count.  Each worker runs ``apl.moe_layer``
unchanged, with every assignment that is not to its expert left out (a
negative expert id: the function's own way of restricting the experts), and
returns the output rows of the requested tokens; the parent adds the
experts' parts.  The layer output (arXiv text §3.3: the weighted sum of the
routed experts' outputs) is a sum over experts, so this is the oracle's
output up to the order of the float64 additions over experts.  Nothing here
changes the arithmetic of ``apl``.

Block data reaches the workers as .npy files (memory-mapped there), so no
gigabyte-sized array goes through a pipe.  Workers are started with
``spawn`` (safe in a process that has initialised CUDA) and import only
numpy and ``oracle.apl``.  BLAS threads per worker = host cores // workers.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import shutil
import tempfile
import time
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

from . import apl

_BLAS_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class _BlasThreads:
    """Sets the BLAS thread variables that spawned workers inherit."""

    def __init__(self, n: int):
        self.n = str(max(1, int(n)))

    def __enter__(self):
        self.saved = {k: os.environ.get(k) for k in _BLAS_VARS}
        for k in _BLAS_VARS:
            os.environ[k] = self.n
        return self

    def __exit__(self, *a):
        for k, v in self.saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


class ExpertFiles:
    """A temporary directory holding one layer's block data as .npy files:
    parent indices (uint8 [rows][cols]) and the LUT of the committed bitwidth
    (fp16 [rows][2^q], row-major) per (expert, u)."""

    def __init__(self):
        base = "/dev/shm" if os.path.isdir("/dev/shm") and os.access("/dev/shm", os.W_OK) else None
        self.dir = tempfile.mkdtemp(prefix="pw_oracle_", dir=base)
        self.files: Dict[int, Dict[int, Tuple[str, str, int]]] = {}

    def add(self, e: int, u: int, idx: np.ndarray, lut_q: np.ndarray, q: int) -> None:
        ip = os.path.join(self.dir, f"idx_{e}_{u}.npy")
        lp = os.path.join(self.dir, f"lut_{e}_{u}.npy")
        np.save(ip, np.ascontiguousarray(idx, dtype=np.uint8))
        np.save(lp, np.ascontiguousarray(lut_q, dtype=np.float16))
        self.files.setdefault(e, {})[u] = (ip, lp, int(q))

    def save_inputs(self, x: np.ndarray, ids: np.ndarray, w: np.ndarray) -> Tuple[str, str, str]:
        paths = tuple(os.path.join(self.dir, n) for n in ("x.npy", "ids.npy", "w.npy"))
        np.save(paths[0], np.asarray(x))
        np.save(paths[1], np.asarray(ids))
        np.save(paths[2], np.asarray(w, dtype=np.float64))
        return paths

    def close(self) -> None:
        shutil.rmtree(self.dir, ignore_errors=True)

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()


def _expert_part(job):
    e, x_path, ids_path, w_path, I, P, files, tokens = job
    x = np.load(x_path)
    ids = np.load(ids_path)
    w = np.load(w_path)
    blocks = {}
    for u in (0, 1):
        idx_path, lut_path, q = files[u]
        blocks[u] = apl.IndexBlock(np.load(idx_path, mmap_mode="r"), {q: np.load(lut_path)}, q, P)
    y = apl.moe_layer(x, np.where(ids == e, ids, -1), w, I, lambda ee, u: blocks[u], tokens=tokens)
    return y[np.asarray(tokens, dtype=np.int64)]


def layer_rows(files: ExpertFiles, x: np.ndarray, ids: np.ndarray, w: np.ndarray, I: int, P: int,
               tokens: Sequence[int], workers: Optional[int] = None) -> np.ndarray:
    """Oracle output rows y[tokens] (float64 [len(tokens)][H]) of one layer,
    the experts those tokens route to computed in parallel.  ``files`` must
    hold both blocks of each such expert at its committed bitwidth."""
    tokens = sorted(int(t) for t in tokens)
    ids = np.asarray(ids)
    experts = sorted({int(e) for e in ids[tokens].ravel() if e >= 0})
    missing = [e for e in experts if e not in files.files]
    if missing:
        raise KeyError(f"no block data for experts {missing}")
    paths = files.save_inputs(x, ids, w)
    jobs = [(e, *paths, I, P, files.files[e], tokens) for e in experts]
    cores = host_cores()
    n = max(1, min(len(jobs), workers or cores))
    if n == 1:
        parts = [_expert_part(j) for j in jobs]
    else:
        with _BlasThreads(cores // n), mp.get_context("spawn").Pool(n) as pool:
            parts = pool.map(_expert_part, jobs, chunksize=1)
    y = np.zeros((len(tokens), np.asarray(x).shape[1]), dtype=np.float64)
    for part in parts:
        y += part
    return y


def covering_tokens(ids: np.ndarray, extra: int = 0, seed: int = 0) -> list:
    """Tokens chosen so that every (expert, slot) pair that occurs in ``ids``
    occurs among them (greedy, in token order), plus ``extra`` random others."""
    ids = np.asarray(ids)
    T, k = ids.shape
    need = {(int(ids[t, j]), j) for t in range(T) for j in range(k)}
    chosen = []
    for t in range(T):
        pairs = {(int(ids[t, j]), j) for j in range(k)}
        if pairs & need:
            chosen.append(t)
            need -= pairs
        if not need:
            break
    rest = sorted(set(range(T)) - set(chosen))
    if extra and rest:
        rng = np.random.default_rng(seed)
        chosen += rng.choice(rest, size=min(extra, len(rest)), replace=False).tolist()
    return sorted(chosen)


# ----------------------------------------------------------------------------
# Timing: one persistent process per active expert
# ----------------------------------------------------------------------------
def _timing_worker(conn, e, paths, I, P, files):
    """Holds expert e's two blocks as packed bit-planes (apl.Block, the
    oracle's plane-reading path) and runs its share of the layer on command:
    ("run", frac) computes the expert's contribution (apl.moe_layer, frac == 1)
    or the same unpack + LUT + matmul on the first frac of each block's rows
    (apl.apl_linear of the oracle on a row range, frac < 1), and answers with
    the seconds it took."""
    x = np.load(paths[0])
    ids = np.load(paths[1])
    w = np.load(paths[2])
    blocks = {}
    for u in (0, 1):
        idx_path, lut_path, q = files[u]
        idx = np.load(idx_path)
        N, K = idx.shape
        blocks[u] = apl.Block(apl.pack_bitplanes(idx, P), {q: np.load(lut_path)}, q, N, K)
        del idx
    mine = np.where(ids == e, ids, -1)
    rows = sorted(set(np.nonzero(mine >= 0)[0].tolist()))
    conn.send("ready")
    while True:
        msg = conn.recv()
        if msg[0] == "stop":
            break
        frac = float(msg[1])
        t0 = time.perf_counter()
        if frac >= 1.0:
            apl.moe_layer(x, mine, w, I, lambda ee, u: blocks[u], tokens=rows)
        else:
            xe = x[rows].astype(np.float64)
            for u in (0, 1):
                b = blocks[u]
                n = max(128, int(round(b.N * frac / 128)) * 128)
                inp = xe if u == 0 else np.ones((len(rows), b.K))     # stand-in of h's shape
                # the oracle's plane path (unpack, LUT, matmul) on rows [0, n)
                W = apl.dequant(apl.unpack_indices(b.planes, b.q, b.N, b.K, (0, n)), b.luts[b.q], (0, n))
                _ = inp @ W.T
        conn.send(time.perf_counter() - t0)
    conn.close()


class ExpertWorkers:
    """One spawned process per active expert of a layer, each holding its
    expert's blocks; ``step(frac)`` runs every expert's share at once and
    returns the wall-clock seconds of the slowest (the layer's time)."""

    def __init__(self, files: ExpertFiles, x, ids, w, I: int, P: int):
        ids = np.asarray(ids)
        self.experts = sorted({int(e) for e in ids.ravel() if e >= 0})
        self.cores = host_cores()
        paths = files.save_inputs(x, ids, w)
        ctx = mp.get_context("spawn")
        self.procs, self.conns = [], []
        with _BlasThreads(self.cores // max(1, len(self.experts))):
            for e in self.experts:
                a, b = ctx.Pipe()
                p = ctx.Process(target=_timing_worker, args=(b, e, paths, I, P, files.files[e]), daemon=True)
                p.start()
                self.procs.append(p)
                self.conns.append(a)
        for c in self.conns:
            if c.recv() != "ready":
                raise RuntimeError("oracle worker failed to start")

    @property
    def threads_per_worker(self) -> int:
        return max(1, self.cores // max(1, len(self.experts)))

    def step(self, frac: float = 1.0) -> float:
        t0 = time.perf_counter()
        for c in self.conns:
            c.send(("run", frac))
        for c in self.conns:
            c.recv()
        return time.perf_counter() - t0

    def close(self) -> None:
        for c in self.conns:
            try:
                c.send(("stop",))
            except (BrokenPipeError, OSError):
                pass
        for p in self.procs:
            p.join(timeout=30)
            if p.is_alive():
                p.terminate()

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()
