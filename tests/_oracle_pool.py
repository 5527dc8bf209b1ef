"""Runs the fp64 oracle over many matrices on all host cores (test helper).

The oracle is plain numpy; one process per matrix (started with `spawn`, so
that no CUDA state is inherited) with its BLAS threads set so that the pool
fills the host's cores.  Workers receive the GPU's bf16 inputs and outputs as
float32 arrays and return the comparison figures, so that only small results
come back.  No method arithmetic is written here: the workers call the oracle.
"""

from __future__ import annotations

import math
import multiprocessing as mp
import os

import numpy as np


def _init(threads):
    os.environ["OMP_NUM_THREADS"] = str(threads)
    os.environ["OPENBLAS_NUM_THREADS"] = str(threads)


def _ns_error_plain(job):
    from oracle import muon_oracle as O
    G, got = job[0], job[1]
    want = O.newton_schulz(G.astype(np.float64))
    got = got.astype(np.float64)
    err = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))
    dev = None
    if len(job) > 2:
        # constructed spectrum G = U diag(s) V^T: the output's singular values
        # along U, V follow the scalar quintic map of s / (||s|| + eps)
        U, s, V = (x.astype(np.float64) for x in job[2:5])
        s0 = s / (math.sqrt(float(np.sum(s * s))) + 1e-7)
        p = s0.copy()
        for _ in range(5):
            p = O.QUINTIC[0] * p + O.QUINTIC[1] * p ** 3 + O.QUINTIC[2] * p ** 5
        core = np.sum((U.T @ got) * V.T, axis=1)      # diag(U^T O V)
        big = s0 >= 1e-2
        dev = float(np.max(np.abs(core[big] - p[big]))) if big.any() else 0.0
    return err, dev


def oracle_errors(jobs, count, workers=None):
    """Maps _ns_error_plain over the `count` jobs that the iterable `jobs` yields
    (built lazily, so that only the jobs in flight are held), on a spawn pool;
    returns the list of results in order."""
    if count == 0:
        return []
    cores = os.cpu_count() or 1
    workers = max(1, min(workers or cores, count, cores))
    threads = max(1, cores // workers)
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS")}
    try:
        _init(threads)   # the spawned children read these at numpy's import
        ctx = mp.get_context("spawn")
        with ctx.Pool(workers, initializer=_init, initargs=(threads,)) as pool:
            out, it = [], iter(jobs)
            while len(out) < count:   # at most two jobs per worker held at a time
                batch = [job for _, job in zip(range(min(2 * workers, count - len(out))), it)]
                out.extend(pool.map(_ns_error_plain, batch, chunksize=1))
            return out
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
