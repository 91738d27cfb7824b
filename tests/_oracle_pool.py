"""Many oracle verify rounds over fixed logits, spread over host processes.

The repeated-draw tests run the fp64 oracle once per uniform set; one round
over the headline's 72 logit rows takes a good fraction of a second of numpy
time, so thousands of rounds go to a pool of worker processes.  The pool is
started with the ``spawn`` method (fresh interpreters that never touch CUDA,
safe to start after the GPU is in use); each worker maps the logits from
``.npy`` files once and runs ``oracle.verify_sampling`` unchanged."""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

_CACHE = {}
KEEP = ("tokens", "num_accepted", "accept_margin", "accept_prob", "draw_lo", "draw_hi", "draw_mass",
        "residual_mass")


def _load(path):
    if path not in _CACHE:
        _CACHE[path] = np.load(path, mmap_mode="r")
    return _CACHE[path]


def _rounds(task):
    zp_path, zq_path, x, us, T = task
    import oracle
    zp, zq = _load(zp_path), _load(zq_path)
    out = []
    for u in us:
        ref = oracle.verify_sampling(zp, zq, x, u, T)
        out.append({k: ref[k] for k in KEEP})
    return out


class OraclePool:
    def __init__(self, processes: int | None = None):
        n = processes or max(1, min(16, (os.cpu_count() or 2) - 1))
        self.pool = mp.get_context("spawn").Pool(n)
        self.n = n

    def verify_rounds(self, tmpdir, tag, z_p, z_q, x, us, T):
        """oracle.verify_sampling(z_p, z_q, x, us[i], T) for every i, in order."""
        zp_path = os.path.join(str(tmpdir), f"{tag}_zp.npy")
        zq_path = os.path.join(str(tmpdir), f"{tag}_zq.npy")
        np.save(zp_path, np.ascontiguousarray(z_p, dtype=np.float64))
        np.save(zq_path, np.ascontiguousarray(z_q, dtype=np.float64))
        per = max(1, len(us) // (4 * self.n))
        tasks = [(zp_path, zq_path, x, us[i:i + per], T) for i in range(0, len(us), per)]
        out = []
        for part in self.pool.imap(_rounds, tasks):
            out.extend(part)
        return out

    def close(self):
        self.pool.terminate()
        self.pool.join()
