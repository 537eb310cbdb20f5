"""Runs the CPU oracle for many sequences at once in worker processes.

Test helper.  Workers start with the "spawn" method, so they never inherit a
CUDA context from the test process, and each builds its own oracle from the
seeded weights once.  A task is one sequence: a seeded prompt, then
teacher-forced frames; the result holds the arrays the parity tests compare.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

_ORACLE = None


def _init(cfg_name: str, max_pos: int) -> None:
    global _ORACLE
    from dualar_inputs import generators as g
    from dualar_inputs.config import CONFIGS
    from oracle import DualAROracle
    cfg = CONFIGS[cfg_name]
    _ORACLE = DualAROracle(cfg, g.make_weights(cfg, seed=0), max_pos=max_pos)


def run_sequence(task: dict) -> dict:
    """task: prompt (int array), forced [F, N], uniforms [F, N+1], sampling
    (dict of oracle.Sampling fields).  Returns the prefill state, each
    frame's restricted slow logits and fast logits, and the state after the
    last frame."""
    from oracle import Sampling
    o = _ORACLE
    prompt = np.asarray(task["prompt"], np.int32)
    seq = o.prefill_one_layer(prompt) if o.cfg.n_layer == 1 else o.prefill(prompt)
    out = {"h0": seq.h_last.copy(), "z0": seq.z_last.copy(), "slow": [], "fast": []}
    smp = Sampling(**task["sampling"])
    for f in range(len(task["forced"])):
        r = o.decode_frame(seq, task["uniforms"][f], smp, forced=task["forced"][f])
        out["slow"].append(r.slow_logits)
        out["fast"].append(r.fast_logits)
    out["h_end"], out["z_end"] = seq.h_last.copy(), seq.z_last.copy()
    return out


def pool(cfg_name: str, max_pos: int, workers: int | None = None):
    """A spawn pool whose workers each hold an oracle of the named config.
    BLAS threads per worker are split so the pool uses the host's cores."""
    n = workers or max(1, min(8, (os.cpu_count() or 2) // 2))
    threads = max(1, (os.cpu_count() or n) // n)
    saved = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS")}
    for k in saved:
        os.environ[k] = str(threads)
    try:
        return mp.get_context("spawn").Pool(n, initializer=_init, initargs=(cfg_name, max_pos))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
