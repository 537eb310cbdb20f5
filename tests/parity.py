"""Shared helpers of the GPU parity tests: tolerances and comparison rules.

Tolerances (teacher-forced logits): max |gpu - oracle| <= 0.05 and relative
L2 <= 1e-2.  Sampled ids are compared through replay: the oracle follows the
GPU's committed codes and each GPU draw must equal the oracle's draw from the
oracle's logits unless the draw lies within 1e-3 (of the kept mass) of a CDF
boundary or the top-p cut lies within 1e-3 of top_p; greedy draws must agree
wherever the oracle's top-1/top-2 gap exceeds 0.1.
"""
from __future__ import annotations

import numpy as np

MAX_ABS = 0.05
REL_L2 = 1e-2
CDF_DELTA = 1e-3
CUT_DELTA = 1e-3
GREEDY_GAP = 0.1


def assert_logits_close(gpu, ref, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), what
    err = np.abs(gpu - ref).max()
    rel = np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= MAX_ABS, f"{what}: max abs {err:.3g} > {MAX_ABS}"
    assert rel <= REL_L2, f"{what}: rel L2 {rel:.3g} > {REL_L2}"
    return err, rel


def draw_decidable(r, temperature: float) -> bool:
    """Whether an oracle draw is far enough from every boundary to compare."""
    if temperature <= 0:
        return r.gap > GREEDY_GAP
    return r.cdf_margin > CDF_DELTA and r.cut_margin > CUT_DELTA


class DrawStats:
    def __init__(self):
        self.compared = 0
        self.excluded = 0

    def check(self, gpu_idx: int, r, temperature: float, what: str):
        if draw_decidable(r, temperature):
            self.compared += 1
            assert int(gpu_idx) == int(r.index), f"{what}: gpu {gpu_idx} oracle {r.index}"
        else:
            self.excluded += 1
