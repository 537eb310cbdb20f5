"""Shared helpers of the GPU parity tests: tolerances and comparison rules.

Tolerances (teacher-forced logits): max |gpu - oracle| <= 0.05 and relative
L2 <= 1e-2.  Sampled ids are compared through replay: the oracle follows the
GPU's committed codes and each GPU draw must equal the oracle's draw from the
oracle's logits unless the draw lies, within what the logit difference and
the GPU sampler's fixed-point arithmetic can move, at a CDF boundary or at
the top-p cut; greedy draws must agree wherever the oracle's top-1/top-2 gap
exceeds 0.1.
"""
from __future__ import annotations

import numpy as np

MAX_ABS = 0.05
REL_L2 = 1e-2
GREEDY_GAP = 0.1
# The GPU sampler's arithmetic: mass = round(expf((z - zmax) * (1/T)) * 2^24)
# in fp32, exact integer sums, integer targets ceil(top_p * Z) and
# floor(u * Zk) + 1.  One mass is off the exact exp(.) * 2^24 by at most
# 0.5 (the rounding) plus MASS_REL of itself (the fp32 exponent argument,
# |a| <= 17.5 where masses are non-zero, and expf).
MASS_UNIT = float(2 ** 24)
MASS_REL = 4e-6


def arith_margins(r, temperature: float) -> tuple[float, float]:
    """(cut, cdf) distances the fixed-point arithmetic can move the
    normalised cumulative masses (the cut over all candidates, the draw over
    the kept ones): relative errors twice (numerator and normaliser) plus
    n/2 rounding units in each of the two sums and one unit for the target."""
    zs = np.asarray(r.z_sorted, np.float64)
    e = np.exp((zs - zs.max()) / temperature)
    n = zs.size
    z_all = MASS_UNIT * e.sum()
    z_kept = MASS_UNIT * e[:r.kept].sum()
    return 2 * MASS_REL + (n + 2) / z_all, 4 * MASS_REL + (n + 2) / z_kept


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


def draw_decidable(r, temperature: float, eps: float = 0.0) -> bool:
    """Whether an oracle draw must be reproduced by a sampler whose logits
    differ from the oracle's by at most eps (max abs) -- i.e. the draw is the
    same for every logit perturbation of that size.

    Greedy: the top-1/top-2 gap exceeds max(0.1, 2 eps).  Sampled: with
    p ~ exp(z / T), a perturbation of eps scales each mass by at most
    exp(+-2 eps / T) after normalisation, so cumulative masses move by at
    most exp(2 eps / T) - 1 (the top-p cut) and normalised-to-kept CDF
    boundaries by at most exp(4 eps / T) - 1 (the draw); adjacent candidates
    whose logits are within 2 eps may swap order.  The draw is decidable when
    the CDF boundaries, the cut, and the logit gaps next to the chosen
    candidate and at the cut all clear those bounds, and the boundaries and
    the cut clear what the GPU's fixed-point arithmetic can move them
    (arith_margins) on top."""
    if temperature <= 0:
        return r.gap > max(GREEDY_GAP, 2 * eps)
    cut_a, cdf_a = arith_margins(r, temperature)
    if not (r.cdf_margin > cdf_a + np.expm1(4 * eps / temperature)
            and r.cut_margin > cut_a + np.expm1(2 * eps / temperature)):
        return False
    if eps > 0 and r.z_sorted is not None:
        zs = r.z_sorted
        for a in (r.pos - 1, r.pos, r.kept - 2, r.kept - 1):
            if 0 <= a and a + 1 < zs.size and zs[a] - zs[a + 1] <= 2 * eps:
                return False
    return True


class DrawStats:
    def __init__(self):
        self.compared = 0
        self.excluded = 0

    def check(self, gpu_idx: int, r, temperature: float, what: str, eps: float = 0.0):
        if draw_decidable(r, temperature, eps):
            self.compared += 1
            assert int(gpu_idx) == int(r.index), f"{what}: gpu {gpu_idx} oracle {r.index}"
        else:
            self.excluded += 1
