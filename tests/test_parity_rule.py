"""The draw-comparison rule used by the GPU tests is itself checked here: a
draw it calls decidable under a logit perturbation eps never changes when the
logits move by at most eps (random and adversarial perturbations)."""
import numpy as np
import pytest

from oracle.sampler import sample_top_p
from parity import draw_decidable


@pytest.mark.parametrize("seed", range(40))
def test_decidable_draws_survive_perturbation(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 300))
    z = rng.standard_normal(n) * rng.choice([0.3, 1.0, 3.0])
    ids = np.arange(n)
    T = float(rng.choice([0.0, 0.5, 0.8, 1.0, 1.5]))
    top_p = float(rng.choice([0.5, 0.8, 0.9, 1.0]))
    eps = float(rng.choice([1e-4, 1e-3, 4e-3, 2e-2]))
    decided = 0
    for trial in range(30):
        u = float(rng.random())
        r = sample_top_p(z, ids, T, top_p, u)
        if not draw_decidable(r, T, eps):
            continue
        decided += 1
        for _ in range(10):
            e = rng.uniform(-eps, eps, n)
            if rng.random() < 0.5:
                e = np.sign(e) * eps          # extreme corners
            r2 = sample_top_p(z + e, ids, T, top_p, u)
            assert r2.index == r.index
