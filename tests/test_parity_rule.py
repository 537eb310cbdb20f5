"""The draw-comparison rule used by the GPU tests is itself checked here: a
draw it calls decidable under a logit perturbation eps never changes when the
logits move by at most eps (random and adversarial perturbations), and a
draw it calls decidable at eps = 0 is the same when made with the GPU
sampler's fixed-point arithmetic (restated below with float32 NumPy)."""
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


def fixed_point_draw(z, temperature: float, top_p: float, u: float) -> int:
    """The GPU sampler's arithmetic, restated: fp32 masses
    round(exp((z - zmax) * (1/T)) * 2^24), exact integer cumulative sums in
    (logit descending, id ascending) order, cut at the first cumulative mass
    >= ceil(top_p * Z), draw at the first >= floor(u * Zk) + 1."""
    z32 = np.asarray(z, np.float32)
    inv_t = np.float32(1.0) / np.float32(temperature)
    m = np.rint(np.exp((z32 - z32.max()) * inv_t).astype(np.float32) * np.float32(2 ** 24)).astype(np.int64)
    order = np.lexsort((np.arange(z32.size), -z32.astype(np.float64)))
    cum = np.cumsum(m[order])
    Z = int(cum[-1])
    tc = Z if top_p >= 1.0 else min(Z, max(1, int(np.ceil(np.float64(np.float32(top_p)) * Z))))
    k = int(np.searchsorted(cum, tc, side="left"))
    zk = int(cum[k])
    td = min(zk, int(np.floor(np.float64(np.float32(u)) * zk)) + 1)
    return int(order[int(np.searchsorted(cum, td, side="left"))])


@pytest.mark.parametrize("seed", range(12))
def test_fixed_point_sampler_agrees_where_decidable(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.choice([128, 1000, 4097]))
    z = (rng.standard_normal(n) * rng.choice([0.5, 1.0, 2.0, 4.0])).astype(np.float32).astype(np.float64)
    ids = np.arange(n)
    decided = 0
    for trial in range(60):
        T = float(rng.choice([0.5, 0.8, 1.0]))
        top_p = float(np.float32(rng.choice([0.6, 0.8, 0.9, 1.0])))
        u = float(np.float32(rng.random()))
        r = sample_top_p(z, ids, T, top_p, u)
        if draw_decidable(r, T, 0.0):
            decided += 1
            assert fixed_point_draw(z, T, top_p, u) == r.index
    assert decided > 30
