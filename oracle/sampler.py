"""Oracle sampler: temperature + top-p draw and the repetition-aware resample.

TEST INFRASTRUCTURE (see oracle/model.py).  float64 throughout.

Pages cited:
  [P2] "Fish Audio S2: a Qwen3-4B on the time axis, ...", section "Two
       autoregressions, because ten codebooks is ten times the sequence":
       sample(biased_logits, ...) for q0, sample(logits, ...) for q1..q9
       (unmasked); each slow step also draws a second sample at temperature
       1.0 and top-p 0.9 and uses it whenever the normal sample repeats a
       semantic token from the last 10 frames (RAS_WIN_SIZE = 10).

The pages show the call, not the sampler's body.  The reading used here is
the plain nucleus rule, driven by a caller-supplied uniform u in [0, 1):
  1. p = softmax(z / T) over the candidates (float64);
  2. order candidates by (p descending, token id ascending);
  3. keep the smallest prefix whose cumulative mass reaches top_p (at least
     one candidate);
  4. with Z the kept mass, return the first kept candidate (in that order)
     whose cumulative mass exceeds u * Z; if none does, the last kept one.
T = 0 is greedy: the largest logit, lowest id on exact ties.
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass
class SampleResult:
    index: int            # chosen candidate (index into the candidate list)
    kept: int             # size of the top-p set
    cdf_margin: float     # min |u*Z - B| / Z over the kept CDF boundaries B (incl. 0)
    cut_margin: float     # min |C - top_p| over the cumulative masses C at the cut
    gap: float            # largest minus second-largest logit
    # diagnostics for comparisons under perturbed logits (not used by the draw)
    pos: int = 0                       # rank of the chosen candidate in the sorted order
    z_sorted: np.ndarray | None = None  # candidate logits in the sorted order
    cum: np.ndarray | None = None       # cumulative normalised mass in that order
    u: float = 0.0


def _gap(z: np.ndarray) -> float:
    if z.size < 2:
        return float("inf")
    top2 = np.partition(z, z.size - 2)[-2:]
    return float(top2[1] - top2[0])


def sample_top_p(z, ids, temperature: float, top_p: float, u: float) -> SampleResult:
    z = np.asarray(z, np.float64)
    ids = np.asarray(ids, np.int64)
    gap = _gap(z)
    if temperature <= 0.0:
        m = z.max()
        cand = np.flatnonzero(z == m)
        idx = int(cand[np.argmin(ids[cand])])
        return SampleResult(idx, 1, float("inf"), float("inf"), gap, u=u)
    p = np.exp((z - z.max()) / temperature)
    p = p / p.sum()
    order = np.lexsort((ids, -p))          # p descending, then id ascending
    cum = np.cumsum(p[order])
    k = int(np.searchsorted(cum, top_p, side="left")) + 1
    k = min(max(k, 1), z.size)
    zk = cum[k - 1]
    target = u * zk
    j = int(np.searchsorted(cum[:k], target, side="right"))
    if j >= k:
        j = k - 1
    bounds = np.concatenate([[0.0], cum[:k]])
    cdf_margin = float(np.min(np.abs(target - bounds)) / zk)
    cut = [abs(cum[k - 1] - top_p)]
    if k >= 2:
        cut.append(abs(cum[k - 2] - top_p))
    return SampleResult(int(order[j]), k, cdf_margin, float(min(cut)), gap, pos=j,
                        z_sorted=z[order], cum=cum, u=u)


def q0_candidates(cfg, allow_eos: bool):
    """Candidate token ids for q0 in restricted-logit order: the semantic
    block, then <|im_end|> (dropped when allow_eos is false)."""
    ids = list(range(cfg.sem_begin, cfg.sem_begin + cfg.n_sem))
    if allow_eos:
        ids.append(cfg.im_end_id)
    return np.array(ids, np.int64)


def sample_q0(cfg, z_restricted, smp, history, u_normal: float, u_ras: float):
    """Returns (normal draw, RAS draw, chosen candidate index).

    Candidate index n_sem stands for <|im_end|>.  The RAS draw is always made;
    it replaces the normal draw when ras_win > 0 and the normal draw is a
    semantic index among the last ras_win committed q0 of this sequence.
    <|im_end|> never triggers the resample."""
    ids = q0_candidates(cfg, smp.allow_eos)
    z = np.asarray(z_restricted, np.float64)[:ids.size]
    normal = sample_top_p(z, ids, smp.temperature, smp.top_p, u_normal)
    ras = sample_top_p(z, ids, smp.ras_temperature, smp.ras_top_p, u_ras)
    chosen = normal.index
    if smp.ras_win > 0 and chosen != cfg.n_sem and chosen in history[-smp.ras_win:]:
        chosen = ras.index
    return normal, ras, chosen
