"""Algorithmic HBM bytes of one Dual-AR frame (the roofline numerator).

What the method must move per batch step, with the restricted head (the
4,097 allowed rows, not the full 155,776-row vocabulary) and no head on fast
pass 0 (its logits are never sampled):

  slow  : n_layer blocks + final norm + restricted head rows
  fast  : N passes x fast_n_layer blocks + (N-1) x (fast norm + fast head)
  gather: per sequence, N+1 fusion rows and N-1 fast-embedding rows (bf16)
  KV    : per sequence, the slow K and V of every attended position and
          layer (bf16) plus the new position's K and V written

Activations (a few KB per row) are left out; they live in L2.

With packed 4-bit projections (dualar_set_w4a16) a packed [n][k] matrix moves
n records of k/2 + roundup(k/64, 16) bytes instead of 2 n k.
"""
from __future__ import annotations


def packed_row_bytes(k: int) -> int:
    return k // 2 + ((k // 64 + 15) // 16) * 16


def projection_shapes(cfg) -> dict[str, tuple[int, int]]:
    """[out][in] of the five projections of a block."""
    qd = cfg.n_head * cfg.head_dim
    qkv = (cfg.n_head + 2 * cfg.n_kv_head) * cfg.head_dim
    return {"wqkv": (qkv, cfg.dim), "wo": (cfg.dim, qd), "w_gate": (cfg.ffn, cfg.dim),
            "w_up": (cfg.ffn, cfg.dim), "w_down": (cfg.dim, cfg.ffn)}


def weight_bytes_per_step(cfg, packed_keys=()) -> int:
    d = cfg.dim
    slow = cfg.n_layer * cfg.layer_params(cfg.slow_qk_norm) + d + cfg.n_cand_q0 * d
    fast = (cfg.n_codebooks * cfg.fast_n_layer * cfg.layer_params(cfg.fast_qk_norm)
            + (cfg.n_codebooks - 1) * (d + cfg.fast_vocab * d))
    total = 2 * (slow + fast)
    shapes = projection_shapes(cfg)
    for key in packed_keys:
        stack, _, name = key.split(".")
        n, k = shapes[name]
        reads = 1 if stack == "slow" else cfg.n_codebooks
        total -= reads * 2 * n * k
        total += reads * n * packed_row_bytes(k)
    return total


def gather_bytes_per_seq(cfg) -> int:
    return 2 * cfg.dim * ((cfg.n_codebooks + 1) + (cfg.n_codebooks - 1))


def kv_bytes_per_seq(cfg, attended: int) -> int:
    """attended = positions the slow step attends over (context incl. new)."""
    per_pos = cfg.n_layer * 2 * cfg.n_kv_head * cfg.head_dim * 2
    return per_pos * attended + per_pos


def frame_bytes(cfg, attended_per_seq, packed_keys=()) -> int:
    """Bytes of one batch step; attended_per_seq: iterable of context lengths."""
    att = list(attended_per_seq)
    return (weight_bytes_per_step(cfg, packed_keys) + len(att) * gather_bytes_per_seq(cfg)
            + sum(kv_bytes_per_seq(cfg, a) for a in att))
