"""4-bit weights with 16-bit activations (w4a16): the oracle's packing rule.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the CPU-baseline
leg of the benchmark may import this module.  It shares no code with the
CUDA library.

Page cited (title, then section):
  [P3] "s2-pro-w4a16-late12attn" (model card), opening line: the S2-Pro
       checkpoint with 4-bit weights, keeping the attention of the late 12
       layers in BF16.

The card names the variant but prints no quantiser and no packing format.
Readings taken here (each is also listed, with its reason, in the design
notes):
  * symmetric per-group quantisation along the input dimension, groups of
    128 consecutive elements of one output row, no zero point;
  * the scale of a group is bf16(m / 7), m its largest |w|, the division in
    float32 and the bf16 rounding to nearest even; codes q = rint(w / s)
    (float32 division, ties to even) clamped to [-8, 7], and q = 0 where s = 0;
  * a weight stands for q * s (exact in float32);
  * "late12attn": the query/key/value and output projections of the last 12
    slow layers stay bf16; every other projection of the slow and fast
    stacks is packed; embeddings, norms and both heads stay bf16;
  * "a16": activations are not quantised (the oracle keeps float32).

Packed bytes (the library's format, checked bit for bit): one record per
output row of k/2 + roundup(k/64, 16) bytes: byte i holds the codes of
elements 2i (low nibble) and 2i+1 (high nibble) as u = q + 8; then the k/128
bf16 scales, little-endian; then zeros.
"""
from __future__ import annotations

import numpy as np

from dualar_inputs.generators import bf16_bits_to_f32, f32_to_bf16_bits

GROUP = 128


def record_bytes(k: int) -> int:
    """Bytes of one packed row of k elements."""
    if k <= 0 or k % GROUP:
        raise ValueError("k must be a positive multiple of 128")
    return k // 2 + ((k // 64 + 15) // 16) * 16


def quantize(w_bits: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """bf16 bits [n, k] -> (codes int8 [n, k] in [-8, 7], scale bits uint16
    [n, k/128]) by the group rule in the module docstring."""
    n, k = w_bits.shape
    if k % GROUP:
        raise ValueError("k must be a multiple of 128")
    w = bf16_bits_to_f32(w_bits).reshape(n, k // GROUP, GROUP)
    m = np.abs(w).max(axis=2)                                        # [n, groups], float32
    s_bits = f32_to_bf16_bits(m / np.float32(7.0))
    s = bf16_bits_to_f32(s_bits)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    q = w / safe[:, :, None]                                         # float32 / float32
    np.rint(q, out=q)                                                # ties to even
    q *= (s > 0)[:, :, None]                                         # q = 0 where s = 0
    np.clip(q, -8, 7, out=q)
    return q.astype(np.int8).reshape(n, k), s_bits


def dequantize(q: np.ndarray, s_bits: np.ndarray) -> np.ndarray:
    """(codes [n, k], scale bits [n, k/128]) -> float32 weights q * s."""
    n, k = q.shape
    s = bf16_bits_to_f32(s_bits)
    return (q.reshape(n, k // GROUP, GROUP).astype(np.float32) * s[:, :, None]).reshape(n, k)


def pack(q: np.ndarray, s_bits: np.ndarray) -> np.ndarray:
    """(codes, scale bits) -> uint8 [n, record_bytes(k)] in the library's
    record format."""
    n, k = q.shape
    rb = record_bytes(k)
    out = np.zeros((n, rb), np.uint8)
    u = (q.astype(np.int16) + 8).astype(np.uint8)
    out[:, :k // 2] = u[:, 0::2] | (u[:, 1::2] << 4)
    sb = np.ascontiguousarray(s_bits.astype("<u2")).view(np.uint8).reshape(n, -1)
    out[:, k // 2:k // 2 + sb.shape[1]] = sb
    return out


def unpack(packed: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    """Inverse of pack: uint8 [n, record_bytes(k)] -> (codes, scale bits)."""
    n = packed.shape[0]
    codes = packed[:, :k // 2]
    u = np.empty((n, k), np.int16)
    u[:, 0::2] = codes & 0x0F
    u[:, 1::2] = codes >> 4
    s_bits = np.ascontiguousarray(packed[:, k // 2:k // 2 + k // 64]).view("<u2").astype(np.uint16)
    return (u - 8).astype(np.int8), s_bits.reshape(n, k // GROUP)


def late_attn_keys(n_layer: int, fast_n_layer: int, n_bf16_attn: int = 12) -> list[str]:
    """Weight keys packed in the "late12attn" variant with n_bf16_attn late
    slow layers keeping their attention in bf16 ([P3], opening line)."""
    keys = []
    for i in range(n_layer):
        if i < n_layer - n_bf16_attn:
            keys += [f"slow.{i}.wqkv", f"slow.{i}.wo"]
        keys += [f"slow.{i}.w_gate", f"slow.{i}.w_up", f"slow.{i}.w_down"]
    for i in range(fast_n_layer):
        keys += [f"fast.{i}.{m}" for m in ("wqkv", "wo", "w_gate", "w_up", "w_down")]
    return keys
