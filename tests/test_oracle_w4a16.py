"""Pins of the oracle's 4-bit weight rule (oracle/w4a16.py) on the CPU.

The model card [P3] "s2-pro-w4a16-late12attn" (opening line) names the
variant -- 4-bit weights, 16-bit activations, the late 12 attention layers
in bf16 -- but prints no quantiser or format, so the pins are a hand-derived
worked example of the format (tests/golden/w4a16_pack_row.txt), exact round
trips on values already on the grid, the rounding bound of a group, a
brute-force dot product over the packed bytes, and the identity of the
whole model on weights the rule leaves unchanged.
"""
import os

import numpy as np
import pytest

from dualar_inputs import S2PRO, TINY
from dualar_inputs import generators as g
from dualar_inputs.generators import bf16_bits_to_f32, f32_to_bf16_bits
from oracle import DualAROracle, Sampling
from oracle import w4a16 as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "w4a16_pack_row.txt")


def golden():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, *v = line.split()
            out[k] = v
    return out


def on_grid(n, k, rng, exps=(-4, -9)):
    """bf16 bits of weights q * 2^e that the rule reproduces exactly: q in
    [-7, 7] with a +-7 in every group, e drawn per group."""
    q = rng.integers(-7, 8, size=(n, k // 128, 128))
    q[:, :, 0] = np.where(rng.random((n, k // 128)) < 0.5, 7, -7)
    e = rng.integers(exps[1], exps[0] + 1, size=(n, k // 128, 1)).astype(np.float64)
    w = (q * np.exp2(e)).astype(np.float32).reshape(n, k)
    bits = f32_to_bf16_bits(w)
    assert np.array_equal(bf16_bits_to_f32(bits), w)   # exact in bf16
    return bits, q.reshape(n, k).astype(np.int8), np.exp2(e[:, :, 0]).astype(np.float32)


def test_pack_matches_hand_worked_row():
    gd = golden()
    k = int(gd["k"][0])
    j = np.arange(k)
    w = (((j % 15) - 7) / 16.0).astype(np.float32)[None, :]
    q, sb = W.quantize(f32_to_bf16_bits(w))
    assert sb[0, 0] == int(gd["scale_bits"][0], 16)
    np.testing.assert_array_equal(q[0], (j % 15) - 7)
    p = W.pack(q, sb)
    assert p.shape == (1, W.record_bytes(k)) == (1, 80)
    assert [int(x, 16) for x in gd["bytes_0_8"]] == list(p[0, :8])
    assert int(gd["byte_63"][0], 16) == p[0, 63]
    assert [int(x, 16) for x in gd["bytes_64_80"]] == list(p[0, 64:80])
    q2, s2 = W.unpack(p, k)
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_array_equal(s2, sb)


def test_record_sizes():
    # k/2 code bytes + k/128 bf16 scales rounded up to 16 bytes
    assert W.record_bytes(128) == 64 + 16
    assert W.record_bytes(2560) == 1280 + 48       # 20 scales = 40 bytes -> 48
    assert W.record_bytes(4096) == 2048 + 64       # 32 scales = 64 bytes
    assert W.record_bytes(9728) == 4864 + 160      # 76 scales = 152 bytes -> 160
    for k in (128, 256, 768, 2560, 4096, 9728):
        assert W.record_bytes(k) % 16 == 0


def test_on_grid_weights_round_trip_exactly():
    rng = np.random.default_rng(1)
    bits, q, s = on_grid(6, 512, rng)
    q2, sb = W.quantize(bits)
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_array_equal(bf16_bits_to_f32(sb), s)
    np.testing.assert_array_equal(W.dequantize(q2, sb), bf16_bits_to_f32(bits))
    q3, s3 = W.unpack(W.pack(q2, sb), 512)
    np.testing.assert_array_equal(q3, q2)
    np.testing.assert_array_equal(s3, sb)


def test_group_rounding_bound_and_scale():
    """Groups of very different size along k: each group's error is within
    half its own step, its scale is bf16(max/7), and no code leaves [-7, 7]
    (max/s <= 7 / (1 - 2^-9) < 7.5)."""
    rng = np.random.default_rng(2)
    n, k = 8, 1024
    mag = 10.0 ** (np.arange(k // 128) % 3 - 2)        # 0.01, 0.1, 1 along k
    w = (rng.standard_normal((n, k)) * np.repeat(mag, 128)[None, :]).astype(np.float32)
    bits = f32_to_bf16_bits(w)
    wf = bf16_bits_to_f32(bits).astype(np.float64)
    q, sb = W.quantize(bits)
    s = bf16_bits_to_f32(sb).astype(np.float64)
    m = np.abs(wf).reshape(n, k // 128, 128).max(axis=2)
    assert np.all(np.abs(s - m / 7) <= (m / 7) * 2.0 ** -8)
    assert q.min() >= -7 and q.max() <= 7
    err = np.abs(W.dequantize(q, sb).astype(np.float64) - wf).reshape(n, k // 128, 128)
    assert np.all(err <= s[:, :, None] * 0.5 * (1 + 1e-6))
    # per group, not per row: the small groups keep small errors
    assert err[:, 0::3].max() < 0.01


def test_zero_group():
    bits = np.zeros((2, 256), np.uint16)
    bits[1, 128:] = f32_to_bf16_bits(np.full(128, 0.5, np.float32))
    q, sb = W.quantize(bits)
    assert sb[0, 0] == 0 and sb[0, 1] == 0 and sb[1, 0] == 0
    assert not q[0].any() and not q[1, :128].any()
    np.testing.assert_array_equal(q[1, 128:], 7)
    np.testing.assert_array_equal(W.dequantize(q, sb)[0], 0.0)


def test_packed_dot_product_brute_force():
    """sum_j (u_j - 8) * s_(j/128) * x_j read nibble by nibble from the bytes
    equals the dequantised matrix times x."""
    rng = np.random.default_rng(3)
    n, k = 3, 256
    bits = f32_to_bf16_bits((rng.standard_normal((n, k)) * 0.02).astype(np.float32))
    q, sb = W.quantize(bits)
    p = W.pack(q, sb)
    x = rng.standard_normal(k)
    ref = W.dequantize(q, sb).astype(np.float64) @ x
    for r in range(n):
        acc = 0.0
        for j in range(k):
            byte = int(p[r, j // 2])
            u = (byte >> 4) if j % 2 else (byte & 15)
            grp = j // 128
            sbits = int(p[r, k // 2 + 2 * grp]) | (int(p[r, k // 2 + 2 * grp + 1]) << 8)
            scale = float(np.array([sbits << 16], np.uint32).view(np.float32)[0])
            acc += (u - 8) * scale * x[j]
        assert abs(acc - ref[r]) <= 1e-9 * max(1.0, abs(ref[r]))


def test_late_attn_keys():
    keys = W.late_attn_keys(S2PRO.n_layer, S2PRO.fast_n_layer, 12)
    # 24 early slow layers pack q/k/v and o; all 36 pack the MLP; the fast AR packs everything
    assert len(keys) == 24 * 2 + 36 * 3 + 4 * 5
    assert "slow.23.wqkv" in keys and "slow.23.wo" in keys
    assert "slow.24.wqkv" not in keys and "slow.35.wo" not in keys
    assert "slow.35.w_down" in keys and "fast.3.wqkv" in keys
    assert not any(k.startswith(("tok_emb", "fast_out", "fusion", "fast_emb")) for k in keys)


def test_model_unchanged_on_grid_weights():
    """Weights the rule reproduces exactly: the oracle through the 4-bit
    rule equals the plain oracle bit for bit (prefill and a frame), so the
    rule replaces exactly the named matrices and nothing else."""
    rng = np.random.default_rng(4)
    bits = g.make_weights(TINY, seed=0)
    keys = W.late_attn_keys(TINY.n_layer, TINY.fast_n_layer, 1)
    for key in keys:
        n, k = bits[key].shape
        bits[key] = on_grid(n, k, rng, exps=(-5, -8))[0]
    prompt = g.make_prompt(TINY, 20, seed=5)
    uni = g.make_uniforms(1, 1, TINY, seed=6)[0, 0]
    smp = Sampling(temperature=0.8, top_p=0.8, ras_win=10)
    outs = []
    for kk in (None, keys):
        o = DualAROracle(TINY, bits, max_pos=256, w4a16_keys=kk)
        seq = o.prefill(prompt)
        r = o.decode_frame(seq, uni, smp)
        outs.append((seq.h_last, r.slow_logits, r.fast_logits, r.codes))
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)


def test_model_changes_off_grid():
    """On the generator's weights the rule does change the logits (the
    matrices are really replaced), by a small relative amount."""
    bits = g.make_weights(TINY, seed=0)
    keys = W.late_attn_keys(TINY.n_layer, TINY.fast_n_layer, 1)
    prompt = g.make_prompt(TINY, 20, seed=5)
    z = []
    for kk in (None, keys):
        o = DualAROracle(TINY, bits, max_pos=256, w4a16_keys=kk)
        z.append(o.prefill(prompt).z_last)
    d = np.abs(z[0] - z[1]).max()
    assert 1e-3 < d < 0.5 * np.abs(z[0]).max()


# ------------------------------------------------------ planted mistakes --
# Each plants a plausible mistake in the oracle's 4-bit rule (on the CPU) and
# checks that one of the pins above fails.

def _expect_failure(monkeypatch, name, bad, pin):
    monkeypatch.setattr(W, name, bad)
    with pytest.raises(AssertionError):
        pin()
    monkeypatch.undo()


def test_planted_nibble_order_swap_is_caught(monkeypatch):
    orig = W.pack

    def bad(q, s_bits):
        p = orig(q, s_bits)
        k = q.shape[1]
        p[:, :k // 2] = (p[:, :k // 2] >> 4) | ((p[:, :k // 2] & 15) << 4)
        return p
    _expect_failure(monkeypatch, "pack", bad, test_pack_matches_hand_worked_row)


def test_planted_scale_divisor_is_caught(monkeypatch):
    def bad(w_bits):
        n, k = w_bits.shape
        w = bf16_bits_to_f32(w_bits).reshape(n, k // 128, 128)
        s_bits = f32_to_bf16_bits(np.abs(w).max(axis=2) / np.float32(8.0))   # /8 instead of /7
        s = bf16_bits_to_f32(s_bits)
        q = np.clip(np.rint(w / np.where(s > 0, s, 1)[:, :, None]), -8, 7)
        return q.astype(np.int8).reshape(n, k), s_bits
    _expect_failure(monkeypatch, "quantize", bad, test_on_grid_weights_round_trip_exactly)


def test_planted_row_scale_is_caught(monkeypatch):
    def bad(w_bits):
        # one scale per row (its largest |w|) instead of one per group of 128
        n, k = w_bits.shape
        w = bf16_bits_to_f32(w_bits)
        s_bits = f32_to_bf16_bits(np.abs(w).max(axis=1) / np.float32(7.0))
        s = bf16_bits_to_f32(s_bits)
        q = np.clip(np.rint(w / np.where(s > 0, s, 1)[:, None]), -8, 7)
        return q.astype(np.int8), np.repeat(s_bits[:, None], k // 128, axis=1)
    _expect_failure(monkeypatch, "quantize", bad, test_group_rounding_bound_and_scale)


def test_planted_offset_sign_is_caught(monkeypatch):
    orig = W.pack

    def bad(q, s_bits):
        return orig((-q.astype(np.int16)).clip(-8, 7).astype(np.int8), s_bits)   # stores 8 - q
    _expect_failure(monkeypatch, "pack", bad, test_pack_matches_hand_worked_row)

