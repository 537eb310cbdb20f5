"""Pins of the CPU oracle against the pages, closed forms and brute force.

Each test checks one oracle function against something other than itself:
figures the pages print (tests/golden/pages_facts.txt), closed forms,
invariants, or brute-force enumeration.  Tests at the end plant mistakes in
the oracle (on the CPU) and check that a pin catches each of them.
"""
import dataclasses
import itertools
import math
import os

import numpy as np
import pytest

from dualar_inputs import S2PRO, TINY, FRAMES_PER_AUDIO_SECOND
from dualar_inputs import generators as g
import oracle
from oracle import model as om
from oracle.sampler import sample_top_p, sample_q0
from oracle.model import Sampling, SeqState

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_facts.txt")


def facts():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            out[k] = float(v) if "." in v else int(v)
    return out


# ---------------------------------------------------------------- shapes --

def test_param_counts_match_pages():
    f = facts()
    assert S2PRO.total_params() == f["total_params"]
    assert S2PRO.slow_params() == f["slow_params"]
    assert round(S2PRO.fast_params() / 1e6, 1) == f["fast_params_millions"]
    assert S2PRO.fusion_rows == f["fusion_rows"]
    assert round(S2PRO.fusion_params() / 1e6, 1) == f["fusion_params_millions"]
    assert round(S2PRO.fast_pass_params() / 1e6, 1) == f["fast_pass_params_millions"]
    assert S2PRO.slow_params() - f["qwen3_4b_params"] == f["extra_embedding_rows"] * S2PRO.dim
    assert S2PRO.sem_begin == f["semantic_first_id"]
    assert S2PRO.sem_begin + S2PRO.n_sem - 1 == f["semantic_last_id"]
    assert S2PRO.vocab == f["vocab"]
    assert S2PRO.n_codebooks == f["n_codebooks"]
    assert round(FRAMES_PER_AUDIO_SECOND, 2) == f["frames_per_second_2dp"]
    assert S2PRO.n_cand_q0 == f["allowed_q0_candidates"]


def test_fusion_offsets_layout():
    # full size: ten codebooks of 4,096 rows stacked in one 40,960-row table
    assert [S2PRO.fusion_offset(k) for k in range(10)] == [4096 * k for k in range(10)]
    # tiny: 1 x 512 semantic + 3 x 128 acoustic = 896 rows
    assert [TINY.fusion_offset(k) for k in range(4)] == [0, 512, 640, 768]
    assert TINY.fusion_rows == 896


# -------------------------------------------------------------- RMSNorm --

def test_rmsnorm_constant_vector_closed_form():
    for c in (0.5, -3.0, 1e-2):
        x = np.full(256, c, np.float32)
        w = np.linspace(0.5, 1.5, 256).astype(np.float32)
        y = om.rmsnorm(x, w, 1e-6)
        expect = w.astype(np.float64) * c / math.sqrt(c * c + 1e-6)
        np.testing.assert_allclose(y, expect, rtol=2e-6)


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 2560)).astype(np.float32) * 7
    y = om.rmsnorm(x, np.ones(2560, np.float32), 1e-6)
    np.testing.assert_allclose(np.sqrt(np.mean(y.astype(np.float64) ** 2, axis=-1)), 1.0, rtol=1e-5)
    np.testing.assert_allclose(om.rmsnorm(3 * x, np.ones(2560, np.float32), 1e-6), y, rtol=1e-5, atol=1e-6)


# ----------------------------------------------------------------- RoPE --

def test_rope_tables_are_rounded_bf16_of_cos_sin():
    cos, sin = om.rope_table(300, 128, 1e6)
    # every entry is a bf16 value
    for t in (cos, sin):
        bits = t.view(np.uint32)
        assert np.all(bits & 0xFFFF == 0)
    # and within half a bf16 ulp of the exact value
    i = np.arange(64)
    for p in (0, 1, 7, 299):
        ang = p * (1e6 ** (-2.0 * i / 128))
        for tab, fn in ((cos, np.cos), (sin, np.sin)):
            exact = fn(ang)
            ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(exact), 1e-30))) - 7)
            assert np.all(np.abs(tab[p] - exact) <= ulp / 2 + 1e-30)


def test_rope_position_zero_is_identity():
    cos, sin = om.rope_table(16, 64, 1e6)
    x = np.random.default_rng(1).standard_normal((3, 64)).astype(np.float32)
    np.testing.assert_array_equal(om.apply_rope(x, 0, cos, sin), x)


def test_rope_pair_layout_and_angle():
    hd, base = 64, 1e6
    cos, sin = om.rope_table(100, hd, base)
    for i in (0, 1, 5, 31):
        for p in (1, 3, 37, 99):
            e = np.zeros((1, hd), np.float32)
            e[0, 2 * i] = 1.0
            y = om.apply_rope(e, p, cos, sin)[0]
            # the unit vector of pair i rotates within its own pair
            others = np.delete(y, [2 * i, 2 * i + 1])
            assert np.all(others == 0)
            ang = p * base ** (-2.0 * i / hd)
            assert abs(y[2 * i] - math.cos(ang)) < 4e-3
            assert abs(y[2 * i + 1] - math.sin(ang)) < 4e-3
            e2 = np.zeros((1, hd), np.float32)
            e2[0, 2 * i + 1] = 1.0
            y2 = om.apply_rope(e2, p, cos, sin)[0]
            assert abs(y2[2 * i] + math.sin(ang)) < 4e-3
            assert abs(y2[2 * i + 1] - math.cos(ang)) < 4e-3


def test_rope_relative_position_property():
    hd = 64
    cos, sin = om.rope_table(200, hd, 1e6)
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, hd)).astype(np.float32)
    k = rng.standard_normal((1, hd)).astype(np.float32)
    d = []
    for p, s in ((10, 3), (50, 43), (107, 100)):
        d.append(float(om.apply_rope(q, p, cos, sin)[0] @ om.apply_rope(k, s, cos, sin)[0]))
    # depends on p - s only (bf16 tables: agreement to ~1e-2 relative)
    assert max(d) - min(d) < 0.03 * max(1.0, abs(d[0]))
    # and norms are preserved up to the bf16 table error
    y = om.apply_rope(q, 77, cos, sin)
    assert abs(np.linalg.norm(y) / np.linalg.norm(q) - 1) < 1e-2


# ------------------------------------------------------------ attention --

def brute_attention(q, k, v, n_rep, causal_offset):
    tq, hq, hd = q.shape
    out = np.zeros((tq, hq, hd))
    for t in range(tq):
        for h in range(hq):
            gk = h // n_rep
            limit = k.shape[0] if causal_offset is None else causal_offset + t + 1
            s = [sum(float(q[t, h, d]) * float(k[j, gk, d]) for d in range(hd)) / math.sqrt(hd)
                 for j in range(limit)]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = sum(e)
            for d in range(hd):
                out[t, h, d] = sum(e[j] / z * float(v[j, gk, d]) for j in range(limit))
    return out


@pytest.mark.parametrize("tq,tk,hq,hkv,off", [(1, 5, 4, 2, 4), (3, 7, 4, 1, 4), (4, 4, 2, 2, 0)])
def test_attention_matches_brute_force(tq, tk, hq, hkv, off):
    rng = np.random.default_rng(3)
    hd = 8
    q = rng.standard_normal((tq, hq, hd)).astype(np.float32)
    k = rng.standard_normal((tk, hkv, hd)).astype(np.float32)
    v = rng.standard_normal((tk, hkv, hd)).astype(np.float32)
    got = om.gqa_attention(q, k, v, hq // hkv, causal_offset=off)
    np.testing.assert_allclose(got, brute_attention(q, k, v, hq // hkv, off), rtol=1e-5, atol=1e-5)


def test_attention_single_key_returns_value():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 4, 16)).astype(np.float32) * 10
    k = rng.standard_normal((1, 2, 16)).astype(np.float32)
    v = rng.standard_normal((1, 2, 16)).astype(np.float32)
    out = om.gqa_attention(q, k, v, 2, causal_offset=0)
    np.testing.assert_allclose(out[0], np.repeat(v[0], 2, axis=0), rtol=1e-6)


def test_silu_values():
    x = np.array([0.0, 1.0, 30.0, -30.0], np.float32)
    y = om.silu(x)
    assert y[0] == 0.0
    assert abs(y[1] - 0.7310585786300049) < 1e-7       # logistic(1)
    assert abs(y[2] - 30.0) < 1e-5 and abs(y[3]) < 1e-10


# ------------------------------------------------- one transformer block --
#
# A block on hand-set weights small enough to work out by hand: width 4,
# four query heads over two KV heads of size 2, FFN width 4.  Every expected
# number below is the closed form written beside it, not a call into the
# oracle.  [P1] "Fast Transformer: The Codebook Decoder" (pre-norm
# TransformerBlock: attention then SwiGLU FFN, each added to the residual);
# [P2] "The slow AR is Qwen3-4B" (fused q/k/v projection in q, k, v order;
# GQA; qk-norm).

BLOCK_CFG = dataclasses.replace(TINY, name="block_pin", dim=4, n_head=4, n_kv_head=2, head_dim=2, ffn=4)


def _block_weights_a(qk_norm: bool) -> om.LayerW:
    """Attention with one key returns its value row unchanged, whatever q
    and k are; the weights route one value component into the residual and
    drive the SwiGLU gate to the closed-form points SiLU(0), SiLU(2), SiLU(+-20)."""
    f = np.float32
    wqkv = np.zeros((16, 4), f)
    wqkv[0:8] = np.random.default_rng(3).standard_normal((8, 4))   # q: irrelevant with one key
    wqkv[8, 0], wqkv[9, 2], wqkv[10, 0], wqkv[11, 2] = -5, 7, 1, 3    # k_h0 = (-5, 7), k_h1 = (1, 3)
    wqkv[12, 0], wqkv[13, 3], wqkv[14, 0], wqkv[15, 0] = 2, -0.25, -1, 3   # v_h0 = (2, .5), v_h1 = (-1, 3)
    wo = np.zeros((4, 8), f)
    wo[1, 2], wo[1, 3] = 1, 4          # head 1's output (= v_h0) -> 2 + 4 * 0.5 = 4 into h[1]
    return om.LayerW(
        attn_norm=np.array([1, 1, 1, 2], f), wqkv=wqkv,
        q_norm=np.array([0.5, 3], f) if qk_norm else None,
        k_norm=np.array([2, 0.5], f) if qk_norm else None,
        wo=wo, ffn_norm=np.array([1, 2, 1, 1], f),
        w_gate=np.diag([0, 1, 20, 20]).astype(f), w_up=np.diag([5, 3, 2, -7]).astype(f),
        w_down=np.eye(4, dtype=f))


def test_block_single_position_closed_form():
    """h = (2,-2,2,-2): RMSNorm gives u = (1,-1,1,-2) (rms 2, gain (1,1,1,2)),
    so k = (-5,7 | 1,3) and v = (2,.5 | -1,3).  One key: every query head
    outputs its KV head's v, so heads are (v_h0, v_h0, v_h1, v_h1) and wo adds
    4 to h[1]: h' = (2,2,2,-2).  RMSNorm(h') with gain (1,2,1,1) is
    (1,2,1,-1); gate = (0,2,20,-20), up = (5,6,2,7), down = I:
    h_out = h' + (0, 12 L(2), 40 L(20), -140 L(-20)), L the logistic."""
    cfg = BLOCK_CFG
    cos, sin = om.rope_table(4, cfg.head_dim, cfg.rope_base)
    h = np.array([[2, -2, 2, -2]], np.float32)
    empty = np.zeros((0, 2, 2), np.float32)
    expect = np.array([2.0, 12.569564935734588, 41.99999991755385, -2.0000002885615067])
    for kv_bf16 in (False, True):
        out, kc, vc = om.block(cfg, _block_weights_a(False), h, 0, empty, empty, cos, sin,
                               qk_norm=False, kv_bf16=kv_bf16)
        np.testing.assert_allclose(out[0], expect, rtol=1e-6, atol=2e-6)
        np.testing.assert_allclose(kc[0], [[-5, 7], [1, 3]], rtol=1e-6)
        np.testing.assert_allclose(vc[0], [[2, 0.5], [-1, 3]], rtol=1e-6)
    # the rounded cache holds the bf16 neighbours exactly: 5 * (1 - 1.25e-7) -> 5
    assert kc[0].tolist() == [[-5, 7], [1, 3]] and vc[0].tolist() == [[2, 0.5], [-1, 3]]


def test_block_qk_norm_is_per_head_before_the_cache():
    """With qk-norm, each K head is RMS-normalised over head_dim and scaled by
    the k_norm gain (2, .5) before it is cached (position 0: RoPE is the
    identity): (-5,7)/sqrt(37) * (2,.5) and (1,3)/sqrt(5) * (2,.5).  V and,
    with one key, the block output are unchanged."""
    cfg = BLOCK_CFG
    cos, sin = om.rope_table(4, cfg.head_dim, cfg.rope_base)
    h = np.array([[2, -2, 2, -2]], np.float32)
    empty = np.zeros((0, 2, 2), np.float32)
    out, kc, vc = om.block(cfg, _block_weights_a(True), h, 0, empty, empty, cos, sin, qk_norm=True)
    np.testing.assert_allclose(kc[0], [[-1.643989873053573, 0.5753964555687505],
                                       [0.8944271909999159, 0.6708203932499369]], rtol=2e-6)
    np.testing.assert_allclose(vc[0], [[2, 0.5], [-1, 3]], rtol=1e-6)
    np.testing.assert_allclose(out[0], [2.0, 12.569564935734588, 41.99999991755385, -2.0000002885615067],
                               rtol=1e-6, atol=2e-6)


def test_block_two_positions_attention_weights():
    """Two positions, RoPE tables set to the identity, gate = 0 (so the FFN
    adds SiLU(0) * up = 0 exactly).  Row 0 sees only key 0; row 1 sees keys 0
    and 1 with scores q.k / sqrt(2).  k = (u[1], 0) per KV head, so the keys
    are (-1,0) then (1,0); query head 0 is (b, 0) with b = ln 3 / sqrt(2),
    giving weights (1/4, 3/4); head 3 is (-b, 0): (3/4, 1/4); heads 1, 2 are 0:
    (1/2, 1/2).  v_h0 = (u[1], 0), v_h1 = (0, 2 u[3]).  wo picks one output
    component of each head: (a0[0], a3[1], a1[0], a2[1])."""
    cfg = BLOCK_CFG
    f = np.float32
    b = f(0.7768361992120932)
    wqkv = np.zeros((16, 4), f)
    wqkv[0, 0], wqkv[6, 0] = b, -b
    wqkv[8, 1], wqkv[10, 1] = 1, 1
    wqkv[12, 1], wqkv[15, 3] = 1, 2
    wo = np.zeros((4, 8), f)
    wo[0, 0], wo[1, 7], wo[2, 2], wo[3, 5] = 1, 1, 1, 1
    rng = np.random.default_rng(4)
    lw = om.LayerW(attn_norm=np.ones(4, f), wqkv=wqkv, q_norm=None, k_norm=None, wo=wo,
                   ffn_norm=np.ones(4, f), w_gate=np.zeros((4, 4), f),
                   w_up=rng.standard_normal((4, 4)).astype(f), w_down=rng.standard_normal((4, 4)).astype(f))
    cos, sin = np.ones((2, 1), f), np.zeros((2, 1), f)
    h = np.array([[2, -2, 2, -2], [2, 2, 2, 2]], f)
    empty = np.zeros((0, 2, 2), f)
    out, kc, vc = om.block(cfg, lw, h, 0, empty, empty, cos, sin, qk_norm=False)
    # row 0: heads (v_h0, v_h0, v_h1, v_h1) at position 0 = ((-1,0), (-1,0), (0,-2), (0,-2))
    # row 1: head 0 (-1/4 + 3/4, 0), head 1 (0, 0), head 2 (0, 0), head 3 (0, -3/2 + 1/2)
    np.testing.assert_allclose(out, [[1, -4, 1, -4], [2.5, 1, 2, 2]], rtol=1e-6, atol=2e-6)


# ------------------------------------------------ incremental == recompute --

def test_slow_incremental_equals_full_recompute(tiny_oracle):
    o = tiny_oracle
    cfg = TINY
    prompt = g.make_prompt(cfg, 20, seed=5)
    seq = o.prefill(prompt[:12])
    # the rest of the prompt one position at a time
    hs = []
    for t in prompt[12:]:
        hs.append(o.slow_rows(seq, o.w.tok_emb[[t]])[0])
    # then 6 forced frames (fusion inputs)
    forced = g.make_forced_codes(6, 1, cfg, seed=6)
    u = g.make_uniforms(6, 1, cfg, seed=7)
    xs = []
    for f in range(6):
        r = o.decode_frame(seq, u[f, 0], Sampling(), forced=forced[f, 0])
        xs.append(r.x_next)
        hs.append(seq.h_last)
    rows = np.concatenate([o.w.tok_emb[prompt], np.stack(xs)], axis=0)
    full = o.slow_full_recompute(rows)
    np.testing.assert_allclose(np.stack(hs), full[12:], rtol=1e-4, atol=1e-4)
    # logits from the full head + bias equal the restricted head on allowed ids
    zfull = o.full_biased_logits(full[-1])
    zr = o.restricted_logits(full[-1])
    np.testing.assert_allclose(zfull[cfg.sem_begin:cfg.sem_begin + cfg.n_sem], zr[:-1], rtol=1e-5, atol=1e-6)
    assert abs(zfull[cfg.im_end_id] - zr[-1]) < 1e-5


def test_fast_incremental_equals_full_recompute(tiny_oracle):
    o = tiny_oracle
    rng = np.random.default_rng(8)
    h = om.rmsnorm(rng.standard_normal(TINY.dim).astype(np.float32), np.ones(TINY.dim, np.float32), 1e-6)
    forced = np.array([300, 5, 77, 127], np.int32)
    u = np.full(TINY.n_codebooks + 1, 0.5, np.float32)
    codes, logits, _ = o.fast_ar(h, int(forced[0]), u, Sampling(), forced=forced)
    assert list(codes) == list(forced)
    full = o.fast_full_recompute(h, forced)
    np.testing.assert_allclose(logits, full, rtol=1e-4, atol=1e-5)


@pytest.mark.parametrize("n", [1, 2, 64, 300])
def test_one_layer_prefill_route_equals_prefill(n):
    """With one slow layer, the short prefill route (K/V of the prompt rows
    from their own inputs, the whole block for the last row only) leaves the
    same cache and state as the plain prefill, with either cache precision,
    and the next frame matches."""
    cfg = dataclasses.replace(TINY, n_layer=1)
    bits = g.make_weights(cfg, seed=0)
    prompt = g.make_prompt(cfg, n, seed=40 + n)
    for kv_bf16 in (True, False):
        o = oracle.DualAROracle(cfg, bits, max_pos=512, slow_kv_bf16=kv_bf16)
        a = o.prefill(prompt)
        b = o.prefill_one_layer(prompt, chunk=48)
        assert a.pos == b.pos == n
        for x, y in zip(a.kv[0], b.kv[0]):
            assert x.shape == y.shape
            np.testing.assert_allclose(x, y, rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(b.h_last, a.h_last, rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(b.z_last, a.z_last, rtol=1e-5, atol=1e-5)
        f = g.make_forced_codes(1, 1, cfg, seed=41)[0, 0]
        u = g.make_uniforms(1, 1, cfg, seed=42)[0, 0]
        ra = o.decode_frame(a, u, Sampling(allow_eos=False), forced=f)
        rb = o.decode_frame(b, u, Sampling(allow_eos=False), forced=f)
        np.testing.assert_allclose(rb.fast_logits, ra.fast_logits, rtol=1e-4, atol=1e-4)
        np.testing.assert_allclose(b.z_last, a.z_last, rtol=1e-4, atol=1e-4)


def _rne_8bit(x: np.ndarray) -> np.ndarray:
    """Round to 8 significant bits, ties to even, via frexp (normal numbers)."""
    m, e = np.frexp(np.asarray(x, np.float64))
    return (np.rint(m * 256.0) / 256.0 * np.exp2(e)).astype(np.float32)


def test_slow_kv_cache_holds_bf16_values(tiny_oracle):
    """The slow cache stores K (after QK-norm and RoPE) and V rounded to bf16;
    the first prompt position's K and V, recomputed here in fp32 from the
    weights, round (ties to even) to exactly what the cache holds.  The fast
    AR's per-frame cache is not rounded."""
    o = tiny_oracle
    cfg = TINY
    prompt = g.make_prompt(cfg, 9, seed=31)
    seq = o.prefill(prompt)
    for k, v in seq.kv:
        for t in (k, v):
            assert not np.any(t.view(np.uint32) & np.uint32(0xFFFF))
    lw = o.w.slow[0]
    # the same product as the prefill's (all prompt rows at once), so the fp32
    # values are bit-identical before rounding
    u = om.rmsnorm(o.w.tok_emb[prompt], lw.attn_norm, cfg.norm_eps)
    qkv = (u @ lw.wqkv.T)[0]
    k0 = qkv[cfg.q_dim:cfg.q_dim + cfg.kv_dim].reshape(cfg.n_kv_head, cfg.head_dim)
    v0 = qkv[cfg.q_dim + cfg.kv_dim:].reshape(cfg.n_kv_head, cfg.head_dim)
    k0 = om.rmsnorm(k0, lw.k_norm, cfg.norm_eps)    # position 0: RoPE is the identity
    np.testing.assert_array_equal(seq.kv[0][0][0], _rne_8bit(k0))
    np.testing.assert_array_equal(seq.kv[0][1][0], _rne_8bit(v0))
    kv = om.empty_kv(cfg, cfg.fast_n_layer)
    o.fast_forward(np.ones(cfg.dim, np.float32), 0, kv)
    assert np.any(kv[0][0].view(np.uint32) & np.uint32(0xFFFF))


def test_fast_kv_overwritten_each_frame(tiny_oracle):
    """The fast AR starts every frame from an empty num_codebooks-long cache:
    the same slow state and codes give the same logits whatever ran before."""
    o = tiny_oracle
    h = np.ones(TINY.dim, np.float32)
    f = np.array([3, 4, 5, 6], np.int32)
    u = np.full(5, 0.3, np.float32)
    a = o.fast_ar(h, 3, u, Sampling(), forced=f)[1]
    o.fast_ar(2 * h, 9, u, Sampling(), forced=np.array([9, 1, 2, 3], np.int32))
    b = o.fast_ar(h, 3, u, Sampling(), forced=f)[1]
    np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------- fusion --

class _FusionStub:
    pass


def _fusion_oracle(cfg, tok_emb, fusion):
    o = object.__new__(om.DualAROracle)
    o.cfg = cfg
    o.w = _FusionStub()
    o.w.tok_emb = tok_emb
    o.w.fusion = fusion
    return o


def test_fusion_unit_rows_closed_form():
    for cfg in (TINY, S2PRO):
        d = 8
        o = _fusion_oracle(cfg, np.ones((cfg.vocab, d), np.float32), np.ones((cfg.fusion_rows, d), np.float32))
        codes = np.zeros(cfg.n_codebooks, np.int32)
        x = o.fuse(codes)
        np.testing.assert_allclose(x, math.sqrt(cfg.n_codebooks + 1), rtol=1e-6)
    # full size: eleven unit rows scaled by 1/sqrt(11)
    assert abs(math.sqrt(11) - x[0]) < 1e-5


def test_fusion_gathers_the_right_rows():
    cfg = TINY
    rng = np.random.default_rng(9)
    # one-hot rows: tok_emb row r has a 1 at column r, fusion row r at V + r
    width = cfg.vocab + cfg.fusion_rows
    tok = np.zeros((cfg.vocab, width), np.float32)
    tok[np.arange(cfg.vocab), np.arange(cfg.vocab)] = 1
    fus = np.zeros((cfg.fusion_rows, width), np.float32)
    fus[np.arange(cfg.fusion_rows), cfg.vocab + np.arange(cfg.fusion_rows)] = 1
    o = _fusion_oracle(cfg, tok, fus)
    for _ in range(5):
        codes = np.array([rng.integers(cfg.n_sem)] + list(rng.integers(cfg.fast_vocab, size=3)), np.int32)
        x = o.fuse(codes) * math.sqrt(cfg.n_codebooks + 1)
        hot = set(np.flatnonzero(np.abs(x) > 0.5).tolist())
        expect = {cfg.sem_begin + codes[0], cfg.vocab + codes[0]} | {
            cfg.vocab + [0, 512, 640, 768][k] + codes[k] for k in range(1, 4)}
        assert hot == expect


# ------------------------------------------------------------------ bias --

def test_bias_keeps_exactly_semantic_and_im_end():
    f = facts()
    o = object.__new__(om.DualAROracle)
    o.cfg = S2PRO
    o.w = _FusionStub()
    o.w.tok_emb = np.ones((S2PRO.vocab, 1), np.float32)
    z = o.full_biased_logits(np.ones(1, np.float32))
    finite = np.flatnonzero(np.isfinite(z))
    assert finite.size == f["allowed_q0_candidates"]
    assert set(finite.tolist()) == set(range(f["semantic_first_id"], f["semantic_last_id"] + 1)) | {S2PRO.im_end_id}


# --------------------------------------------------------------- sampler --

def brute_nucleus(p, ids, top_p):
    """Smallest set of candidates reaching top_p, preferring higher mass, then
    lower ids -- by enumeration of all subsets."""
    n = len(p)
    best = None
    for r in range(1, n + 1):
        for sub in itertools.combinations(range(n), r):
            m = sum(p[i] for i in sub)
            if m >= top_p - 1e-12:
                key = (-m, sorted(ids[i] for i in sub))
                if best is None or key < best[0]:
                    best = (key, sub)
        if best is not None:
            return set(best[1])
    return set(range(n))


@pytest.mark.parametrize("seed", range(6))
def test_top_p_distribution_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 9))
    z = rng.standard_normal(n) * 2
    ids = rng.permutation(100)[:n]
    T = float(rng.choice([0.5, 0.8, 1.0, 1.7]))
    top_p = float(rng.choice([0.3, 0.6, 0.8, 0.9, 1.0]))
    p = np.exp(z / T - np.max(z / T))
    p /= p.sum()
    kept = brute_nucleus(p, ids, top_p)
    zk = sum(p[i] for i in kept)
    m = 20000
    counts = np.zeros(n)
    for j in range(m):
        counts[sample_top_p(z, ids, T, top_p, (j + 0.5) / m).index] += 1
    for i in range(n):
        expect = p[i] / zk if i in kept else 0.0
        assert abs(counts[i] / m - expect) <= 1.5 / m


def test_top_p_temperature_two_candidates():
    a, T = 1.3, 0.7
    z = np.array([0.0, a])
    m = 40000
    hits = sum(sample_top_p(z, [0, 1], T, 1.0, (j + 0.5) / m).index == 1 for j in range(m))
    assert abs(hits / m - 1 / (1 + math.exp(-a / T))) < 1e-4


def test_top_p_one_is_plain_inverse_cdf():
    rng = np.random.default_rng(11)
    z = rng.standard_normal(6)
    p = np.exp(z - z.max())
    p /= p.sum()
    order = sorted(range(6), key=lambda i: -p[i])
    for u in np.linspace(0.001, 0.999, 57):
        c = 0.0
        for i in order:
            c += p[i]
            if c > u:
                break
        assert sample_top_p(z, np.arange(6), 1.0, 1.0, u).index == i


def test_greedy_and_low_temperature_limit():
    z = np.array([0.1, 2.0, -1.0, 2.0, 1.5])
    ids = np.array([10, 7, 3, 5, 1])
    assert sample_top_p(z, ids, 0.0, 0.8, 0.9).index == 3     # tie at 2.0 -> lowest id (5)
    z2 = np.array([0.1, 2.0, -1.0, 1.9, 1.5])
    for u in (0.0, 0.5, 0.999):
        assert sample_top_p(z2, ids, 1e-3, 0.8, u).index == 1


def test_sampler_margins_reported():
    r = sample_top_p(np.array([0.0, 0.0]), [0, 1], 1.0, 1.0, 0.5)
    assert r.cdf_margin < 1e-12           # u*Z sits on the boundary 0.5


# ------------------------------------------------------------------- RAS --

def _q0(history, normal_target, ras_win=10, allow_eos=True):
    """Logits that make the normal draw (T=0) pick normal_target; the RAS
    draw (T=1, top-p 0.9) with u=0 picks the top candidate too, so make the
    RAS draw land elsewhere with u close to 1."""
    cfg = TINY
    z = np.zeros(cfg.n_sem + 1)
    z[normal_target] = 5.0
    smp = Sampling(temperature=0.0, top_p=0.8, ras_win=ras_win, allow_eos=allow_eos)
    return sample_q0(cfg, z, smp, history, 0.5, 0.999)


def test_ras_cases():
    # repeat inside the window -> resample (the RAS draw differs from 7)
    n, r, c = _q0([1, 2, 7], 7)
    assert n.index == 7 and c == r.index and c != 7
    # repeat only outside the last 10 frames -> keep
    n, r, c = _q0([7] + list(range(100, 110)), 7)
    assert c == 7
    # window shorter than 10 frames so far
    n, r, c = _q0([7], 7)
    assert c != 7
    # no repeat
    n, r, c = _q0([1, 2, 3], 7)
    assert c == 7
    # window 0 disables RAS
    n, r, c = _q0([7], 7, ras_win=0)
    assert c == 7
    # <|im_end|> never triggers the resample
    n, r, c = _q0([TINY.n_sem], TINY.n_sem)
    assert c == TINY.n_sem
    # allow_eos=False removes <|im_end|> from the candidates
    n, r, c = _q0([], TINY.n_sem, allow_eos=False)
    assert c != TINY.n_sem


def test_eos_frame_finishes_sequence(tiny_oracle):
    o = tiny_oracle
    seq = o.prefill(g.make_prompt(TINY, 8, seed=12))
    seq.z_last = np.full(TINY.n_sem + 1, -5.0, np.float32)
    seq.z_last[TINY.n_sem] = 50.0
    r = o.decode_frame(seq, np.full(5, 0.5, np.float32), Sampling())
    assert r.status == 1 and np.all(r.codes == -1) and seq.finished


# ----------------------------------------------------------------- pages --

def test_page_oracle_lowest_free_first():
    p = oracle.PageOracle(8, 4)
    p.append(0, 5)          # positions 0..4 -> pages 0, 1
    p.append(1, 1)          # page 2
    p.append(0, 4)          # positions 5..8 -> page 3 at position 8
    assert p.table == {0: [0, 1, 3], 1: [2]}
    p.release(0)
    p.append(2, 9)          # pages 0, 1, 3 again, lowest first
    assert p.table[2] == [0, 1, 3]
    with pytest.raises(MemoryError):
        p.append(3, 4 * 5)


def test_page_oracle_shared_prefix():
    p = oracle.PageOracle(8, 4)
    p.append(0, 6)          # positions 0..5 -> pages 0, 1
    p.share(0, 1, 5)        # page 0 by reference, the partly filled page copied: lowest free = 2
    assert p.table[1] == [0, 2] and p.length[1] == 5
    p.append(1, 4)          # positions 5..7 stay in page 2; position 8 -> page 3
    assert p.table[1] == [0, 2, 3]
    p.release(0)            # page 0 is still held by slot 1; page 1 returns
    p.append(2, 1)
    assert p.table[2] == [1]
    p.share(1, 3, 8)        # whole pages only: no copy
    assert p.table[3] == [0, 2]
    p.release(1)            # pages 0 and 2 still held by slot 3; page 3 returns
    p.append(4, 1)
    assert p.table[4] == [3]
    p.release(3)
    p.append(5, 9)          # pages 0, 2 and then the lowest free (4)
    assert p.table[5] == [0, 2, 4]
    with pytest.raises(ValueError):
        p.share(5, 2, 3)    # busy destination
    with pytest.raises(ValueError):
        p.share(5, 6, 10)   # longer than the source


# ------------------------------------------------------ planted mistakes --

def _expect_pin_failure(monkeypatch, target, name, bad, pin, *args):
    monkeypatch.setattr(target, name, bad)
    with pytest.raises(AssertionError):
        pin(*args)
    monkeypatch.undo()


def test_planted_rope_sign_error_is_caught(monkeypatch):
    orig = om.apply_rope

    def bad(x, pos, cos, sin):
        return orig(x, pos, cos, -sin)
    _expect_pin_failure(monkeypatch, om, "apply_rope", bad, test_rope_pair_layout_and_angle)


def test_planted_gqa_mapping_error_is_caught(monkeypatch):
    def bad(q, k, v, n_rep, causal_offset=None):
        kk = np.tile(k, (1, n_rep, 1))        # head h -> kv head h % Hkv
        vv = np.tile(v, (1, n_rep, 1))
        return om.gqa_attention.__wrapped__(q, kk, vv, 1, causal_offset) if hasattr(
            om.gqa_attention, "__wrapped__") else _plain_attention(q, kk, vv, causal_offset)
    _expect_pin_failure(monkeypatch, om, "gqa_attention", bad,
                        test_attention_matches_brute_force, 1, 5, 4, 2, 4)


def _plain_attention(q, k, v, off):
    s = np.einsum("qhd,khd->hqk", q, k) / math.sqrt(q.shape[-1])
    tq, tk = q.shape[0], k.shape[0]
    allowed = np.arange(tk)[None, :] <= (off + np.arange(tq))[:, None]
    s = np.where(allowed[None], s, -np.inf)
    p = np.exp(s - s.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    return np.einsum("hqk,khd->qhd", p, v).astype(np.float32)


def test_planted_causal_off_by_one_is_caught(monkeypatch):
    orig = om.gqa_attention

    def bad(q, k, v, n_rep, causal_offset=None):
        return orig(q, k, v, n_rep, None if causal_offset is None else causal_offset + 1)
    _expect_pin_failure(monkeypatch, om, "gqa_attention", bad,
                        test_attention_matches_brute_force, 3, 7, 4, 1, 3)


def test_planted_fusion_scale_error_is_caught(monkeypatch):
    orig = om.DualAROracle.fuse

    def bad(self, codes):
        return orig(self, codes) * math.sqrt(self.cfg.n_codebooks + 1) / math.sqrt(self.cfg.n_codebooks)
    _expect_pin_failure(monkeypatch, om.DualAROracle, "fuse", bad, test_fusion_unit_rows_closed_form)


_BLOCK_PINS = (test_block_single_position_closed_form, test_block_qk_norm_is_per_head_before_the_cache,
               test_block_two_positions_attention_weights)


def _expect_block_pins_fail(monkeypatch, bad):
    """A mistaken block must fail at least one of the block pins."""
    monkeypatch.setattr(om, "block", bad)
    failed = 0
    for pin in _BLOCK_PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    monkeypatch.undo()
    assert failed, "no block pin caught the planted mistake"


def _with(w, **kw):
    return dataclasses.replace(w, **kw)


def _qkv_rows(cfg, order):
    """Row permutation of wqkv that makes a correct block read it in another
    layout: "kv" swaps the k and v row blocks; "grouped" reads each KV group
    as [its query heads, its k, its v] in turn."""
    q, kv = cfg.q_dim, cfg.kv_dim
    if order == "kv":
        return list(range(q)) + list(range(q + kv, q + 2 * kv)) + list(range(q, q + kv))
    g = cfg.n_head // cfg.n_kv_head
    hd = cfg.head_dim
    per = (g + 2) * hd
    qs, ks, vs = [], [], []
    for j in range(cfg.n_kv_head):
        base = j * per
        qs += list(range(base, base + g * hd))
        ks += list(range(base + g * hd, base + (g + 1) * hd))
        vs += list(range(base + (g + 1) * hd, base + per))
    return qs + ks + vs


def test_planted_block_gate_up_swap_is_caught(monkeypatch):
    orig = om.block

    def bad(cfg, w, *a, **k):          # SiLU(up) * gate
        return orig(cfg, _with(w, w_gate=w.w_up, w_up=w.w_gate), *a, **k)
    _expect_block_pins_fail(monkeypatch, bad)


def test_planted_block_ffn_reads_pre_attention_state_is_caught(monkeypatch):
    orig = om.block

    def bad(cfg, w, h, *a, **k):       # h + attn(h) + FFN(RMSNorm(h))
        ha, kc, vc = orig(cfg, _with(w, w_gate=np.zeros_like(w.w_gate)), h, *a, **k)
        hf, _, _ = orig(cfg, _with(w, wo=np.zeros_like(w.wo)), h, *a, **k)
        return ha + hf - h, kc, vc
    _expect_block_pins_fail(monkeypatch, bad)


def test_planted_block_ffn_norm_gain_mixup_is_caught(monkeypatch):
    orig = om.block

    def bad(cfg, w, *a, **k):          # the FFN normalised with the attention gain
        return orig(cfg, _with(w, ffn_norm=w.attn_norm), *a, **k)
    _expect_block_pins_fail(monkeypatch, bad)


@pytest.mark.parametrize("order", ["kv", "grouped"])
def test_planted_block_qkv_row_order_is_caught(monkeypatch, order):
    orig = om.block

    def bad(cfg, w, *a, **k):
        return orig(cfg, _with(w, wqkv=w.wqkv[_qkv_rows(cfg, order)]), *a, **k)
    _expect_block_pins_fail(monkeypatch, bad)


def test_planted_block_missing_attention_scale_is_caught(monkeypatch):
    orig_attn = om.gqa_attention

    def bad(q, k, v, n_rep, causal_offset=None):
        return orig_attn(q * np.float32(math.sqrt(q.shape[-1])), k, v, n_rep, causal_offset)
    monkeypatch.setattr(om, "gqa_attention", bad)
    with pytest.raises(AssertionError):
        test_block_two_positions_attention_weights()
    monkeypatch.undo()


def test_planted_top_p_off_by_one_is_caught(monkeypatch):
    import oracle.sampler as osm
    orig = osm.sample_top_p

    def bad(z, ids, temperature, top_p, u):
        # keeps one candidate too many
        r = orig(z, ids, temperature, min(1.0, top_p + 0.15), u)
        return r
    monkeypatch.setattr(osm, "sample_top_p", bad)
    with pytest.raises(AssertionError):
        for s in range(6):
            _tp_check(s, osm.sample_top_p)


def _tp_check(seed, fn):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 9))
    z = rng.standard_normal(n) * 2
    ids = rng.permutation(100)[:n]
    T = float(rng.choice([0.5, 0.8, 1.0, 1.7]))
    top_p = float(rng.choice([0.3, 0.6, 0.8, 0.9, 1.0]))
    p = np.exp(z / T - np.max(z / T))
    p /= p.sum()
    kept = brute_nucleus(p, ids, top_p)
    zk = sum(p[i] for i in kept)
    m = 4000
    counts = np.zeros(n)
    for j in range(m):
        counts[fn(z, ids, T, top_p, (j + 0.5) / m).index] += 1
    for i in range(n):
        expect = p[i] / zk if i in kept else 0.0
        assert abs(counts[i] / m - expect) <= 1.5 / m


def test_page_oracle_under_replacement_churn():
    """The batch-128 replacement workload's page traffic (124 contexts of
    2-4K that finish at seeded frames and are replaced from a queue, 4
    resident contexts of 16K), 64 steps: the page oracle agrees step by step
    with a naive allocator (a sorted free list, lowest page first), every page
    is held by at most one slot, and releasing everything frees the pool."""
    wl = g.make_replacement_workload(128, 4, 256, seed=4)
    pt = 64
    need = sum(-(-int(c + 64) // pt) for c in wl["ctx"]) + 512
    po = oracle.PageOracle(need, pt)
    naive_free = list(range(need))
    naive = {}

    def naive_append(slot, old_len, n):
        tab = naive.setdefault(slot, [])
        for p in range(old_len, old_len + n):
            if p % pt == 0:
                tab.append(naive_free.pop(0))

    def naive_release(slot):
        naive_free.extend(naive.pop(slot))
        naive_free.sort()

    length, finish = {}, {}
    for s in range(128):
        po.append(s, int(wl["ctx"][s]))
        naive_append(s, 0, int(wl["ctx"][s]))
        length[s], finish[s] = int(wl["ctx"][s]), int(wl["finish"][s])
    q = 0
    for step in range(1, 65):
        for s in range(128):
            po.append(s, 1)
            naive_append(s, length[s], 1)
            length[s] += 1
        for s in range(128):
            if finish[s] == step:
                po.release(s)
                naive_release(s)
                n = int(wl["queue_ctx"][q])
                po.append(s, n)
                naive_append(s, 0, n)
                length[s], finish[s] = n, step + int(wl["queue_finish"][q])
                q += 1
        assert po.table == naive
        held = [pg for tab in po.table.values() for pg in tab]
        assert len(held) == len(set(held))
        assert sorted(po.free) == naive_free
    assert q > 100                                  # most short sequences were replaced, some twice
    for s in list(po.table):
        po.release(s)
    assert sorted(po.free) == list(range(need)) and not any(po.holders)
