"""CPU oracle of the Dual-AR per-frame decode (NumPy, fp32 over bf16 weights).

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the CPU-baseline
leg of the benchmark may import this module.  It shares no code with the
CUDA library; its one common dependency is the seeded input generator.

Pages cited (title, then section):
  [P1] "How the Dual-Autoregressive Architecture Works in Fish Speech S2:
       A Deep Dive"
  [P2] "Fish Audio S2: a Qwen3-4B on the time axis, four layers on the
       codebook axis, and tags that are only text"

Readings taken where the pages are silent (each one is also listed, with
its reason, in the design notes):
  * the slow hidden state that feeds fast pass 0 is the final-RMSNorm output
    (the vector the head multiplies), with no further norm
    ([P1] DualARModelArgs: norm_fastlayer_input=False);
  * every RMSNorm uses eps = 1e-6 (the pages name norm_eps, not its value);
  * QK-norm is a per-head RMSNorm over head_dim applied before RoPE, slow AR
    only ([P2] "The slow AR is Qwen3-4B": qk-norm; the fast AR lacks it);
  * RoPE rotates interleaved pairs (2i, 2i+1) by pos * base^(-2i/head_dim)
    with cos/sin computed in float64 and rounded once to bf16 ([P2]
    "Streaming: whose numbers": bf16 tables; base 1e6);
  * GQA maps query head h to KV head h // (n_head / n_kv_head);
  * the fast AR uses the same RoPE table, position = codebook index;
  * q0 indexes the fast embedding as min(q0, fast_vocab - 1) (a no-op at
    full size, where fast_vocab = n_sem);
  * after prefill the sequence holds the final hidden state and restricted
    logits of its last prompt position; a frame samples q0 from them, runs
    the fast AR, fuses the codes and runs one slow position on the fused
    vector;
  * the slow AR's KV cache holds bf16 values: K (after QK-norm and RoPE) and
    V are rounded to bf16 (nearest even) when appended.  The pages do not say
    what precision the cache has: their fact table ([P2] "Two
    autoregressions") gives the checkpoint's parameters as BF16, and [P2]
    "Streaming: whose numbers" says the model runs on bf16 tables, which
    suggests, without stating it, a model served in bf16 throughout.  This is
    a departure from a pure "fp32 activations over bf16 weights" oracle, taken
    for the cache only; slow_kv_bf16=False gives that pure form, and the
    full-size parity test reports how far the two lie apart.  The fast AR's
    per-frame cache stays float32.

Precision: every activation is float32; weights are bf16 widened exactly to
float32; the slow KV cache holds bf16 values (widened to float32), the fast
KV cache is float32; sampling probabilities are float64.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from dualar_inputs.config import DualARConfig
from dualar_inputs.generators import bf16_bits_to_f32, f32_to_bf16_bits

from .sampler import SampleResult, sample_q0, sample_top_p


# --------------------------------------------------------------------------
# Building blocks
# --------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * w.

    [P1] "Fast Transformer: The Codebook Decoder": RMSNorm(dim, eps=norm_eps);
    [P1] table "What Is the Dual-Autoregressive Architecture?": RMSNorm in
    the slow transformer."""
    x = np.asarray(x, dtype=np.float32)
    ms = np.mean(np.square(x, dtype=np.float32), axis=-1, keepdims=True, dtype=np.float32)
    return (x * (np.float32(1.0) / np.sqrt(ms + np.float32(eps)))) * w


def rope_table(max_pos: int, head_dim: int, base: float) -> tuple[np.ndarray, np.ndarray]:
    """cos/sin tables [max_pos, head_dim/2], computed in float64, rounded
    once to bf16 and returned widened to float32.

    [P2] "Streaming: whose numbers": the model was trained with bf16 RoPE
    tables and the fp32 table is the wrong one; [P2] "The slow AR is
    Qwen3-4B": rope_base 1,000,000."""
    half = head_dim // 2
    inv_freq = base ** (-(2.0 * np.arange(half, dtype=np.float64)) / head_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    cos = bf16_bits_to_f32(f32_to_bf16_bits(np.cos(ang).astype(np.float32)))
    sin = bf16_bits_to_f32(f32_to_bf16_bits(np.sin(ang).astype(np.float32)))
    return cos, sin


def apply_rope(x: np.ndarray, pos: np.ndarray | int, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate the interleaved pairs (x[2i], x[2i+1]) of the last axis.

    x: [..., heads, head_dim]; pos: int or int array broadcastable to
    x.shape[:-2]."""
    x = np.asarray(x, dtype=np.float32)
    c = cos[pos][..., None, :]
    s = sin[pos][..., None, :]
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x1 * c + x0 * s
    return out


def silu(x: np.ndarray) -> np.ndarray:
    return x / (np.float32(1.0) + np.exp(-x))


def gqa_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, n_rep: int,
                  causal_offset: int | None = None) -> np.ndarray:
    """softmax(q k^T / sqrt(hd)) v with grouped KV heads.

    q: [Tq, Hq, hd]; k, v: [Tk, Hkv, hd]; query head h reads KV head
    h // n_rep.  With causal_offset = c, query row i sees keys 0..c+i.
    [P2] fact table: 32 query heads over 8 KV heads."""
    tq, hq, hd = q.shape
    kr = np.repeat(k, n_rep, axis=1)          # [Tk, Hq, hd]
    vr = np.repeat(v, n_rep, axis=1)
    s = np.einsum("qhd,khd->hqk", q, kr, dtype=np.float32) * np.float32(1.0 / math.sqrt(hd))
    if causal_offset is not None:
        tk = k.shape[0]
        allowed = np.arange(tk)[None, :] <= (causal_offset + np.arange(tq))[:, None]
        s = np.where(allowed[None], s, np.float32(-np.inf))
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    return np.einsum("hqk,khd->qhd", p, vr, dtype=np.float32)


# --------------------------------------------------------------------------
# Weights
# --------------------------------------------------------------------------

@dataclasses.dataclass
class LayerW:
    attn_norm: np.ndarray
    wqkv: np.ndarray
    q_norm: np.ndarray | None
    k_norm: np.ndarray | None
    wo: np.ndarray
    ffn_norm: np.ndarray
    w_gate: np.ndarray
    w_up: np.ndarray
    w_down: np.ndarray


class Weights:
    """float32 views of the bf16 weights, keyed like the generator."""

    def __init__(self, cfg: DualARConfig, bits: dict[str, np.ndarray]):
        f = {k: bf16_bits_to_f32(v) for k, v in bits.items()}
        self.tok_emb = f["tok_emb"]
        self.final_norm = f["final_norm"]
        self.fast_emb = f["fast_emb"]
        self.fast_norm = f["fast_norm"]
        self.fast_out = f["fast_out"]
        self.fusion = f["fusion"]

        def layer(p: str, qk: bool) -> LayerW:
            return LayerW(f[p + ".attn_norm"], f[p + ".wqkv"],
                          f[p + ".q_norm"] if qk else None,
                          f[p + ".k_norm"] if qk else None,
                          f[p + ".wo"], f[p + ".ffn_norm"], f[p + ".w_gate"],
                          f[p + ".w_up"], f[p + ".w_down"])

        self.slow = [layer(f"slow.{i}", cfg.slow_qk_norm) for i in range(cfg.n_layer)]
        self.fast = [layer(f"fast.{i}", cfg.fast_qk_norm) for i in range(cfg.fast_n_layer)]


# --------------------------------------------------------------------------
# One transformer block over Tq new rows, with a contiguous KV cache
# --------------------------------------------------------------------------

def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 values rounded to the nearest bf16 (ties to even), as float32."""
    return bf16_bits_to_f32(f32_to_bf16_bits(np.asarray(x, np.float32)))


def block(cfg: DualARConfig, w: LayerW, h: np.ndarray, pos0: int,
          kcache: np.ndarray, vcache: np.ndarray, cos, sin,
          qk_norm: bool, kv_bf16: bool = False) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Pre-norm block: h += Wo attn(RoPE(QKnorm(q,k)), v); h += down(SiLU(gate) * up).

    h: [Tq, D] rows at positions pos0..pos0+Tq-1; kcache/vcache: [Tk, Hkv, hd]
    holding positions 0..pos0-1.  With kv_bf16 the new K and V rows are
    rounded to bf16 before they join the cache (and the attention reads them
    from it).  Returns (h_out, kcache', vcache').
    [P1] "Fast Transformer": TransformerBlock; [P2] "The slow AR is
    Qwen3-4B" (Qwen3 layer: GQA, SwiGLU FFN 9728, qk-norm)."""
    hd, hq, hkv = cfg.head_dim, cfg.n_head, cfg.n_kv_head
    tq = h.shape[0]
    u = rmsnorm(h, w.attn_norm, cfg.norm_eps)
    qkv = u @ w.wqkv.T                                    # [Tq, qkv_dim]
    q = qkv[:, :cfg.q_dim].reshape(tq, hq, hd)
    k = qkv[:, cfg.q_dim:cfg.q_dim + cfg.kv_dim].reshape(tq, hkv, hd)
    v = qkv[:, cfg.q_dim + cfg.kv_dim:].reshape(tq, hkv, hd)
    if qk_norm:
        q = rmsnorm(q, w.q_norm, cfg.norm_eps)
        k = rmsnorm(k, w.k_norm, cfg.norm_eps)
    pos = np.arange(pos0, pos0 + tq)
    q = apply_rope(q, pos, cos, sin)
    k = apply_rope(k, pos, cos, sin)
    if kv_bf16:
        k, v = bf16_round(k), bf16_round(v)
    kc = np.concatenate([kcache, k.astype(np.float32)], axis=0)
    vc = np.concatenate([vcache, v.astype(np.float32)], axis=0)
    a = gqa_attention(q, kc, vc, hq // hkv, causal_offset=pos0)
    h = h + a.reshape(tq, cfg.q_dim) @ w.wo.T
    u = rmsnorm(h, w.ffn_norm, cfg.norm_eps)
    g = u @ w.w_gate.T
    up = u @ w.w_up.T
    h = h + (silu(g) * up) @ w.w_down.T
    return h.astype(np.float32), kc, vc


def empty_kv(cfg: DualARConfig, n_layers: int) -> list[list[np.ndarray]]:
    z = np.zeros((0, cfg.n_kv_head, cfg.head_dim), np.float32)
    return [[z, z] for _ in range(n_layers)]


# --------------------------------------------------------------------------
# The oracle
# --------------------------------------------------------------------------

@dataclasses.dataclass
class SeqState:
    """Per-sequence decode state."""
    kv: list                      # slow KV: per layer [K, V], each [T, Hkv, hd]
    pos: int = 0                  # next slow position
    h_last: np.ndarray | None = None   # final-normed hidden of the last position [D]
    z_last: np.ndarray | None = None   # restricted logits of the last position [S+1]
    history: list = dataclasses.field(default_factory=list)  # committed q0 (semantic idx)
    finished: bool = False


@dataclasses.dataclass
class Sampling:
    temperature: float = 0.8
    top_p: float = 0.8
    ras_win: int = 10
    allow_eos: bool = True
    ras_temperature: float = 1.0
    ras_top_p: float = 0.9


@dataclasses.dataclass
class FrameResult:
    codes: np.ndarray             # int32 [N]; q0 as semantic index; -1 if finished
    status: int                   # 0 ok, 1 end of sequence (q0 = <|im_end|>)
    slow_logits: np.ndarray       # restricted logits q0 was drawn from [S+1]
    fast_logits: np.ndarray       # [N-1, fast_vocab]
    draws: list                   # SampleResult per draw (q0 then q1..q(N-1))
    x_next: np.ndarray | None     # fused slow input of this frame [D]


class DualAROracle:
    def __init__(self, cfg: DualARConfig, weight_bits: dict[str, np.ndarray],
                 max_pos: int = 20_000, w4a16_keys: list[str] | None = None,
                 slow_kv_bf16: bool = True):
        """slow_kv_bf16: whether the slow AR's cache holds bf16 values (the
        reading this oracle takes); False keeps it in float32, so a test can
        show how far that reading moves the results.
        w4a16_keys: projections (generator keys such as "slow.0.wqkv") that
        the model reads through the 4-bit rule of oracle.w4a16 ([P3]
        "s2-pro-w4a16-late12attn", opening line): each such matrix is
        replaced by its quantised-then-dequantised float32 values."""
        self.cfg = cfg
        self.slow_kv_bf16 = slow_kv_bf16
        self.w = Weights(cfg, weight_bits)
        if w4a16_keys:
            from .w4a16 import dequantize, quantize
            for key in w4a16_keys:
                stack, i, name = key.split(".")
                layer = (self.w.slow if stack == "slow" else self.w.fast)[int(i)]
                setattr(layer, name, dequantize(*quantize(weight_bits[key])))
        self.cos, self.sin = rope_table(max(max_pos, cfg.n_codebooks), cfg.head_dim, cfg.rope_base)
        self.rep = cfg.n_head // cfg.n_kv_head

    # ---- slow AR ---------------------------------------------------------
    def slow_rows(self, seq: SeqState, x: np.ndarray) -> np.ndarray:
        """Run the slow stack on rows x [T, D] at positions seq.pos.. and
        append their KV; returns the final-normed hidden rows [T, D]."""
        cfg = self.cfg
        h = np.asarray(x, np.float32)
        for i, lw in enumerate(self.w.slow):
            k, v = seq.kv[i]
            h, k, v = block(cfg, lw, h, seq.pos, k, v, self.cos, self.sin, cfg.slow_qk_norm,
                            kv_bf16=self.slow_kv_bf16)
            seq.kv[i] = [k, v]
        seq.pos += h.shape[0]
        return rmsnorm(h, self.w.final_norm, cfg.norm_eps)

    def restricted_logits(self, hn: np.ndarray) -> np.ndarray:
        """Logits of the semantic block and <|im_end|> only, from the tied
        embedding: [..., S+1] with the im_end logit last.

        [P2] "Two autoregressions": the bias is -inf everywhere except the
        semantic ids and <|im_end|>; [P2] "The slow AR is Qwen3-4B": the head
        is tied to the embedding."""
        cfg = self.cfg
        rows = self.w.tok_emb[cfg.sem_begin:cfg.sem_begin + cfg.n_sem]
        z = hn @ rows.T
        ze = hn @ self.w.tok_emb[cfg.im_end_id]
        return np.concatenate([z, np.asarray(ze, np.float32)[..., None]], axis=-1).astype(np.float32)

    def full_biased_logits(self, hn: np.ndarray) -> np.ndarray:
        """Full-vocabulary logits plus the semantic bias (-inf elsewhere),
        the way the reference code computes them ([P2] "The slow AR is
        Qwen3-4B": logits over the whole vocabulary, then masking)."""
        cfg = self.cfg
        z = (hn @ self.w.tok_emb.T).astype(np.float32)
        bias = np.full(cfg.vocab, -np.inf, np.float32)
        bias[cfg.sem_begin:cfg.sem_begin + cfg.n_sem] = 0.0
        bias[cfg.im_end_id] = 0.0
        return z + bias

    def new_sequence(self) -> SeqState:
        return SeqState(kv=empty_kv(self.cfg, self.cfg.n_layer))

    def prefill(self, tokens: np.ndarray, seq: SeqState | None = None) -> SeqState:
        """Embed prompt ids (x = e_LM[tok], no fusion) and run the slow AR over
        them; keeps the last position's normed hidden and restricted logits."""
        seq = seq or self.new_sequence()
        x = self.w.tok_emb[np.asarray(tokens, np.int64)]
        hn = self.slow_rows(seq, x)
        seq.h_last = hn[-1].copy()
        seq.z_last = self.restricted_logits(hn[-1])
        return seq

    def prefill_one_layer(self, tokens: np.ndarray, chunk: int = 2048) -> SeqState:
        """prefill() of a slow stack with exactly one layer, by the short route.

        With one layer, the K and V that position t leaves in the cache are
        the layer's projections of its own input e_LM[tok_t] (RMSNorm, the k
        and v rows of wqkv, QK-norm on k, RoPE at t, the cache rounding): no
        other position enters them.  Only the last position's output is kept
        after a prefill, so positions 0..n-2 need their K and V and nothing
        else, and the last position runs the whole block over that cache.
        The result equals prefill() up to the order of float rounding (a
        test compares the two on a one-layer model); it costs a fifth of the
        projections and no attention over the prompt, which is what makes
        prompts of many thousands of tokens affordable on the host."""
        cfg = self.cfg
        assert cfg.n_layer == 1, "the short route holds for one slow layer only"
        lw = self.w.slow[0]
        tokens = np.asarray(tokens, np.int64)
        n = tokens.size
        hkv, hd = cfg.n_kv_head, cfg.head_dim
        wk = lw.wqkv[cfg.q_dim:cfg.q_dim + cfg.kv_dim]
        wv = lw.wqkv[cfg.q_dim + cfg.kv_dim:]
        ks, vs = [], []
        for c0 in range(0, n - 1, chunk):
            c1 = min(c0 + chunk, n - 1)
            u = rmsnorm(self.w.tok_emb[tokens[c0:c1]], lw.attn_norm, cfg.norm_eps)
            k = (u @ wk.T).reshape(c1 - c0, hkv, hd)
            v = (u @ wv.T).reshape(c1 - c0, hkv, hd)
            if cfg.slow_qk_norm:
                k = rmsnorm(k, lw.k_norm, cfg.norm_eps)
            k = apply_rope(k, np.arange(c0, c1), self.cos, self.sin)
            if self.slow_kv_bf16:
                k, v = bf16_round(k), bf16_round(v)
            ks.append(k.astype(np.float32))
            vs.append(v.astype(np.float32))
        seq = self.new_sequence()
        if ks:
            seq.kv[0] = [np.concatenate(ks), np.concatenate(vs)]
        seq.pos = n - 1
        hn = self.slow_rows(seq, self.w.tok_emb[tokens[-1:]])
        seq.h_last = hn[-1].copy()
        seq.z_last = self.restricted_logits(hn[-1])
        return seq

    # ---- fast AR ---------------------------------------------------------
    def fast_forward(self, x: np.ndarray, pos: int, kv: list) -> np.ndarray:
        """One fast pass: the fast layers on one row at codebook position pos."""
        cfg = self.cfg
        h = np.asarray(x, np.float32)[None, :]
        for i, lw in enumerate(self.w.fast):
            k, v = kv[i]
            h, k, v = block(cfg, lw, h, pos, k, v, self.cos, self.sin, cfg.fast_qk_norm)
            kv[i] = [k, v]
        return h[0]

    def fast_head(self, h: np.ndarray) -> np.ndarray:
        return (rmsnorm(h, self.w.fast_norm, self.cfg.norm_eps) @ self.w.fast_out.T).astype(np.float32)

    def fast_ar(self, h_slow: np.ndarray, q0: int, uniforms: np.ndarray, smp: Sampling,
                forced: np.ndarray | None = None):
        """N fast passes for one frame ([P2] "Two autoregressions", the
        decode_one_token_ar order): pass 0 puts the slow hidden state into a
        fresh num_codebooks-long cache at position 0; pass k >= 1 reads the
        embedding of code k-1 at position k and samples code k from the fast
        head, unmasked, with the frame's temperature and top-p."""
        cfg = self.cfg
        kv = empty_kv(cfg, cfg.fast_n_layer)
        self.fast_forward(h_slow, 0, kv)
        codes = [q0]
        logits = np.zeros((cfg.n_codebooks - 1, cfg.fast_vocab), np.float32)
        draws = []
        prev = min(q0, cfg.fast_vocab - 1)
        ids = np.arange(cfg.fast_vocab)
        for k in range(1, cfg.n_codebooks):
            h = self.fast_forward(self.w.fast_emb[prev], k, kv)
            z = self.fast_head(h)
            logits[k - 1] = z
            r = sample_top_p(z, ids, smp.temperature, smp.top_p, float(uniforms[k + 1]))
            draws.append(r)
            qk = int(forced[k]) if forced is not None else int(r.index)
            codes.append(qk)
            prev = qk
        return np.array(codes, np.int32), logits, draws

    # ---- fusion -----------------------------------------------------------
    def fuse(self, codes: np.ndarray) -> np.ndarray:
        """Multi-codebook fusion, [P2] "Two autoregressions", Eq. 1 with the
        code's 1/sqrt(N+1) scale: x = (e_LM[q0] + sum_k E^(k)[q_k]) / sqrt(N+1).
        e_LM[q0] is the semantic token's row of the slow embedding; E^(k) is
        codebook k's block of the fusion table."""
        cfg = self.cfg
        n = cfg.n_codebooks
        acc = self.w.tok_emb[cfg.sem_begin + int(codes[0])].astype(np.float64)
        for k in range(n):
            acc = acc + self.w.fusion[cfg.fusion_offset(k) + int(codes[k])]
        return (acc / math.sqrt(n + 1)).astype(np.float32)

    # ---- one frame ----------------------------------------------------------
    def decode_frame(self, seq: SeqState, uniforms: np.ndarray, smp: Sampling,
                     forced: np.ndarray | None = None) -> FrameResult:
        """q0 from the held restricted logits (with the repetition-aware
        resample), the fast AR, fusion, and one slow position on the fused
        vector.  uniforms: [N+1] = (u_q0, u_ras, u_q1 .. u_q(N-1)).
        With forced codes [N] the draws are still made (and returned) but
        the forced codes are committed."""
        cfg = self.cfg
        assert not seq.finished, "decode on a finished sequence"
        z = seq.z_last
        r0, rras, chosen = sample_q0(cfg, z, smp, seq.history, float(uniforms[0]), float(uniforms[1]))
        q0 = int(forced[0]) if forced is not None else chosen
        draws = [(r0, rras, chosen)]
        if q0 == cfg.n_sem:   # <|im_end|> (candidate index S)
            seq.finished = True
            return FrameResult(np.full(cfg.n_codebooks, -1, np.int32), 1, z,
                               np.zeros((cfg.n_codebooks - 1, cfg.fast_vocab), np.float32),
                               draws, None)
        seq.history.append(q0)
        codes, flog, fdraws = self.fast_ar(seq.h_last, q0, uniforms, smp, forced)
        draws += fdraws
        x = self.fuse(codes)
        hn = self.slow_rows(seq, x[None, :])[0]
        seq.h_last = hn
        seq.z_last = self.restricted_logits(hn)
        return FrameResult(codes, 0, z, flog, draws, x)

    # ---- reference recompute (training-style forward) ------------------------
    def slow_full_recompute(self, x_rows: np.ndarray) -> np.ndarray:
        """All positions at once with a causal mask and no incremental cache:
        returns the final-normed hidden rows.  Used to pin the incremental
        path ([P1] "Forward Pass: How the Two Stages Interact", Step 1)."""
        cfg = self.cfg
        h = np.asarray(x_rows, np.float32)
        kv = empty_kv(cfg, cfg.n_layer)
        for i, lw in enumerate(self.w.slow):
            h, _, _ = block(cfg, lw, h, 0, kv[i][0], kv[i][1], self.cos, self.sin, cfg.slow_qk_norm,
                            kv_bf16=self.slow_kv_bf16)
        return rmsnorm(h, self.w.final_norm, cfg.norm_eps)

    def fast_full_recompute(self, h_slow: np.ndarray, codes: np.ndarray) -> np.ndarray:
        """The fast AR over its whole codebook sequence in one causal pass,
        [slow hidden, emb(q0), emb(q1), ...] like the training forward of
        [P1] "Step 3: Fast Sub-Network Construction"; returns the fast-head
        logits of positions 1..N-1 [N-1, fast_vocab]."""
        cfg = self.cfg
        prev = [min(int(codes[0]), cfg.fast_vocab - 1)] + [int(c) for c in codes[1:cfg.n_codebooks - 1]]
        x = np.concatenate([np.asarray(h_slow, np.float32)[None, :], self.w.fast_emb[prev]], axis=0)
        kv = empty_kv(cfg, cfg.fast_n_layer)
        h = x
        for i, lw in enumerate(self.w.fast):
            h, _, _ = block(cfg, lw, h, 0, kv[i][0], kv[i][1], self.cos, self.sin, cfg.fast_qk_norm)
        return (rmsnorm(h[1:], self.w.fast_norm, cfg.norm_eps) @ self.w.fast_out.T).astype(np.float32)


__all__ = ["DualAROracle", "SeqState", "Sampling", "FrameResult", "SampleResult",
           "rmsnorm", "rope_table", "apply_rope", "gqa_attention", "silu", "block"]
