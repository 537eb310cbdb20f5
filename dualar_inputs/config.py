"""Model shapes and token-id layout of the Dual-AR decoder.

Shared by the CPU oracle and the CUDA path.  Holds shapes, ids and
parameter counts only; no part of the decode arithmetic lives here.

Sources (page titles, sections):
  * "Fish Audio S2: a Qwen3-4B on the time axis ..." -- fact table
    (checkpoint 4,561,852,416 params; slow AR 36 x 2560, 32 Q / 8 KV heads,
    FFN 9728, vocab 155,776; fast AR 4 layers at 2560 with 4,096-row
    embedding and head; fusion table 40,960 x 2560), section "The slow AR is
    Qwen3-4B" (head_dim 128, rope_base 1e6, qk-norm in the slow AR only,
    tied embeddings, 4,096 semantic ids at 151,678..155,773).
  * "How the Dual-Autoregressive Architecture Works in Fish Speech S2" --
    DualARModelArgs: fast fields fall back to the slow ones,
    norm_fastlayer_input=False.
"""
from __future__ import annotations

import dataclasses


@dataclasses.dataclass(frozen=True)
class DualARConfig:
    name: str
    dim: int            # model width D (slow and fast AR share it: no fast_project_in)
    n_layer: int        # slow-AR layers
    n_head: int         # query heads
    n_kv_head: int      # key/value heads (GQA)
    head_dim: int
    ffn: int            # SwiGLU intermediate size
    vocab: int          # slow-AR vocabulary (tied embedding / head rows)
    sem_begin: int      # first <|semantic:i|> id
    n_sem: int          # number of semantic ids S
    im_end_id: int      # <|im_end|> id (the one non-semantic id the bias keeps)
    fast_n_layer: int
    fast_vocab: int     # fast-AR codebook_size C_f (embedding and head rows)
    n_codebooks: int    # N: codebooks per frame (1 semantic + N-1 acoustic)
    slow_qk_norm: bool = True
    fast_qk_norm: bool = False
    rope_base: float = 1.0e6
    norm_eps: float = 1.0e-6
    page_tokens: int = 64

    # ---- derived shapes -------------------------------------------------
    @property
    def q_dim(self) -> int:
        return self.n_head * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_head * self.head_dim

    @property
    def qkv_dim(self) -> int:
        return self.q_dim + 2 * self.kv_dim

    @property
    def fusion_rows(self) -> int:
        """Rows of the fusion table: codebook 0 has n_sem rows, codebooks
        1..N-1 have fast_vocab rows each (40,960 = 10 x 4,096 at full size)."""
        return self.n_sem + (self.n_codebooks - 1) * self.fast_vocab

    def fusion_offset(self, k: int) -> int:
        """First fusion-table row of codebook k."""
        return 0 if k == 0 else self.n_sem + (k - 1) * self.fast_vocab

    @property
    def n_cand_q0(self) -> int:
        """Restricted head rows: the semantic block plus <|im_end|>."""
        return self.n_sem + 1

    # ---- parameter counts (shape check against the pages' figures) -----
    def layer_params(self, qk_norm: bool) -> int:
        d, hd = self.dim, self.head_dim
        n = d                                   # attention_norm
        n += self.qkv_dim * d                   # fused wqkv, no bias
        n += (2 * hd) if qk_norm else 0         # q_norm, k_norm
        n += d * self.q_dim                     # wo, no bias
        n += d                                  # ffn_norm
        n += 3 * self.ffn * d                   # w_gate, w_up, w_down
        return n

    def slow_params(self) -> int:
        return (self.n_layer * self.layer_params(self.slow_qk_norm)
                + self.vocab * self.dim + self.dim)   # tied emb/head + final norm

    def fast_params(self) -> int:
        return (self.fast_n_layer * self.layer_params(self.fast_qk_norm)
                + 2 * self.fast_vocab * self.dim + self.dim)  # emb + untied head + norm

    def fusion_params(self) -> int:
        return self.fusion_rows * self.dim

    def total_params(self) -> int:
        return self.slow_params() + self.fast_params() + self.fusion_params()

    def fast_pass_params(self) -> int:
        """Weights one fast pass reads with a head (layers + output head)."""
        return (self.fast_n_layer * self.layer_params(self.fast_qk_norm)
                + self.fast_vocab * self.dim)

    # ---- weight tensor inventory -----------------------------------------
    def weight_shapes(self) -> list[tuple[str, tuple[int, ...], str]]:
        """(name, shape, init kind) for every tensor, in a fixed order.

        init kind: "w" = matrix/embedding N(0, 0.02); "g" = norm gain
        1 + N(0, 0.02)."""
        d, hd = self.dim, self.head_dim
        out: list[tuple[str, tuple[int, ...], str]] = [
            ("tok_emb", (self.vocab, d), "w"),
            ("final_norm", (d,), "g"),
        ]

        def layer(prefix: str, qk: bool):
            items = [(f"{prefix}.attn_norm", (d,), "g"),
                     (f"{prefix}.wqkv", (self.qkv_dim, d), "w")]
            if qk:
                items += [(f"{prefix}.q_norm", (hd,), "g"),
                          (f"{prefix}.k_norm", (hd,), "g")]
            items += [(f"{prefix}.wo", (d, self.q_dim), "w"),
                      (f"{prefix}.ffn_norm", (d,), "g"),
                      (f"{prefix}.w_gate", (self.ffn, d), "w"),
                      (f"{prefix}.w_up", (self.ffn, d), "w"),
                      (f"{prefix}.w_down", (d, self.ffn), "w")]
            return items

        for i in range(self.n_layer):
            out += layer(f"slow.{i}", self.slow_qk_norm)
        out.append(("fast_emb", (self.fast_vocab, d), "w"))
        for i in range(self.fast_n_layer):
            out += layer(f"fast.{i}", self.fast_qk_norm)
        out += [("fast_norm", (d,), "g"),
                ("fast_out", (self.fast_vocab, d), "w"),
                ("fusion", (self.fusion_rows, d), "w")]
        return out


# Full S2-Pro-shaped model.  im_end_id is a placeholder: the pages do not
# print the id of <|im_end|>; any non-semantic id behaves the same under
# random weights.
S2PRO = DualARConfig(
    name="s2pro", dim=2560, n_layer=36, n_head=32, n_kv_head=8, head_dim=128,
    ffn=9728, vocab=155_776, sem_begin=151_678, n_sem=4_096, im_end_id=151_677,
    fast_n_layer=4, fast_vocab=4_096, n_codebooks=10)

# Tiny Dual-AR used for parity: 2+2 layers, dim 256, 4/2 heads of 64,
# FFN 768, vocab 1,024 (512 semantic ids at 512..1023), fast vocab 128,
# N = 4 codebooks (fusion table 512 + 3 x 128 = 896 rows).
TINY = DualARConfig(
    name="tiny", dim=256, n_layer=2, n_head=4, n_kv_head=2, head_dim=64,
    ffn=768, vocab=1_024, sem_begin=512, n_sem=512, im_end_id=3,
    fast_n_layer=2, fast_vocab=128, n_codebooks=4)

# Profiling case: S2-Pro layer shapes (dim 2560, 32/8 heads of 128, FFN 9728,
# 4,096 semantic ids, fast vocab 4,096, N = 10) with one slow and one fast
# layer and an 8,192-id vocabulary, so one process holds well under 1 GB.
S2PRO_L1 = DualARConfig(
    name="s2pro_l1", dim=2560, n_layer=1, n_head=32, n_kv_head=8, head_dim=128,
    ffn=9728, vocab=8_192, sem_begin=4_000, n_sem=4_096, im_end_id=3_999,
    fast_n_layer=1, fast_vocab=4_096, n_codebooks=10)

CONFIGS = {"tiny": TINY, "s2pro": S2PRO, "s2pro_l1": S2PRO_L1}

# Audio frames per second of the codec: 44,100 Hz / hop 2,048.
FRAMES_PER_AUDIO_SECOND = 44_100 / 2_048
