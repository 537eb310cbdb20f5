"""Thin Python wrapper over the C ABI: holds the handle and the weight tensors.

PyTorch is used for device memory and streams only; each method marshals its
arguments and calls one libdualar.so entry point.
"""
from __future__ import annotations

import ctypes
import dataclasses

import numpy as np
import torch

from . import _lib as L


@dataclasses.dataclass
class Sampling:
    temperature: float = 0.8
    top_p: float = 0.8
    ras_win: int = 10
    allow_eos: bool = True
    ras_temperature: float = 1.0
    ras_top_p: float = 0.9

    def c(self) -> L.dualar_sampling:
        return L.dualar_sampling(self.temperature, self.top_p, self.ras_win, self.ras_temperature,
                                 self.ras_top_p, int(self.allow_eos))


def upload_weights(bits: dict[str, np.ndarray], device="cuda") -> dict[str, torch.Tensor]:
    """bf16 bit arrays (uint16) -> bf16 device tensors, unchanged bytes."""
    out = {}
    for k, v in bits.items():
        t = torch.from_numpy(np.ascontiguousarray(v).view(np.int16))
        out[k] = t.to(device).view(torch.bfloat16)
    return out


PROJECTIONS = ("wqkv", "wo", "w_gate", "w_up", "w_down")


def late_attn_keys(n_layer: int, fast_n_layer: int, n_bf16_attn: int = 12) -> list[str]:
    """Weight names packed in the "late12attn" 4-bit variant (the model card
    "s2-pro-w4a16-late12attn"): every projection except the query/key/value
    and output projections of the last n_bf16_attn slow layers."""
    out = []
    for i in range(n_layer):
        late = i >= n_layer - n_bf16_attn
        out += [f"slow.{i}.{m}" for m in PROJECTIONS if not (late and m in ("wqkv", "wo"))]
    out += [f"fast.{i}.{m}" for i in range(fast_n_layer) for m in PROJECTIONS]
    return out


def pack_w4a16(w: torch.Tensor, stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """bf16 device matrix [n][k] -> its packed 4-bit records (uint8 [n][record
    bytes]) via dualar_quantize_w4a16, queued on the stream."""
    lib = L.lib()
    n, k = w.shape
    nbytes = lib.dualar_w4a16_bytes(n, k)
    if nbytes < 0:
        raise L.DualARError(-1, f"dualar_w4a16_bytes({n}, {k}): k must be a positive multiple of 128")
    out = torch.empty(nbytes, dtype=torch.uint8, device=w.device)
    st = stream or torch.cuda.current_stream()
    rc = lib.dualar_quantize_w4a16(ctypes.c_void_p(w.contiguous().data_ptr()), n, k,
                                   ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(st.cuda_stream))
    if rc != L.DUALAR_OK:
        raise L.DualARError(rc, "dualar_quantize_w4a16 failed")
    return out.view(n, nbytes // max(n, 1)) if n else out


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


class DualARDecoder:
    def __init__(self, cfg, weights: dict[str, torch.Tensor], max_pages: int, max_seqs: int,
                 max_ctx: int, stream: torch.cuda.Stream | None = None):
        self.lib = L.lib()
        self.cfg = cfg
        self.max_pages = max_pages
        self.max_seqs = max_seqs
        self.max_ctx = max_ctx
        self.weights = weights        # keeps the device memory alive
        self.stream = stream or torch.cuda.current_stream()
        c = L.dualar_config(
            dim=cfg.dim, n_layer=cfg.n_layer, n_head=cfg.n_head, n_kv_head=cfg.n_kv_head,
            head_dim=cfg.head_dim, ffn=cfg.ffn, vocab=cfg.vocab, sem_begin=cfg.sem_begin,
            n_sem=cfg.n_sem, im_end_id=cfg.im_end_id, fast_n_layer=cfg.fast_n_layer,
            fast_vocab=cfg.fast_vocab, n_codebooks=cfg.n_codebooks, slow_qk_norm=int(cfg.slow_qk_norm),
            fast_qk_norm=int(cfg.fast_qk_norm), page_tokens=cfg.page_tokens, max_pages=max_pages,
            max_seqs=max_seqs, max_ctx=max_ctx, rope_base=cfg.rope_base, norm_eps=cfg.norm_eps)
        w = weights

        def layer(p, qk):
            return L.dualar_layer_weights(
                w[p + ".attn_norm"].data_ptr(), w[p + ".wqkv"].data_ptr(),
                w[p + ".q_norm"].data_ptr() if qk else None, w[p + ".k_norm"].data_ptr() if qk else None,
                w[p + ".wo"].data_ptr(), w[p + ".ffn_norm"].data_ptr(), w[p + ".w_gate"].data_ptr(),
                w[p + ".w_up"].data_ptr(), w[p + ".w_down"].data_ptr())

        slow = (L.dualar_layer_weights * cfg.n_layer)(
            *[layer(f"slow.{i}", cfg.slow_qk_norm) for i in range(cfg.n_layer)])
        fast = (L.dualar_layer_weights * cfg.fast_n_layer)(
            *[layer(f"fast.{i}", cfg.fast_qk_norm) for i in range(cfg.fast_n_layer)])
        cw = L.dualar_weights(w["tok_emb"].data_ptr(), w["final_norm"].data_ptr(), slow,
                              w["fast_emb"].data_ptr(), fast, w["fast_norm"].data_ptr(),
                              w["fast_out"].data_ptr(), w["fusion"].data_ptr())
        h = ctypes.c_void_p()
        rc = self.lib.dualar_create(ctypes.byref(c), ctypes.byref(cw),
                                    ctypes.c_void_p(self.stream.cuda_stream), ctypes.byref(h))
        if rc != L.DUALAR_OK:
            raise L.DualARError(rc, "dualar_create failed (message on stderr)")
        self.h = h

    def set_w4a16(self, packed: dict[str, torch.Tensor] | None) -> None:
        """Reads the named projections ("slow.3.w_down", ...) from their packed
        4-bit records (pack_w4a16) from now on; None or {} restores bf16."""
        packed = packed or {}
        cfg = self.cfg

        def layers(stack, n):
            arr = (L.dualar_w4a16_layer * n)()
            for i in range(n):
                for m in PROJECTIONS:
                    t = packed.get(f"{stack}.{i}.{m}")
                    if t is not None:
                        setattr(arr[i], m, t.data_ptr())
            return arr

        any_slow = any(k.startswith("slow.") for k in packed)
        any_fast = any(k.startswith("fast.") for k in packed)
        slow = layers("slow", cfg.n_layer) if any_slow else None
        fast = layers("fast", cfg.fast_n_layer) if any_fast else None
        self._check(self.lib.dualar_set_w4a16(self.h, slow, fast))
        self.packed = dict(packed)    # keeps the device memory alive

    # ---- helpers ----------------------------------------------------------
    def _check(self, rc: int):
        if rc != L.DUALAR_OK:
            buf = ctypes.create_string_buffer(512)
            self.lib.dualar_get_error(self.h, buf, 512)
            raise L.DualARError(rc, buf.value.decode())

    def close(self):
        if getattr(self, "h", None):
            self.lib.dualar_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- C ABI ------------------------------------------------------------
    def prefill(self, slot: int, tokens) -> None:
        t = np.ascontiguousarray(np.asarray(tokens, np.int32))
        self._check(self.lib.dualar_prefill(self.h, slot, t.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                            t.size))

    def prefill_append(self, slot: int, tokens) -> None:
        """Continues the prompt of a slot (after share_prefix)."""
        t = np.ascontiguousarray(np.asarray(tokens, np.int32))
        self._check(self.lib.dualar_prefill_append(self.h, slot, t.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                                   t.size))

    def share_prefix(self, src: int, dst: int, n_tokens: int) -> None:
        """Starts slot dst from the first n_tokens positions of slot src (shared pages)."""
        self._check(self.lib.dualar_share_prefix(self.h, src, dst, n_tokens))

    def decode_frame(self, slots, uniforms: torch.Tensor, sampling: Sampling,
                     codes: torch.Tensor | None = None, status: torch.Tensor | None = None):
        s = np.ascontiguousarray(np.asarray(slots, np.int32))
        b = s.size
        n = self.cfg.n_codebooks
        if codes is None:
            codes = torch.empty((b, n), dtype=torch.int32, device=uniforms.device)
        if status is None:
            status = torch.empty((b,), dtype=torch.int32, device=uniforms.device)
        smp = sampling.c()
        self._check(self.lib.dualar_decode_frame(
            self.h, b, s.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), _ptr(uniforms),
            ctypes.byref(smp), _ptr(codes), _ptr(status)))
        return codes, status

    def decode_frame_noalloc(self, slots, uniforms: torch.Tensor, sampling: Sampling,
                             codes: torch.Tensor, status: torch.Tensor):
        """dualar_decode_frame_noalloc: the caller passes every output buffer;
        the call itself allocates nothing."""
        s = np.ascontiguousarray(np.asarray(slots, np.int32))
        smp = sampling.c()
        self._check(self.lib.dualar_decode_frame_noalloc(
            self.h, s.size, s.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), _ptr(uniforms),
            ctypes.byref(smp), _ptr(codes), _ptr(status)))
        return codes, status

    def decode_frame_forced(self, slots, uniforms: torch.Tensor, sampling: Sampling,
                            forced: torch.Tensor | None, want_logits: bool = True):
        s = np.ascontiguousarray(np.asarray(slots, np.int32))
        b = s.size
        cfg = self.cfg
        dev = uniforms.device
        codes = torch.empty((b, cfg.n_codebooks), dtype=torch.int32, device=dev)
        status = torch.empty((b,), dtype=torch.int32, device=dev)
        slow = torch.empty((b, cfg.n_sem + 1), dtype=torch.float32, device=dev) if want_logits else None
        fastl = (torch.empty((b, cfg.n_codebooks - 1, cfg.fast_vocab), dtype=torch.float32, device=dev)
                 if want_logits else None)
        draws = torch.empty((b, cfg.n_codebooks + 2), dtype=torch.int32, device=dev)
        smp = sampling.c()
        self._check(self.lib.dualar_decode_frame_forced(
            self.h, b, s.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), _ptr(uniforms),
            ctypes.byref(smp), _ptr(forced), _ptr(codes), _ptr(status), _ptr(slow), _ptr(fastl),
            _ptr(draws)))
        return codes, status, slow, fastl, draws

    def release(self, slot: int) -> None:
        self._check(self.lib.dualar_release(self.h, slot))

    def sync(self) -> None:
        self._check(self.lib.dualar_sync(self.h))

    def page_table(self, slot: int) -> list[int]:
        n = ctypes.c_int32()
        self._check(self.lib.dualar_get_page_table(self.h, slot, None, 0, ctypes.byref(n)))
        buf = (ctypes.c_int32 * max(1, n.value))()
        self._check(self.lib.dualar_get_page_table(self.h, slot, buf, n.value, ctypes.byref(n)))
        return list(buf)[:n.value]

    def rope_table(self, n_pos: int) -> tuple[np.ndarray, np.ndarray]:
        half = self.cfg.head_dim // 2
        c = np.empty((n_pos, half), np.uint16)
        s = np.empty((n_pos, half), np.uint16)
        self._check(self.lib.dualar_get_rope_table(self.h, n_pos, c.ctypes.data, s.ctypes.data))
        return c, s

    def read_state(self, slot: int) -> tuple[np.ndarray, np.ndarray]:
        hid = np.empty(self.cfg.dim, np.float32)
        z = np.empty(self.cfg.n_sem + 1, np.float32)
        self._check(self.lib.dualar_read_state(self.h, slot, hid.ctypes.data, z.ctypes.data))
        return hid, z

    def slot_length(self, slot: int) -> int:
        return int(self.lib.dualar_slot_length(self.h, slot))

    def set_wait_limit(self, ns: int) -> None:
        self._check(self.lib.dualar_set_wait_limit(self.h, ns))

    def last_launch_count(self) -> int:
        return int(self.lib.dualar_last_launch_count(self.h))

    def set_persistent(self, enable: bool) -> None:
        self._check(self.lib.dualar_set_persistent(self.h, int(enable)))

    def set_tensor_cores(self, enable: bool) -> None:
        self._check(self.lib.dualar_set_tensor_cores(self.h, int(enable)))

    def debug_barrier_extra(self, extra: int) -> None:
        self._check(self.lib.dualar_debug_barrier_extra(self.h, extra))

    def synthetic_context(self, slot: int, n_tokens: int, seed: int = 0) -> None:
        """Benchmark/test hook: a context of n_tokens seeded positions, no prefill."""
        self._check(self.lib.dualar_debug_synthetic_context(self.h, slot, n_tokens, seed & 0xFFFFFFFF))

    def set_prefetch(self, bytes_per_sm: int) -> None:
        self._check(self.lib.dualar_set_prefetch(self.h, bytes_per_sm))

    def set_trace(self, buf: torch.Tensor | None):
        """Per-op timeline of the persistent kernel into buf (uint64 device
        tensor); returns (n_ops, n_ctas) for a batch of 1."""
        n_ops, n_ctas = ctypes.c_int32(), ctypes.c_int32()
        self._check(self.lib.dualar_set_trace(self.h, _ptr(buf), buf.numel() * 8 if buf is not None else 0,
                                              ctypes.byref(n_ops), ctypes.byref(n_ctas)))
        return n_ops.value, n_ctas.value

    def profile(self, enable: bool) -> None:
        self._check(self.lib.dualar_profile(self.h, int(enable)))

    def profile_read(self) -> dict:
        n = ctypes.c_int64()
        t = ctypes.c_double()
        b = ctypes.c_double()
        m = ctypes.c_double()
        self._check(self.lib.dualar_profile_read(self.h, ctypes.byref(n), ctypes.byref(t), ctypes.byref(b),
                                                 ctypes.byref(m)))
        return {"launches": n.value, "total_ms": t.value, "total_bytes": b.value, "max_ms": m.value}
