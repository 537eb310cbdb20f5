"""ctypes binding of libdualar.so (include/dualar.h), names unchanged.

Argument marshalling only: every step of the decode runs in the CUDA
library.  Importing this module does not load the library; ``lib()`` does,
and raises if the in-tree build is missing (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdualar.so")

DUALAR_OK = 0
ERRORS = {
    -1: "DUALAR_ERR_INVALID_ARG", -2: "DUALAR_ERR_OOM_PAGES", -3: "DUALAR_ERR_SLOT_BUSY",
    -4: "DUALAR_ERR_SLOT_EMPTY", -5: "DUALAR_ERR_CUDA", -6: "DUALAR_ERR_TIMEOUT",
    -7: "DUALAR_ERR_DEVICE", -8: "DUALAR_ERR_CONTEXT_FULL",
}

# Every symbol include/dualar.h declares.
EXPORTED = [
    "dualar_create", "dualar_prefill", "dualar_prefill_append", "dualar_share_prefix",
    "dualar_decode_frame", "dualar_decode_frame_forced",
    "dualar_decode_frame_noalloc",
    "dualar_release", "dualar_sync", "dualar_get_error", "dualar_destroy",
    "dualar_get_page_table", "dualar_get_rope_table", "dualar_read_state", "dualar_slot_length",
    "dualar_set_wait_limit", "dualar_last_launch_count", "dualar_set_persistent", "dualar_set_tensor_cores",
    "dualar_debug_barrier_extra", "dualar_debug_synthetic_context", "dualar_set_trace", "dualar_set_prefetch", "dualar_profile", "dualar_profile_read",
    "dualar_w4a16_bytes", "dualar_quantize_w4a16", "dualar_set_w4a16",
]

c_i32 = ctypes.c_int32
c_f32 = ctypes.c_float
c_vp = ctypes.c_void_p


class dualar_config(ctypes.Structure):
    _fields_ = [(n, c_i32) for n in (
        "dim", "n_layer", "n_head", "n_kv_head", "head_dim", "ffn", "vocab", "sem_begin", "n_sem",
        "im_end_id", "fast_n_layer", "fast_vocab", "n_codebooks", "slow_qk_norm", "fast_qk_norm",
        "page_tokens", "max_pages", "max_seqs", "max_ctx")] + [("rope_base", c_f32), ("norm_eps", c_f32)]


class dualar_layer_weights(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in ("attn_norm", "wqkv", "q_norm", "k_norm", "wo", "ffn_norm",
                                    "w_gate", "w_up", "w_down")]


class dualar_weights(ctypes.Structure):
    _fields_ = [("tok_emb", c_vp), ("final_norm", c_vp), ("slow", ctypes.POINTER(dualar_layer_weights)),
                ("fast_emb", c_vp), ("fast", ctypes.POINTER(dualar_layer_weights)),
                ("fast_norm", c_vp), ("fast_out", c_vp), ("fusion", c_vp)]


class dualar_w4a16_layer(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in ("wqkv", "wo", "w_gate", "w_up", "w_down")]


class dualar_sampling(ctypes.Structure):
    _fields_ = [("temperature", c_f32), ("top_p", c_f32), ("ras_win", c_i32),
                ("ras_temperature", c_f32), ("ras_top_p", c_f32), ("allow_eos", c_i32)]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads the shared library without touching the GPU."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with dual_ar_tts_frame_gb300.build.build() "
                           "(nvcc, sm_103a); there is no CPU fallback")
    _lib = bind(ctypes.CDLL(path))
    return _lib


def bind(L: ctypes.CDLL) -> ctypes.CDLL:
    """Declares the argument and result types of every entry point."""
    H = c_vp
    L.dualar_create.argtypes = [ctypes.POINTER(dualar_config), ctypes.POINTER(dualar_weights), c_vp,
                                ctypes.POINTER(H)]
    L.dualar_prefill.argtypes = [H, c_i32, ctypes.POINTER(c_i32), c_i32]
    L.dualar_prefill_append.argtypes = [H, c_i32, ctypes.POINTER(c_i32), c_i32]
    L.dualar_share_prefix.argtypes = [H, c_i32, c_i32, c_i32]
    L.dualar_decode_frame.argtypes = [H, c_i32, ctypes.POINTER(c_i32), c_vp,
                                      ctypes.POINTER(dualar_sampling), c_vp, c_vp]
    L.dualar_decode_frame_forced.argtypes = [H, c_i32, ctypes.POINTER(c_i32), c_vp,
                                             ctypes.POINTER(dualar_sampling), c_vp, c_vp, c_vp, c_vp,
                                             c_vp, c_vp]
    L.dualar_decode_frame_noalloc.argtypes = [H, c_i32, ctypes.POINTER(c_i32), c_vp,
                                              ctypes.POINTER(dualar_sampling), c_vp, c_vp]
    L.dualar_release.argtypes = [H, c_i32]
    L.dualar_sync.argtypes = [H]
    L.dualar_get_error.argtypes = [H, ctypes.c_char_p, ctypes.c_size_t]
    L.dualar_destroy.argtypes = [H]
    L.dualar_destroy.restype = None
    L.dualar_get_page_table.argtypes = [H, c_i32, ctypes.POINTER(c_i32), c_i32, ctypes.POINTER(c_i32)]
    L.dualar_get_rope_table.argtypes = [H, c_i32, c_vp, c_vp]
    L.dualar_read_state.argtypes = [H, c_i32, c_vp, c_vp]
    L.dualar_slot_length.argtypes = [H, c_i32]
    L.dualar_slot_length.restype = c_i32
    L.dualar_set_wait_limit.argtypes = [H, ctypes.c_uint64]
    L.dualar_last_launch_count.argtypes = [H]
    L.dualar_last_launch_count.restype = c_i32
    L.dualar_set_persistent.argtypes = [H, c_i32]
    L.dualar_set_tensor_cores.argtypes = [H, c_i32]
    L.dualar_debug_barrier_extra.argtypes = [H, ctypes.c_uint32]
    L.dualar_debug_synthetic_context.argtypes = [H, c_i32, c_i32, ctypes.c_uint32]
    L.dualar_set_prefetch.argtypes = [H, ctypes.c_uint64]
    L.dualar_set_trace.argtypes = [H, c_vp, ctypes.c_int64, ctypes.POINTER(c_i32), ctypes.POINTER(c_i32)]
    L.dualar_profile.argtypes = [H, c_i32]
    L.dualar_profile_read.argtypes = [H, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double),
                                      ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
    L.dualar_w4a16_bytes.argtypes = [c_i32, c_i32]
    L.dualar_w4a16_bytes.restype = ctypes.c_int64
    L.dualar_quantize_w4a16.argtypes = [c_vp, c_i32, c_i32, c_vp, c_vp]
    L.dualar_set_w4a16.argtypes = [H, ctypes.POINTER(dualar_w4a16_layer), ctypes.POINTER(dualar_w4a16_layer)]
    for n in EXPORTED:
        getattr(L, n)
    return L


def lib() -> ctypes.CDLL:
    return load()


class DualARError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code
