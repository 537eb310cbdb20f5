"""Seeded synthetic inputs: weights, prompts, uniforms, forced codes.

Both the CPU oracle and the CUDA path take their inputs from here, so the
two sides see the same bytes.  Everything is generated on the host by the
counter-based generator in ``gen.c`` and returned as NumPy arrays; the CUDA
harness copies them to the device unchanged.

Distributions (random-init model, no checkpoint):
  * matrices and embeddings: N(0, 0.02), stored as bf16;
  * RMSNorm gains: 1 + N(0, 0.02) (unit gains keep the logits O(1), so the
    tolerance rules on logits stay meaningful);
  * prompt tokens: uniform over the non-semantic ids other than <|im_end|>;
  * sampling uniforms: U[0, 1) with 24 random bits.
"""
from __future__ import annotations

import ctypes
import os
import statistics
import subprocess
import threading
import zlib

import numpy as np

from .config import DualARConfig

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libdualar_gen.so")
_lib = None
_lock = threading.Lock()

_M32 = 0xFFFFFFFF


def build_generator(force: bool = False) -> str:
    """Compile gen.c with the host C compiler (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC",
                               "-o", tmp, _SRC])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_generator())
            lib.dualar_gen_table16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                               ctypes.c_uint32, ctypes.c_uint32]
            lib.dualar_gen_uniform.argtypes = [ctypes.c_void_p, ctypes.c_int64,
                                               ctypes.c_uint32, ctypes.c_uint32]
            lib.dualar_gen_randint.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint32,
                                               ctypes.c_uint32, ctypes.c_int64, ctypes.c_int64]
            _lib = lib
    return _lib


def _fmix32(x: int) -> int:
    x &= _M32
    x ^= x >> 16
    x = (x * 0x85EBCA6B) & _M32
    x ^= x >> 13
    x = (x * 0xC2B2AE35) & _M32
    x ^= x >> 16
    return x


def stream_keys(seed: int, stream: str) -> tuple[int, int]:
    """Keys of one named stream under one seed."""
    s = zlib.crc32(stream.encode())
    k1 = _fmix32((seed * 0x9E3779B1 + s) & _M32)
    k2 = _fmix32(k1 ^ 0xA511E9B3 ^ ((seed >> 32) & _M32))
    return k1, k2


# ---- bf16 helpers (storage only) -----------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest even); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bits (uint16) to float32 exactly."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32)
    u <<= np.uint32(16)          # in place: one new array, not two
    return u.view(np.float32)


_tables: dict[str, np.ndarray] = {}


def _quantile_table(kind: str) -> np.ndarray:
    """65,536 bf16 quantiles: std * Phi^-1((k + 1/2) / 65536) (+ 1 for gains)."""
    if kind not in _tables:
        nd = statistics.NormalDist()
        q = np.array([nd.inv_cdf((k + 0.5) / 65536.0) for k in range(65536)], dtype=np.float64)
        v = 0.02 * q + (1.0 if kind == "g" else 0.0)
        _tables[kind] = f32_to_bf16_bits(v.astype(np.float32))
    return _tables[kind]


def gen_bf16(shape, seed: int, stream: str, kind: str = "w") -> np.ndarray:
    """bf16 bits (uint16) with the given shape from one named stream."""
    lib = _load()
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    tab = _quantile_table(kind)
    k1, k2 = stream_keys(seed, stream)
    lib.dualar_gen_table16(out.ctypes.data, n, tab.ctypes.data, k1, k2)
    return out.reshape(shape)


def gen_uniform(shape, seed: int, stream: str) -> np.ndarray:
    lib = _load()
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    k1, k2 = stream_keys(seed, stream)
    lib.dualar_gen_uniform(out.ctypes.data, n, k1, k2)
    return out.reshape(shape)


def gen_randint(shape, lo: int, hi: int, seed: int, stream: str) -> np.ndarray:
    lib = _load()
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.int64)
    k1, k2 = stream_keys(seed, stream)
    lib.dualar_gen_randint(out.ctypes.data, n, k1, k2, lo, hi)
    return out.reshape(shape)


# ---- model weights --------------------------------------------------------

def make_weights(cfg: DualARConfig, seed: int = 0) -> dict[str, np.ndarray]:
    """All weights of the random-init model as bf16 bits (uint16 arrays)."""
    return {name: gen_bf16(shape, seed, "w:" + name, kind)
            for name, shape, kind in cfg.weight_shapes()}


# ---- workloads ------------------------------------------------------------

def make_prompt(cfg: DualARConfig, n_tokens: int, seed: int, stream: str = "prompt") -> np.ndarray:
    """Prompt ids uniform over [0, sem_begin) without <|im_end|> (int32)."""
    t = gen_randint((n_tokens,), 0, cfg.sem_begin - 1, seed, stream)
    t = t + (t >= cfg.im_end_id)
    return t.astype(np.int32)


def make_uniforms(n_frames: int, batch: int, cfg: DualARConfig, seed: int,
                  stream: str = "uniforms") -> np.ndarray:
    """Sampling uniforms, float32 [frames][batch][N+1]."""
    return gen_uniform((n_frames, batch, cfg.n_codebooks + 1), seed, stream)


def make_forced_codes(n_frames: int, batch: int, cfg: DualARConfig, seed: int,
                      stream: str = "forced") -> np.ndarray:
    """Teacher-forcing codes int32 [frames][batch][N]: q0 in [0, n_sem),
    q1..q(N-1) in [0, fast_vocab)."""
    q0 = gen_randint((n_frames, batch, 1), 0, cfg.n_sem, seed, stream + ":q0")
    qk = gen_randint((n_frames, batch, cfg.n_codebooks - 1), 0, cfg.fast_vocab, seed,
                     stream + ":qk")
    return np.concatenate([q0, qk], axis=2).astype(np.int32)


def make_lengths(n: int, lo: int, hi_inclusive: int, seed: int, stream: str) -> np.ndarray:
    """Context/prompt lengths uniform on [lo, hi] (int64)."""
    return gen_randint((n,), lo, hi_inclusive + 1, seed, stream)


def make_replacement_workload(batch: int, n_long: int, n_queue: int, seed: int) -> dict:
    """The batch-128 replacement workload: `batch - n_long` contexts uniform
    on [2,048, 4,096], `n_long` contexts of 16,384 that stay resident, a
    finish frame uniform on [1, 64] for every sequence (the long ones never
    finish), and a queue of `n_queue` replacement contexts uniform on
    [2,048, 4,096] with their own finish frames, taken in order."""
    short = make_lengths(batch - n_long, 2048, 4096, seed, "repl_ctx")
    ctx = np.concatenate([short, np.full(n_long, 16384, np.int64)])
    finish = np.concatenate([make_lengths(batch - n_long, 1, 64, seed, "repl_finish"),
                             np.full(n_long, -1, np.int64)])
    return {"ctx": ctx, "finish": finish,
            "queue_ctx": make_lengths(n_queue, 2048, 4096, seed, "repl_queue_ctx"),
            "queue_finish": make_lengths(n_queue, 1, 64, seed, "repl_queue_finish")}
