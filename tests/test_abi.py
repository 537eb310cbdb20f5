"""Host-only checks of the C ABI: the library loads, exports every symbol the
header declares, struct layouts agree with the header, and argument
validation rejects bad input before touching a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

from dual_ar_tts_frame_gb300 import _lib as L
from dual_ar_tts_frame_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dualar.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return L.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dualar_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(L.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    syms = set(re.findall(r"\bT (dualar_\w+)", out))
    for name in declared_functions():
        assert name in syms, name
        assert hasattr(lib, name)


def test_struct_layouts_match_header(tmp_path):
    src = tmp_path / "sz.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "dualar.h"\n'
                   'int main(void){printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(dualar_config),'
                   ' sizeof(dualar_layer_weights), sizeof(dualar_weights), sizeof(dualar_sampling),'
                   ' offsetof(dualar_config, rope_base), offsetof(dualar_weights, fusion));return 0;}\n')
    exe = tmp_path / "sz"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = list(map(int, subprocess.check_output([str(exe)]).split()))
    assert got == [ctypes.sizeof(L.dualar_config), ctypes.sizeof(L.dualar_layer_weights),
                   ctypes.sizeof(L.dualar_weights), ctypes.sizeof(L.dualar_sampling),
                   L.dualar_config.rope_base.offset, L.dualar_weights.fusion.offset]


def _tiny_config(**over):
    from dualar_inputs import TINY as c
    kw = dict(dim=c.dim, n_layer=c.n_layer, n_head=c.n_head, n_kv_head=c.n_kv_head,
              head_dim=c.head_dim, ffn=c.ffn, vocab=c.vocab, sem_begin=c.sem_begin, n_sem=c.n_sem,
              im_end_id=c.im_end_id, fast_n_layer=c.fast_n_layer, fast_vocab=c.fast_vocab,
              n_codebooks=c.n_codebooks, slow_qk_norm=1, fast_qk_norm=0, page_tokens=64,
              max_pages=8, max_seqs=2, max_ctx=256, rope_base=1e6, norm_eps=1e-6)
    kw.update(over)
    return L.dualar_config(**kw)


@pytest.mark.parametrize("over", [dict(head_dim=96), dict(page_tokens=32), dict(n_head=3),
                                  dict(n_codebooks=17), dict(im_end_id=600), dict(max_seqs=0),
                                  dict(dim=250), dict(n_sem=5000)])
def test_create_rejects_bad_config_without_gpu(lib, over):
    cfg = _tiny_config(**over)
    w = L.dualar_weights()
    h = ctypes.c_void_p()
    assert lib.dualar_create(ctypes.byref(cfg), ctypes.byref(w), None, ctypes.byref(h)) == -1
    assert not h.value


def test_create_rejects_null_or_misaligned_weights(lib):
    cfg = _tiny_config()
    w = L.dualar_weights(tok_emb=16, final_norm=32, fast_emb=48, fast_norm=64, fast_out=80, fusion=None)
    h = ctypes.c_void_p()
    assert lib.dualar_create(ctypes.byref(cfg), ctypes.byref(w), None, ctypes.byref(h)) == -1
    w.fusion = 97
    assert lib.dualar_create(ctypes.byref(cfg), ctypes.byref(w), None, ctypes.byref(h)) == -1


def test_null_handle_calls_are_rejected(lib):
    assert lib.dualar_prefill(None, 0, None, 0) == -1
    assert lib.dualar_release(None, 0) == -1
    assert lib.dualar_sync(None) == -1
    assert lib.dualar_slot_length(None, 0) == -1
    lib.dualar_destroy(None)


def test_w4a16_layout_and_argument_checks_without_gpu(lib):
    """Packed 4-bit records: k/2 code bytes + k/128 bf16 scales padded to 16
    bytes per row; sizes and pointers are checked before any GPU work."""
    assert lib.dualar_w4a16_bytes(1, 128) == 80
    assert lib.dualar_w4a16_bytes(2560, 9728) == 2560 * (4864 + 160)
    assert lib.dualar_w4a16_bytes(6144, 2560) == 6144 * (1280 + 48)
    assert lib.dualar_w4a16_bytes(0, 256) == 0
    for n, k in ((1, 100), (1, 0), (-1, 128), (3, 192)):
        assert lib.dualar_w4a16_bytes(n, k) == -1
    assert lib.dualar_quantize_w4a16(None, 4, 100, None, None) == -1     # k not a multiple of 128
    assert lib.dualar_quantize_w4a16(None, 4, 128, None, None) == -1     # NULL pointers
    assert lib.dualar_quantize_w4a16(16, 4, 128, 40, None) == -1         # unaligned output
    assert lib.dualar_quantize_w4a16(None, 0, 128, None, None) == 0      # nothing to do
    assert lib.dualar_set_w4a16(None, None, None) == -1
    assert ctypes.sizeof(L.dualar_w4a16_layer) == 5 * ctypes.sizeof(ctypes.c_void_p)


def test_late_attn_keys_agree_with_oracle():
    from dual_ar_tts_frame_gb300.decoder import late_attn_keys
    from oracle import w4a16
    for n, f, b in ((36, 4, 12), (2, 2, 1), (2, 2, 0), (2, 2, 2)):
        assert sorted(late_attn_keys(n, f, b)) == sorted(w4a16.late_attn_keys(n, f, b))


def test_byte_model_counts_packed_records_like_the_library(lib):
    """The 4-bit frame bytes of the byte model use the same record size as
    dualar_w4a16_bytes, and every packed projection is read once per slow
    step and once per fast pass."""
    from dualar_inputs import S2PRO
    from dual_ar_tts_frame_gb300 import bytemodel
    from dual_ar_tts_frame_gb300.decoder import late_attn_keys
    keys = late_attn_keys(S2PRO.n_layer, S2PRO.fast_n_layer, 12)
    shapes = bytemodel.projection_shapes(S2PRO)
    saved = 0
    for k in keys:
        stack, _, name = k.split(".")
        n, kk = shapes[name]
        reads = 1 if stack == "slow" else S2PRO.n_codebooks
        saved += reads * (2 * n * kk - lib.dualar_w4a16_bytes(n, kk))
    assert bytemodel.weight_bytes_per_step(S2PRO) - bytemodel.weight_bytes_per_step(S2PRO, keys) == saved
    assert bytemodel.weight_bytes_per_step(S2PRO, keys) == 4_649_059_328


def test_pack_w4a16_rejects_bad_shapes_before_any_gpu_work(lib):
    torch = pytest.importorskip("torch")
    from dual_ar_tts_frame_gb300 import pack_w4a16
    with pytest.raises(L.DualARError):
        pack_w4a16(torch.zeros((4, 100), dtype=torch.bfloat16))
