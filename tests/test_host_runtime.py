"""The library's host runtime (api.cu) on the CPU, without a GPU.

api.cu is compiled with a plain C++ compiler against tests/hostsim: a host
stand-in for the CUDA runtime ("device" memory is host memory, copies are
memcpy) whose kernel launchers do nothing, except that the setup launch
writes its page-table updates as the setup kernel does.  What is tested is
the host-side bookkeeping the GPU tests also cover, now on the CPU:

- page tables (read back through dualar_get_page_table, i.e. from the table
  the kernels would use) against the page oracle, through prefills, decode
  steps, releases, shared prefixes and prompt continuations;
- the error contract of include/dualar.h: INVALID_ARG, SLOT_BUSY,
  SLOT_EMPTY, OOM_PAGES and CONTEXT_FULL, each leaving the state unchanged;
- the 4-bit weight selection's argument checks.

The stand-in library never ships: the library itself is built only by nvcc for
sm_103a and has no CPU path.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

from dual_ar_tts_frame_gb300 import _lib as L
from dualar_inputs import TINY
from oracle import PageOracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HOSTSIM = os.path.join(ROOT, "tests", "hostsim")
CSRC = os.path.join(ROOT, "dual_ar_tts_frame_gb300", "csrc")

OK, INVALID, OOM, BUSY, EMPTY, FULL = 0, -1, -2, -3, -4, -8


@pytest.fixture(scope="module")
def hl(tmp_path_factory):
    if shutil.which("g++") is None:
        pytest.skip("no host C++ compiler")
    out = tmp_path_factory.mktemp("hostsim")
    inc = ["-I", HOSTSIM, "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    api_o, stubs_o = str(out / "api.o"), str(out / "stubs.o")
    subprocess.check_call(["g++", "-std=c++17", "-O1", "-fPIC", "-c", "-x", "c++", *inc,
                           os.path.join(CSRC, "api.cu"), "-o", api_o])
    subprocess.check_call(["g++", "-std=c++17", "-O1", "-fPIC", "-c", *inc,
                           os.path.join(HOSTSIM, "stubs.cpp"), "-o", stubs_o])
    so = str(out / "libdualar_hostsim.so")
    subprocess.check_call(["g++", "-shared", "-o", so, api_o, stubs_o])
    return L.bind(ctypes.CDLL(so))


class Host:
    """A tiny-config handle on the host stand-in, with fake (never read)
    16-byte-aligned weight addresses."""

    def __init__(self, lib, max_pages=12, max_seqs=4, max_ctx=400, **shape):
        self.lib, self.max_pages, self.max_seqs = lib, max_pages, max_seqs
        c = TINY
        kw = dict(dim=c.dim, n_layer=c.n_layer, n_head=c.n_head, n_kv_head=c.n_kv_head, head_dim=c.head_dim,
                  ffn=c.ffn, vocab=c.vocab, sem_begin=c.sem_begin, n_sem=c.n_sem, im_end_id=c.im_end_id,
                  fast_n_layer=c.fast_n_layer, fast_vocab=c.fast_vocab, n_codebooks=c.n_codebooks,
                  slow_qk_norm=1, fast_qk_norm=0, page_tokens=64, max_pages=max_pages, max_seqs=max_seqs,
                  max_ctx=max_ctx, rope_base=1e6, norm_eps=1e-6)
        kw.update(shape)
        cfg = L.dualar_config(**kw)
        addr = iter(range(0x10000, 0x10000 + 4096 * 4096, 4096))

        def layer():
            return L.dualar_layer_weights(*[next(addr) for _ in range(9)])

        self.slow = (L.dualar_layer_weights * c.n_layer)(*[layer() for _ in range(c.n_layer)])
        self.fast = (L.dualar_layer_weights * c.fast_n_layer)(*[layer() for _ in range(c.fast_n_layer)])
        w = L.dualar_weights(next(addr), next(addr), self.slow, next(addr), self.fast, next(addr), next(addr),
                             next(addr))
        self.h = ctypes.c_void_p()
        assert lib.dualar_create(ctypes.byref(cfg), ctypes.byref(w), None, ctypes.byref(self.h)) == OK
        n = c.n_codebooks
        self.uni = np.zeros((max_seqs, n + 1), np.float32)
        self.codes = np.zeros((max_seqs, n), np.int32)
        self.status = np.zeros(max_seqs, np.int32)
        self.smp = L.dualar_sampling(0.8, 0.8, 10, 1.0, 0.9, 1)

    def prefill(self, slot, n, append=False):
        tok = np.arange(n, dtype=np.int32) % 500 + 4
        f = self.lib.dualar_prefill_append if append else self.lib.dualar_prefill
        return f(self.h, slot, tok.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n)

    def decode(self, slots):
        s = np.asarray(slots, np.int32)
        return self.lib.dualar_decode_frame(self.h, len(s), s.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                            self.uni.ctypes.data, ctypes.byref(self.smp),
                                            self.codes.ctypes.data, self.status.ctypes.data)

    def table(self, slot):
        n = ctypes.c_int32()
        assert self.lib.dualar_get_page_table(self.h, slot, None, 0, ctypes.byref(n)) == OK
        buf = (ctypes.c_int32 * max(1, n.value))()
        assert self.lib.dualar_get_page_table(self.h, slot, buf, n.value, ctypes.byref(n)) == OK
        return list(buf)[:n.value]

    def length(self, slot):
        return self.lib.dualar_slot_length(self.h, slot)

    def state(self):
        return [(self.length(s), self.table(s)) for s in range(self.max_seqs)]

    def close(self):
        self.lib.dualar_destroy(self.h)


def check_tables(h, po):
    for s in range(h.max_seqs):
        assert h.table(s) == po.table.get(s, []), f"slot {s}"
        assert h.length(s) == po.length.get(s, -1)


def test_page_tables_follow_the_oracle_through_prefill_decode_release_and_sharing(hl):
    h = Host(hl, max_pages=40, max_seqs=4, max_ctx=600)
    po = PageOracle(40, 64)
    for slot, n in ((0, 130), (2, 64), (1, 1)):
        assert h.prefill(slot, n) == OK
        po.append(slot, n)
    check_tables(h, po)
    for _ in range(70):                             # crosses page boundaries for every slot
        assert h.decode([2, 0, 1]) == OK
        for s in (2, 0, 1):
            po.append(s, 1)
    check_tables(h, po)
    assert hl.dualar_release(h.h, 0) == OK
    po.release(0)
    assert h.prefill(3, 200) == OK                  # reuses the lowest freed pages first
    po.append(3, 200)
    check_tables(h, po)
    # a shared prefix: 100 of slot 3's positions (one full page shared, one copied)
    assert hl.dualar_share_prefix(h.h, 3, 0, 100) == OK
    po.share(3, 0, 100)
    check_tables(h, po)
    assert h.decode([0]) == INVALID                 # a bare prefix cannot decode
    assert h.prefill(0, 37, append=True) == OK
    po.append(0, 37)
    assert h.decode([0, 3]) == OK
    po.append(0, 1)
    po.append(3, 1)
    check_tables(h, po)
    # the shared page returns to the pool only with its last holder
    assert hl.dualar_release(h.h, 3) == OK
    po.release(3)
    check_tables(h, po)
    assert hl.dualar_release(h.h, 0) == OK
    po.release(0)
    assert hl.dualar_release(h.h, 2) == OK
    po.release(2)
    assert hl.dualar_release(h.h, 1) == OK
    po.release(1)
    check_tables(h, po)
    assert sorted(po.free) == list(range(40))
    for slot in range(4):                           # the whole pool is free again: 4 x 10 pages
        assert h.prefill(slot, 600) == OK
        po.append(slot, 600)
    check_tables(h, po)
    assert not po.free
    h.close()


def test_errors_leave_the_state_unchanged(hl):
    h = Host(hl, max_pages=6, max_seqs=3, max_ctx=300)
    assert h.prefill(0, 128) == OK                  # pages 0, 1
    assert h.prefill(1, 192) == OK                  # pages 2, 3, 4
    before = h.state()
    assert h.prefill(0, 10) == BUSY                 # slot holds a sequence
    assert h.prefill(2, 128) == OOM                 # 2 pages needed, 1 free
    assert h.prefill(2, 301) == FULL                # longer than max_ctx
    assert h.prefill(2, 0) == INVALID
    bad = np.array([TINY.vocab], np.int32)
    assert hl.dualar_prefill(h.h, 2, bad.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), 1) == INVALID
    assert h.decode([2]) == EMPTY                   # never prefilled
    assert h.decode([0, 0]) == INVALID              # repeated slot
    assert h.decode([0, 5]) == INVALID              # slot out of range
    assert h.prefill(2, 1, append=True) == EMPTY
    assert hl.dualar_share_prefix(h.h, 0, 1, 10) == BUSY
    assert hl.dualar_share_prefix(h.h, 2, 1, 10) in (EMPTY, INVALID)
    assert hl.dualar_share_prefix(h.h, 0, 2, 129) == INVALID   # longer than the source
    assert h.state() == before
    # two slots cross a page boundary on the same step with no page free
    assert h.prefill(2, 63) == OK                   # page 5, the last one
    assert h.decode([2]) == OK                      # position 63: still page 5
    before = h.state()
    assert h.decode([0, 2]) == OOM                  # positions 128 and 64 need two pages, none free
    assert h.state() == before
    h.close()


def test_context_full_on_decode(hl):
    h = Host(hl, max_pages=8, max_seqs=2, max_ctx=130)
    assert h.prefill(0, 128) == OK
    assert h.decode([0]) == OK
    assert h.decode([0]) == OK
    before = h.state()
    assert h.decode([0]) == FULL                    # position 130 = max_ctx
    assert h.state() == before
    h.close()


def test_w4a16_selection_checks(hl):
    h = Host(hl)
    c = TINY
    slow = (L.dualar_w4a16_layer * c.n_layer)()
    fast = (L.dualar_w4a16_layer * c.fast_n_layer)()
    assert hl.dualar_set_w4a16(h.h, slow, fast) == OK          # all NULL: bf16
    slow[0].w_gate = 0x20000
    assert hl.dualar_set_w4a16(h.h, slow, None) == INVALID     # gate without up
    slow[0].w_up = 0x20008
    assert hl.dualar_set_w4a16(h.h, slow, None) == INVALID     # not 16-byte aligned
    slow[0].w_up = 0x30000
    assert hl.dualar_set_w4a16(h.h, slow, None) == OK
    assert h.prefill(0, 70) == OK and h.decode([0]) == OK     # packed weights drive the same bookkeeping
    assert hl.dualar_set_w4a16(h.h, None, None) == OK
    h.close()


def test_decode_dispatch(hl):
    """Batches of 1-2 run as one setup plus one persistent-kernel launch
    (also with packed projections); batch 3, or the persistent kernel turned
    off, queues one kernel per op."""
    h = Host(hl, max_pages=16, max_seqs=4, max_ctx=300)
    for s in range(3):
        assert h.prefill(s, 20 + s) == OK
    assert h.decode([0]) == OK and hl.dualar_last_launch_count(h.h) == 2
    assert h.decode([1, 0]) == OK and hl.dualar_last_launch_count(h.h) == 2
    assert h.decode([2, 1, 0]) == OK and hl.dualar_last_launch_count(h.h) > 2
    slow = (L.dualar_w4a16_layer * TINY.n_layer)()
    slow[0].w_down = 0x40000
    assert hl.dualar_set_w4a16(h.h, slow, None) == OK
    assert h.decode([0]) == OK and hl.dualar_last_launch_count(h.h) == 2
    assert hl.dualar_set_persistent(h.h, 0) == OK
    assert h.decode([0]) == OK and hl.dualar_last_launch_count(h.h) > 2
    h.close()


def test_noalloc_batch_limit_at_the_s2pro_attention_shape(hl):
    """The no-allocation call keeps the split-KV scratch in a fixed 4 MiB
    array: at the S2-Pro attention shape (32 query heads, 8 KV heads of 128)
    that holds 3 sequences per call, as the header states."""
    h = Host(hl, max_pages=16, max_seqs=4, max_ctx=300, n_head=32, n_kv_head=8, head_dim=128)
    for sl in range(4):
        assert h.prefill(sl, 10) == OK
    s = np.arange(4, dtype=np.int32)

    def noalloc(n):
        return hl.dualar_decode_frame_noalloc(h.h, n, s.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                              h.uni.ctypes.data, ctypes.byref(h.smp), h.codes.ctypes.data,
                                              h.status.ctypes.data)
    before = h.state()
    assert noalloc(4) == INVALID
    buf = ctypes.create_string_buffer(512)
    hl.dualar_get_error(h.h, buf, 512)
    assert b"at most 3 sequences" in buf.value
    assert h.state() == before
    assert noalloc(3) == OK
    assert [h.length(i) for i in range(4)] == [11, 11, 11, 10]
    h.close()


def test_whole_sequence_share_and_synthetic_context(hl):
    """Sharing a slot's whole length hands over its held state, so the new
    slot decodes at once; the synthetic-context hook takes pages exactly as
    a prefill of the same length."""
    h = Host(hl, max_pages=20, max_seqs=4, max_ctx=400)
    po = PageOracle(20, 64)
    assert h.prefill(0, 150) == OK
    po.append(0, 150)
    assert hl.dualar_share_prefix(h.h, 0, 1, 150) == OK
    po.share(0, 1, 150)
    assert h.decode([1, 0]) == OK
    po.append(1, 1)
    po.append(0, 1)
    assert hl.dualar_debug_synthetic_context(h.h, 2, 130, 7) == OK
    po.append(2, 130)
    check_tables(h, po)
    assert hl.dualar_debug_synthetic_context(h.h, 2, 10, 7) == BUSY
    assert hl.dualar_debug_synthetic_context(h.h, 3, 401, 7) == FULL
    check_tables(h, po)
    h.close()
