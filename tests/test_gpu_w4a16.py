"""GPU parity of the 4-bit weight path (w4a16) against the CPU oracle.

[P3] "s2-pro-w4a16-late12attn" (model card, opening line): 4-bit weights,
16-bit activations, the late attention layers kept in bf16.  The library
packs bf16 matrices on the GPU (dualar_quantize_w4a16) and reads the packed
projections in the weight-streaming GEMV; the oracle applies its own copy of
the rule (oracle/w4a16.py) and runs the same model on the dequantised
weights.

- packing: the GPU's bytes equal the oracle's record bytes exactly (tiny
  shapes, the full-size 2560 x 9728 down projection, exact rounding ties);
- decode: teacher-forced frames of the tiny model (batches 1 and 2 through
  both decode paths, 12 per op; the late slow layer's attention in bf16) and
  of the one-layer full-width model
  (every projection packed, K = 2560 / 4096 / 9728) against the oracle on
  the same packed plan: logits within the tolerance, draws of the oracle's
  sampler on the GPU's logits equal to the GPU's;
- batches of 1-2 run packed and bf16 GEMVs in one persistent-kernel
  program, whose cached program follows every change of weights.
"""
import numpy as np
import pytest

from dualar_inputs import TINY, CONFIGS
from dualar_inputs import generators as g
from dualar_inputs.generators import f32_to_bf16_bits
from oracle import DualAROracle, PageOracle, Sampling as OSampling
from oracle import w4a16 as OW
from oracle.sampler import sample_q0, sample_top_p
from parity import DrawStats, assert_logits_close

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

S2PRO_L1 = CONFIGS["s2pro_l1"]


@pytest.fixture(scope="module")
def lib_built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dual_ar_tts_frame_gb300 import build
    build()


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.cuda() if dtype is None else t.to(dtype).cuda()


def gpu_pack(bits: np.ndarray) -> np.ndarray:
    from dual_ar_tts_frame_gb300 import pack_w4a16
    w = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)
    p = pack_w4a16(w)
    torch.cuda.synchronize()
    return p.cpu().numpy()


def ref_pack(bits: np.ndarray) -> np.ndarray:
    return OW.pack(*OW.quantize(bits))


# ------------------------------------------------------------------ packing --

def test_packing_bit_exact(lib_built):
    rng = np.random.default_rng(11)
    cases = []
    for n, k in ((1, 128), (7, 256), (33, 768), (2560, 9728)):
        cases.append(f32_to_bf16_bits((rng.standard_normal((n, k)) * 0.02).astype(np.float32)))
    # exact ties: (q + 1/2) * 2^-6 with a 7 * 2^-6 in every group (scale 2^-6)
    q = rng.integers(-7, 7, size=(16, 512)).astype(np.float32) + 0.5
    q[:, ::128] = 7.0
    cases.append(f32_to_bf16_bits((q / 64.0).astype(np.float32)))
    # zero groups, tiny and large groups in one row
    z = (rng.standard_normal((4, 512)) * 0.02).astype(np.float32)
    z[:, :128] = 0.0
    z[:, 128:256] *= 1e-4
    z[:, 256:384] *= 1e3
    cases.append(f32_to_bf16_bits(z))
    for bits in cases:
        got = gpu_pack(bits)
        want = ref_pack(bits)
        assert got.shape == want.shape
        np.testing.assert_array_equal(got, want)


# ---------------------------------------------------------- forced decode --

def packed_decoder(cfg, bits, keys, max_pages, max_seqs, max_ctx):
    from dual_ar_tts_frame_gb300 import DualARDecoder, pack_w4a16, upload_weights
    w = upload_weights(bits)
    d = DualARDecoder(cfg, w, max_pages=max_pages, max_seqs=max_seqs, max_ctx=max_ctx)
    d.set_w4a16({k: pack_w4a16(w[k]) for k in keys})
    return d


def gpu_sampling(o):
    from dual_ar_tts_frame_gb300 import Sampling
    return Sampling(o.temperature, o.top_p, o.ras_win, o.allow_eos, o.ras_temperature, o.ras_top_p)


def run_forced(cfg, d, o, prompts, n_frames, smp, seed, persistent=None):
    """persistent: True -- every frame is one persistent-kernel launch (plus
    setup); False -- one kernel per op; None -- not checked."""
    slots = list(prompts)
    seqs = {}
    pages = PageOracle(d.max_pages, cfg.page_tokens)
    for s, p in prompts.items():
        d.prefill(s, p)
        seqs[s] = o.prefill(p)
        pages.append(s, len(p))
        hid, z = d.read_state(s)
        assert_logits_close(hid, seqs[s].h_last, f"prefill hidden slot {s}")
        assert_logits_close(z, seqs[s].z_last, f"prefill logits slot {s}")
    b = len(slots)
    forced = g.make_forced_codes(n_frames, b, cfg, seed=seed)
    uni = g.make_uniforms(n_frames, b, cfg, seed=seed + 1)
    stats = DrawStats()
    for f in range(n_frames):
        codes, status, slow, fast, draws = d.decode_frame_forced(slots, dev(uni[f]), gpu_sampling(smp),
                                                                 dev(forced[f]))
        d.sync()
        if persistent is not None:
            assert (d.last_launch_count() <= 2) == persistent, d.last_launch_count()
        codes, status = codes.cpu().numpy(), status.cpu().numpy()
        slow, fast, draws = slow.cpu().numpy(), fast.cpu().numpy(), draws.cpu().numpy()
        np.testing.assert_array_equal(codes, forced[f])
        np.testing.assert_array_equal(status, 0)
        for i, s in enumerate(slots):
            hist = list(seqs[s].history)
            r = o.decode_frame(seqs[s], uni[f, i], smp, forced=forced[f, i])
            assert_logits_close(slow[i], r.slow_logits, f"slow logits f{f} slot {s}")
            assert_logits_close(fast[i], r.fast_logits, f"fast logits f{f} slot {s}")
            n0, ras, _ = sample_q0(cfg, slow[i], smp, hist, float(uni[f, i, 0]), float(uni[f, i, 1]))
            stats.check(draws[i, 0], n0, smp.temperature, f"q0 draw f{f}")
            stats.check(draws[i, 1], ras, smp.ras_temperature, f"ras draw f{f}")
            for k in range(1, cfg.n_codebooks):
                rk = sample_top_p(fast[i, k - 1], np.arange(cfg.fast_vocab), smp.temperature, smp.top_p,
                                  float(uni[f, i, k + 1]))
                stats.check(draws[i, k + 2], rk, smp.temperature, f"q{k} draw f{f}")
            pages.append(s, 1)
    for s in slots:
        assert d.page_table(s) == pages.table[s]
    assert stats.compared > 0


@pytest.fixture(scope="module")
def tiny_packed(lib_built, tiny_bits):
    keys = OW.late_attn_keys(TINY.n_layer, TINY.fast_n_layer, 1)
    return keys, DualAROracle(TINY, tiny_bits, max_pos=4096, w4a16_keys=keys)


@pytest.mark.parametrize("nseq,persistent", [(1, True), (1, False), (2, True), (2, False), (12, False)])
def test_tiny_forced_frames(tiny_bits, tiny_packed, nseq, persistent):
    """Batches 1 and 2 through the persistent frame kernel (packed and bf16
    GEMVs in one program) and one kernel per op, and batch 12 (the bf16 late
    attention on the tensor cores, packed projections in GEMV passes of <= 8
    rows)."""
    keys, o = tiny_packed
    smp = OSampling(temperature=0.8, top_p=0.8, ras_win=10)
    lens = g.make_lengths(nseq, 20, 200, seed=50 + nseq, stream="w4_tiny")
    prompts = {s: g.make_prompt(TINY, int(n), seed=60 + s) for s, n in enumerate(lens)}
    d = packed_decoder(TINY, tiny_bits, keys, max_pages=128, max_seqs=16, max_ctx=1024)
    d.set_persistent(persistent)
    run_forced(TINY, d, o, prompts, 4, smp, seed=70 + nseq, persistent=persistent and nseq <= 2)
    d.close()


def test_one_layer_full_width_forced_frames(lib_built):
    """Full widths (K = 2560, 4096, 9728: several records per tile, two
    warps per row for the down projection), every projection packed;
    batches 1 and 2 through the persistent frame kernel, 3 per op, ragged
    contexts across pages."""
    cfg = S2PRO_L1
    bits = g.make_weights(cfg, seed=0)
    keys = OW.late_attn_keys(cfg.n_layer, cfg.fast_n_layer, 0)
    o = DualAROracle(cfg, bits, max_pos=1024, w4a16_keys=keys)
    smp = OSampling(temperature=0.8, top_p=0.8, ras_win=10, allow_eos=False)
    for nseq, lens, pers in ((1, [70], True), (2, [200, 33], True), (3, [64, 130, 9], False)):
        prompts = {s: g.make_prompt(cfg, n, seed=80 + s) for s, n in enumerate(lens)}
        d = packed_decoder(cfg, bits, keys, max_pages=32, max_seqs=4, max_ctx=512)
        run_forced(cfg, d, o, prompts, 2, smp, seed=90 + nseq, persistent=pers)
        d.close()
    torch.cuda.empty_cache()


def test_switching_weights_rebuilds_the_persistent_program(lib_built, tiny_bits, tiny_oracle, tiny_packed):
    """One decoder: bf16 frames, then packed frames, then bf16 again; the
    persistent kernel's program follows each switch (each segment against
    its own oracle; each slot is released before the next one starts, so
    page numbers start from the bottom again)."""
    from dual_ar_tts_frame_gb300 import DualARDecoder, pack_w4a16, upload_weights
    keys, o4 = tiny_packed
    w = upload_weights(tiny_bits)
    packed = {k: pack_w4a16(w[k]) for k in keys}
    smp = OSampling(temperature=0.8, top_p=0.8, ras_win=10)
    d = DualARDecoder(TINY, w, max_pages=64, max_seqs=4, max_ctx=1024)
    for slot, (pk, o) in enumerate(((None, tiny_oracle), (packed, o4), (None, tiny_oracle))):
        d.set_w4a16(pk)
        run_forced(TINY, d, o, {slot: g.make_prompt(TINY, 40, seed=7 + slot)}, 3, smp, seed=8 + slot,
                   persistent=True)
        d.release(slot)
    d.close()
