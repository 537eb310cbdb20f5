"""GPU parity of the tiny Dual-AR against the CPU oracle, through the C ABI.

Tiny config: 2+2 layers, dim 256, 4/2 heads of 64, FFN 768, vocab 1,024
(512 semantic ids), fast vocab 128, N = 4; 32-token prompt, 16 frames under
teacher forcing, greedy and sampled decoding.  Sizes span several GEMV
tiles, several KV pages and split-KV chunks, and ragged batches.
"""
import numpy as np
import pytest

from dualar_inputs import TINY
from dualar_inputs import generators as g
from oracle import DualAROracle, PageOracle, Sampling as OSampling
from oracle import model as om
from oracle.sampler import sample_q0, sample_top_p
from parity import DrawStats, assert_logits_close

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev_weights(tiny_bits):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dual_ar_tts_frame_gb300 import build, upload_weights
    build()
    return upload_weights(tiny_bits)


def make(dev_weights, max_pages=64, max_seqs=4, max_ctx=1024, persistent=True):
    from dual_ar_tts_frame_gb300 import DualARDecoder
    d = DualARDecoder(TINY, dev_weights, max_pages=max_pages, max_seqs=max_seqs, max_ctx=max_ctx)
    d.set_persistent(persistent)
    return d


def gpu_sampling(o: OSampling):
    from dual_ar_tts_frame_gb300 import Sampling
    return Sampling(o.temperature, o.top_p, o.ras_win, o.allow_eos, o.ras_temperature, o.ras_top_p)


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.cuda() if dtype is None else t.to(dtype).cuda()


# ------------------------------------------------------------------ tables --

def test_rope_table_bit_exact(dev_weights):
    d = make(dev_weights)
    n = 1025
    c, s = d.rope_table(n)
    oc, os_ = om.rope_table(n, TINY.head_dim, TINY.rope_base)
    np.testing.assert_array_equal(c, (oc.view(np.uint32) >> 16).astype(np.uint16))
    np.testing.assert_array_equal(s, (os_.view(np.uint32) >> 16).astype(np.uint16))
    d.close()


# ----------------------------------------------------------------- prefill --

def test_prefill_state_matches_oracle(dev_weights, tiny_oracle):
    d = make(dev_weights)
    prompt = g.make_prompt(TINY, 32, seed=0)
    d.prefill(0, prompt)
    hid, z = d.read_state(0)
    d.sync()
    seq = tiny_oracle.prefill(prompt)
    assert_logits_close(hid, seq.h_last, "prefill hidden")
    assert_logits_close(z, seq.z_last, "prefill logits")
    assert d.slot_length(0) == 32
    d.close()


# --------------------------------------------------------- teacher forcing --

def run_forced(d, o, slot_prompts, n_frames, smp, seed):
    """Teacher-forced frames for several slots; checks logits, codes, draws
    (sampler on the GPU's own logits) and page tables."""
    slots = list(slot_prompts)
    seqs = {}
    pages = PageOracle(d.max_pages, TINY.page_tokens)
    for s, p in slot_prompts.items():
        d.prefill(s, p)
        seqs[s] = o.prefill(p)
        pages.append(s, len(p))
    b = len(slots)
    forced = g.make_forced_codes(n_frames, b, TINY, seed=seed)
    uni = g.make_uniforms(n_frames, b, TINY, seed=seed + 1)
    stats = DrawStats()
    for f in range(n_frames):
        codes, status, slow, fast, draws = d.decode_frame_forced(
            slots, dev(uni[f]), gpu_sampling(smp), dev(forced[f]))
        d.sync()
        codes, status = codes.cpu().numpy(), status.cpu().numpy()
        slow, fast, draws = slow.cpu().numpy(), fast.cpu().numpy(), draws.cpu().numpy()
        np.testing.assert_array_equal(codes, forced[f])
        np.testing.assert_array_equal(status, 0)
        for i, s in enumerate(slots):
            hist = list(seqs[s].history)
            r = o.decode_frame(seqs[s], uni[f, i], smp, forced=forced[f, i])
            assert_logits_close(slow[i], r.slow_logits, f"slow logits f{f} slot {s}")
            assert_logits_close(fast[i], r.fast_logits, f"fast logits f{f} slot {s}")
            # sampler alone: the oracle's draws from the GPU's logits
            n0, ras, ch = sample_q0(TINY, slow[i], smp, hist, float(uni[f, i, 0]), float(uni[f, i, 1]))
            stats.check(draws[i, 0], n0, smp.temperature, f"q0 draw f{f}")
            stats.check(draws[i, 1], ras, smp.ras_temperature, f"ras draw f{f}")
            for k in range(1, TINY.n_codebooks):
                rk = sample_top_p(fast[i, k - 1], np.arange(TINY.fast_vocab), smp.temperature, smp.top_p,
                                  float(uni[f, i, k + 1]))
                stats.check(draws[i, k + 2], rk, smp.temperature, f"q{k} draw f{f}")
            pages.append(s, 1)
    for s in slots:
        assert d.page_table(s) == pages.table[s]
        assert d.slot_length(s) == len(slot_prompts[s]) + n_frames
    assert stats.compared > 0
    return stats


@pytest.fixture(params=[True, False], ids=["persistent", "per-op"])
def dec(dev_weights, request):
    """Both decode paths: the persistent frame kernel (batches of 1-2) and one
    kernel per op (any batch)."""
    d = make(dev_weights, persistent=request.param)
    yield d
    d.close()


def test_teacher_forced_b1(dec, tiny_oracle):
    smp = OSampling(temperature=0.8, top_p=0.8, ras_win=10)
    run_forced(dec, tiny_oracle, {0: g.make_prompt(TINY, 32, seed=0)}, 16, smp, seed=3)


def test_teacher_forced_b2(dec, tiny_oracle):
    """Two sequences (the persistent kernel's largest batch), contexts across
    several pages and split-KV chunks."""
    smp = OSampling(temperature=0.8, top_p=0.8, ras_win=10)
    prompts = {3: g.make_prompt(TINY, 150, seed=14), 1: g.make_prompt(TINY, 60, seed=15)}
    run_forced(dec, tiny_oracle, prompts, 8, smp, seed=16)


@pytest.mark.parametrize("rows", [1, 2])
def test_paths_bit_identical(dev_weights, rows):
    """The persistent kernel and the per-op path commit the same codes and
    hold bit-identical state after sampled frames (one and two rows: the
    GEMV consumer's grouped lane sums must give the per-tile sums' bits)."""
    prompts = [g.make_prompt(TINY, 90, seed=17), g.make_prompt(TINY, 45, seed=19)][:rows]
    uni = g.make_uniforms(8, rows, TINY, seed=18)
    smp = gpu_sampling(OSampling(temperature=0.8, top_p=0.8, ras_win=10))
    out = []
    for persistent in (True, False):
        d = make(dev_weights, persistent=persistent)
        for s, p in enumerate(prompts):
            d.prefill(s, p)
        codes = []
        for f in range(8):
            c, s_ = d.decode_frame(list(range(rows)), dev(uni[f]), smp)
            codes.append(c.cpu().numpy())
        d.sync()
        out.append((np.stack(codes), [d.read_state(s) for s in range(rows)]))
        d.close()
    np.testing.assert_array_equal(out[0][0], out[1][0])
    for s in range(rows):
        np.testing.assert_array_equal(out[0][1][s][0], out[1][1][s][0])
        np.testing.assert_array_equal(out[0][1][s][1], out[1][1][s][1])


def test_teacher_forced_ragged_batch(dec, tiny_oracle):
    """Three slots with ragged contexts: multi-chunk prefill (300 > 128 rows),
    several pages and split-KV chunks with the last-arriver combine."""
    smp = OSampling(temperature=1.0, top_p=0.95, ras_win=10)
    prompts = {2: g.make_prompt(TINY, 40, seed=10), 0: g.make_prompt(TINY, 300, seed=11),
               3: g.make_prompt(TINY, 127, seed=12)}
    run_forced(dec, tiny_oracle, prompts, 6, smp, seed=13)


# --------------------------------------------------------- sampled replay --

def run_replay(d, o, prompt, n_frames, smp, seed, twin_main_entry=False):
    """Sampled decoding, replayed by the oracle along the GPU's trajectory.

    Each GPU draw is compared with the oracle's draw from the oracle's logits
    whenever that draw is stable under the measured logit difference eps
    (tests/parity.py: draw_decidable).  With twin_main_entry, a second slot
    with the same prompt runs through dualar_decode_frame and must commit
    bit-identical codes."""
    from parity import draw_decidable
    d.prefill(1, prompt)
    if twin_main_entry:
        d.prefill(2, prompt)
    seq = o.prefill(prompt)
    uni = g.make_uniforms(n_frames, 1, TINY, seed=seed)
    stats = DrawStats()      # oracle logits, draws stable under the measured eps
    samp = DrawStats()       # oracle sampler on the GPU's own logits
    for f in range(n_frames):
        codes, status, slow, fast, draws = d.decode_frame_forced([1], dev(uni[f]), gpu_sampling(smp), None)
        if twin_main_entry:
            c2, s2 = d.decode_frame([2], dev(uni[f]), gpu_sampling(smp))
        d.sync()
        codes, status = codes.cpu().numpy()[0], int(status.cpu()[0])
        slow, fast, draws = slow.cpu().numpy()[0], fast.cpu().numpy()[0], draws.cpu().numpy()[0]
        assert status == 0
        if twin_main_entry:
            np.testing.assert_array_equal(c2.cpu().numpy()[0], codes)
            assert int(s2.cpu()[0]) == 0
        hist = list(seq.history)
        # the sampler alone, on the GPU's logits
        g0, gr, gch = sample_q0(TINY, slow, smp, hist, float(uni[f, 0, 0]), float(uni[f, 0, 1]))
        samp.check(draws[0], g0, smp.temperature, f"q0 draw f{f}")
        samp.check(draws[1], gr, smp.ras_temperature, f"ras draw f{f}")
        if draw_decidable(g0, smp.temperature) and draw_decidable(gr, smp.ras_temperature):
            assert draws[2] == gch and codes[0] == gch
        for k in range(1, TINY.n_codebooks):
            rk = sample_top_p(fast[k - 1], np.arange(TINY.fast_vocab), smp.temperature, smp.top_p,
                              float(uni[f, 0, k + 1]))
            samp.check(codes[k], rk, smp.temperature, f"q{k} draw f{f}")
        # replay the GPU trajectory in the oracle
        r = o.decode_frame(seq, uni[f, 0], smp, forced=codes)
        n0, ras, chosen = r.draws[0]
        assert_logits_close(slow, r.slow_logits, f"slow f{f}")
        assert_logits_close(fast, r.fast_logits, f"fast f{f}")
        eps0 = float(np.abs(slow - r.slow_logits).max())
        triggered = smp.ras_win > 0 and n0.index != TINY.n_sem and n0.index in hist[-smp.ras_win:]
        if draw_decidable(n0, smp.temperature, eps0) and (
                not triggered or draw_decidable(ras, smp.ras_temperature, eps0)):
            stats.compared += 1
            assert codes[0] == chosen, f"q0 f{f}: gpu {codes[0]} oracle {chosen}"
        else:
            stats.excluded += 1
        for k in range(1, TINY.n_codebooks):
            epsk = float(np.abs(fast[k - 1] - r.fast_logits[k - 1]).max())
            stats.check(codes[k], r.draws[k], smp.temperature, f"q{k} f{f}", epsk)
    assert samp.compared > 0
    if smp.temperature <= 0:
        assert stats.compared > 0
    print(f"draws on oracle logits: {stats.compared} compared, {stats.excluded} not stable under eps; "
          f"sampler on GPU logits: {samp.compared} compared, {samp.excluded} at a boundary")
    return stats


@pytest.mark.parametrize("ras_win", [0, 10])
def test_greedy_replay(dec, tiny_oracle, ras_win):
    smp = OSampling(temperature=0.0, top_p=0.8, ras_win=ras_win)
    run_replay(dec, tiny_oracle, g.make_prompt(TINY, 32, seed=0), 16, smp, seed=21)


def test_sampled_replay_and_main_entry_point(dec, tiny_oracle):
    smp = OSampling(temperature=0.8, top_p=0.8, ras_win=10)
    run_replay(dec, tiny_oracle, g.make_prompt(TINY, 32, seed=0), 16, smp, seed=22, twin_main_entry=True)


def test_sampled_replay_other_params(dec, tiny_oracle):
    smp = OSampling(temperature=1.3, top_p=0.6, ras_win=4)
    run_replay(dec, tiny_oracle, g.make_prompt(TINY, 70, seed=5), 12, smp, seed=23)


# ---------------------------------------------------------- end of stream --

def test_eos_and_finished_slot(dec):
    p = g.make_prompt(TINY, 20, seed=1)
    dec.prefill(0, p)
    dec.prefill(1, p)
    uni = dev(g.make_uniforms(1, 2, TINY, seed=2)[0])
    forced = dev(np.array([[TINY.n_sem, 1, 2, 3], [5, 1, 2, 3]], np.int32))
    smp = gpu_sampling(OSampling())
    codes, status, _, _, _ = dec.decode_frame_forced([0, 1], uni, smp, forced)
    dec.sync()
    assert status.cpu().tolist() == [1, 0]
    assert codes.cpu().numpy()[0].tolist() == [-1] * TINY.n_codebooks
    assert codes.cpu().numpy()[1].tolist() == [5, 1, 2, 3]
    codes, status = dec.decode_frame([0, 1], uni, smp)
    dec.sync()
    assert status.cpu().tolist()[0] == 2
    assert codes.cpu().numpy()[0].tolist() == [-1] * TINY.n_codebooks
    dec.release(0)
    dec.prefill(0, p)           # the slot is reusable
    codes, status = dec.decode_frame([0], uni[:1], smp)
    dec.sync()
    assert status.cpu().tolist() == [0]


@pytest.mark.parametrize("rows", [2, 3])
def test_replacement_flow_matches_oracle(dec, tiny_oracle, rows):
    """A sequence finishes (forced <|im_end|>), its slot is released and
    restarted from a queued prompt, and the batch decodes on: every live
    row's slow and fast logits match the oracle (the restarted one against a
    fresh oracle sequence), statuses and codes are exact, and the page tables
    follow the page oracle through the release and the new prefill (the
    freed pages are taken again, lowest first)."""
    o = tiny_oracle
    smp = OSampling(temperature=0.8, top_p=0.8, ras_win=10, allow_eos=True)
    lens = [30, 70, 45][:rows]
    prompts = {s: g.make_prompt(TINY, n, seed=60 + s) for s, n in enumerate(lens)}
    queued = g.make_prompt(TINY, 90, seed=69)
    slots = list(range(rows))
    pages = PageOracle(dec.max_pages, TINY.page_tokens)
    seqs = {}
    for s in slots:
        dec.prefill(s, prompts[s])
        seqs[s] = o.prefill(prompts[s])
        pages.append(s, lens[s])
    forced = g.make_forced_codes(4, rows, TINY, seed=61)
    forced[1, 0, 0] = TINY.n_sem               # slot 0 ends at frame 1
    uni = g.make_uniforms(4, rows, TINY, seed=62)
    for f in range(4):
        codes, status, slow, fast, _ = dec.decode_frame_forced(slots, dev(uni[f]), gpu_sampling(smp),
                                                               dev(forced[f]))
        dec.sync()
        codes, status = codes.cpu().numpy(), status.cpu().numpy()
        slow, fast = slow.cpu().numpy(), fast.cpu().numpy()
        for i, s in enumerate(slots):
            r = o.decode_frame(seqs[s], uni[f, i], smp, forced=forced[f, i])
            assert status[i] == r.status
            np.testing.assert_array_equal(codes[i], r.codes)
            assert_logits_close(slow[i], r.slow_logits, f"slow logits f{f} slot {s}")
            if r.status == 0:
                assert_logits_close(fast[i], r.fast_logits, f"fast logits f{f} slot {s}")
                pages.append(s, 1)
        if f == 1:
            assert status[0] == 1
            dec.release(0)
            pages.release(0)
            dec.prefill(0, queued)
            seqs[0] = o.prefill(queued)
            pages.append(0, len(queued))
        for s in slots:
            assert dec.page_table(s) == pages.table[s], f"page table of slot {s} after frame {f}"
    assert dec.slot_length(0) == len(queued) + 2


def test_eos_excluded_when_disallowed(dec):
    """allow_eos = 0 removes <|im_end|> from the q0 candidates: with greedy
    sampling and the held logits unchanged, q0 is never <|im_end|>."""
    p = g.make_prompt(TINY, 20, seed=1)
    dec.prefill(0, p)
    uni = dev(g.make_uniforms(4, 1, TINY, seed=4))
    smp = gpu_sampling(OSampling(temperature=0.0, ras_win=0, allow_eos=False))
    for f in range(4):
        codes, status = dec.decode_frame([0], uni[f], smp)
        dec.sync()
        assert status.cpu().tolist() == [0]
        assert 0 <= int(codes.cpu()[0, 0]) < TINY.n_sem


# ------------------------------------------------------------ error paths --

def test_grid_barrier_timeout_reports_error(dev_weights):
    """A grid barrier of the persistent kernel that never completes (the test
    hook asks for one arrival more than the grid has) gives up after the wait
    limit; the kernel finishes and dualar_sync reports DUALAR_ERR_TIMEOUT."""
    from dual_ar_tts_frame_gb300._lib import DualARError
    d = make(dev_weights)
    d.prefill(0, g.make_prompt(TINY, 20, seed=1))
    d.sync()
    d.set_wait_limit(20_000_000)          # 20 ms
    d.debug_barrier_extra(1)
    uni = dev(g.make_uniforms(1, 1, TINY, seed=2)[0])
    d.decode_frame([0], uni, gpu_sampling(OSampling()))
    with pytest.raises(DualARError) as e:
        d.sync()
    assert e.value.code == -6
    d.close()

def test_error_codes(dev_weights):
    from dual_ar_tts_frame_gb300._lib import DualARError
    d = make(dev_weights, max_pages=3, max_seqs=2, max_ctx=200)
    p = g.make_prompt(TINY, 128, seed=1)
    d.prefill(0, p)                                         # 2 pages
    with pytest.raises(DualARError) as e:
        d.prefill(0, p)
    assert e.value.code == -3                               # SLOT_BUSY
    with pytest.raises(DualARError) as e:
        d.prefill(1, g.make_prompt(TINY, 129, seed=1))      # needs 3 pages, 1 free
    assert e.value.code == -2                               # OOM_PAGES
    uni = dev(g.make_uniforms(1, 1, TINY, seed=2)[0])
    smp = gpu_sampling(OSampling())
    with pytest.raises(DualARError) as e:
        d.decode_frame([1], uni, smp)
    assert e.value.code == -4                               # SLOT_EMPTY
    with pytest.raises(DualARError) as e:
        d.decode_frame([0], uni, gpu_sampling(OSampling(top_p=0.0)))
    assert e.value.code == -1                               # INVALID_ARG
    with pytest.raises(DualARError) as e:
        d.prefill(1, g.make_prompt(TINY, 201, seed=1))
    assert e.value.code == -8                               # CONTEXT_FULL
    d.decode_frame([0], uni, smp)                           # position 128 takes page 3
    d.sync()
    assert d.page_table(0) == [0, 1, 2]
    d.release(0)
    d.close()


# ------------------------------------------------------ synthetic context --

def test_synthetic_context_hook(dev_weights):
    """The benchmark's context hook takes pages like prefill (lowest free
    first), sets the length, and the slot decodes (both paths)."""
    d = make(dev_weights, max_pages=32)
    pages = PageOracle(32, TINY.page_tokens)
    d.synthetic_context(2, 300, seed=5)
    pages.append(2, 300)
    p = g.make_prompt(TINY, 70, seed=6)
    d.prefill(0, p)
    pages.append(0, 70)
    assert d.slot_length(2) == 300 and d.slot_length(0) == 70
    assert d.page_table(2) == pages.table[2] and d.page_table(0) == pages.table[0]
    smp = gpu_sampling(OSampling(temperature=0.8, top_p=0.8, ras_win=10, allow_eos=False))
    uni = dev(g.make_uniforms(2, 2, TINY, seed=7))
    for f, persistent in enumerate((True, False)):
        d.set_persistent(persistent)
        codes, status = d.decode_frame([2, 0], uni[f], smp)
        d.sync()
        assert status.cpu().tolist() == [0, 0]
        c = codes.cpu().numpy()
        assert np.all((c[:, 0] >= 0) & (c[:, 0] < TINY.n_sem)) and np.all((c[:, 1:] >= 0) & (c[:, 1:] < TINY.fast_vocab))
    assert d.slot_length(2) == 302
    d.close()


# ----------------------------------------------------- tensor-core batches --

def test_teacher_forced_batch12_tensor_cores(dev_weights, tiny_oracle):
    """Twelve sequences (ragged contexts, several pages and chunks): every
    projection runs on the tensor cores (tcgen05, 9..128 rows), against the
    oracle; the same frames with the tensor cores off (GEMV passes of <= 8
    rows) agree to fp32 rounding, and two runs of the tensor-core path are
    bit-identical (the attention's dynamic unit schedule must not change
    the rounding)."""
    smp = OSampling(temperature=0.8, top_p=0.8, ras_win=10)
    prompts = {s: g.make_prompt(TINY, int(n), seed=40 + s)
               for s, n in enumerate(g.make_lengths(12, 20, 200, seed=41, stream="tc_b12"))}
    d = make(dev_weights, max_pages=128, max_seqs=16)
    run_forced(d, tiny_oracle, prompts, 3, smp, seed=42)
    d.close()
    # the two projection paths on identical inputs
    outs = []
    for tc in (True, True, False):
        d = make(dev_weights, max_pages=128, max_seqs=16)
        d.set_tensor_cores(tc)
        for s, p in prompts.items():
            d.prefill(s, p)
        forced = g.make_forced_codes(1, 12, TINY, seed=43)[0]
        uni = g.make_uniforms(1, 12, TINY, seed=44)[0]
        _, _, slow, fast, _ = d.decode_frame_forced(list(prompts), dev(uni), gpu_sampling(smp), dev(forced))
        d.sync()
        outs.append((slow.cpu().numpy(), fast.cpu().numpy()))
        d.close()
    for a, b in zip(outs[0], outs[1]):
        np.testing.assert_array_equal(a, b)
    for a, b in zip(outs[0], outs[2]):
        assert np.abs(a - b).max() <= 2e-3 * max(1.0, float(np.abs(b).max()))


# ---------------------------------------------------------- shared prefix --

def test_shared_prefix_matches_full_prompts(dev_weights, tiny_oracle):
    """A common prompt prefix (a reference voice) shared between slots: the
    full pages by reference, the partly filled one copied; each slot then
    continues its own prompt.  Every slot's state and teacher-forced frames
    equal the oracle's run of its whole prompt; a whole-sequence share equals
    its source bit for bit; page tables follow the oracle's allocator with
    shared pages, also after the source is released."""
    prefix = g.make_prompt(TINY, 150, seed=60)
    rest = {1: g.make_prompt(TINY, 40, seed=61), 2: g.make_prompt(TINY, 90, seed=62)}
    n_shared = 100                       # page 0 (positions 0..63) shared, page 1 copied
    d = make(dev_weights, max_pages=64, max_seqs=4)
    pages = PageOracle(d.max_pages, TINY.page_tokens)
    d.prefill(0, prefix)
    pages.append(0, len(prefix))
    for s, r in rest.items():
        d.share_prefix(0, s, n_shared)
        pages.share(0, s, n_shared)
        with pytest.raises(Exception):   # a bare prefix cannot decode
            d.decode_frame_forced([s], dev(np.full((1, TINY.n_codebooks + 1), 0.5, np.float32)),
                                  gpu_sampling(OSampling()), dev(np.zeros((1, TINY.n_codebooks), np.int32)))
        d.prefill_append(s, r)
        pages.append(s, len(r))
    d.share_prefix(0, 3, len(prefix))    # the whole sequence, held state included
    pages.share(0, 3, len(prefix))
    d.sync()
    for s in range(4):
        assert d.page_table(s) == pages.table[s], f"slot {s}"
    assert d.page_table(1)[0] == d.page_table(0)[0] and d.page_table(1)[1] != d.page_table(0)[1]
    prompts = {0: prefix, 1: np.concatenate([prefix[:n_shared], rest[1]]),
               2: np.concatenate([prefix[:n_shared], rest[2]]), 3: prefix}
    seqs = {s: tiny_oracle.prefill(p) for s, p in prompts.items()}
    states = {s: d.read_state(s) for s in range(4)}
    for s in range(4):
        assert_logits_close(states[s][0], seqs[s].h_last, f"hidden, slot {s}")
        assert_logits_close(states[s][1], seqs[s].z_last, f"logits, slot {s}")
    np.testing.assert_array_equal(states[3][0], states[0][0])
    np.testing.assert_array_equal(states[3][1], states[0][1])
    # the source goes away; its shared pages stay with the other slots
    d.release(0)
    pages.release(0)
    slots = [1, 2, 3]
    smp = OSampling(temperature=0.8, top_p=0.8, ras_win=10)
    forced = g.make_forced_codes(2, 3, TINY, seed=63)
    uni = g.make_uniforms(2, 3, TINY, seed=64)
    for f in range(2):
        codes, status, slow, fast, _ = d.decode_frame_forced(slots, dev(uni[f]), gpu_sampling(smp), dev(forced[f]))
        d.sync()
        slow, fast = slow.cpu().numpy(), fast.cpu().numpy()
        np.testing.assert_array_equal(status.cpu().numpy(), 0)
        for i, s in enumerate(slots):
            r = tiny_oracle.decode_frame(seqs[s], uni[f, i], smp, forced=forced[f, i])
            assert_logits_close(slow[i], r.slow_logits, f"slow logits f{f} slot {s}")
            assert_logits_close(fast[i], r.fast_logits, f"fast logits f{f} slot {s}")
            pages.append(s, 1)
    for s in slots:
        assert d.page_table(s) == pages.table[s], f"slot {s} after frames"
    d.close()


def test_shared_prefix_rejects_bad_arguments(dev_weights):
    d = make(dev_weights, max_pages=64, max_seqs=4)
    d.prefill(0, g.make_prompt(TINY, 20, seed=65))
    with pytest.raises(Exception):
        d.share_prefix(1, 2, 5)          # empty source
    with pytest.raises(Exception):
        d.share_prefix(0, 0, 5)          # same slot
    with pytest.raises(Exception):
        d.share_prefix(0, 1, 21)         # longer than the source
    d.share_prefix(0, 1, 20)
    with pytest.raises(Exception):
        d.share_prefix(0, 1, 5)          # busy destination
    with pytest.raises(Exception):
        d.prefill_append(2, g.make_prompt(TINY, 4, seed=66))   # empty slot
    d.close()
