"""Full-size parity at batches 16, 64 and 128: the S2-Pro-shaped model in the
launch configuration of the benchmark's batch-64 line (the per-op path:
tcgen05 projections with the batch padded to 16, 64 or 128 rows, the
tensor-core paged attention over all sequences, programmatic dependent
launches), checked against the CPU oracle on sampled sequences.

The prompts (lengths uniform in [64, 320], [64, 192] at batch 128; seed 7) are
prefilled (chunks of up to 128 rows on the tensor cores), then two
teacher-forced frames run for the whole batch (T 0.8, top-p 0.8,
repetition-aware window 10, <|im_end|> excluded).  The oracle replays two of
the sequences one by one:

- the state the prefill leaves (final-normed hidden, restricted logits);
- slow and fast logits of both frames within the tolerance;
- every GPU draw equal to the oracle sampler's draw from the GPU's own logits
  (the integer arithmetic of the draw is fixed);
- the page tables of all slots bit-exact against the oracle's allocator.

The oracle needs ~30 GB of host memory and well under a minute of CPU time.
"""
import numpy as np
import pytest

from dualar_inputs import S2PRO
from dualar_inputs import generators as g
from oracle import DualAROracle, PageOracle, Sampling as OSampling
from oracle.sampler import sample_q0, sample_top_p
from parity import DrawStats, assert_logits_close

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
torch = pytest.importorskip("torch")

FRAMES = 2


@pytest.mark.parametrize("batch", [16, 64, 128])
def test_s2pro_batch_sampled_sequences_match_oracle(batch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dual_ar_tts_frame_gb300 import DualARDecoder, Sampling, build, upload_weights
    build()
    cfg = S2PRO
    bits = g.make_weights(cfg, seed=0)
    lens = g.make_lengths(batch, 64, 320 if batch <= 64 else 192, seed=7, stream=f"b{batch}_parity")
    sampled = (0, batch * 5 // 7)
    prompts = {s: g.make_prompt(cfg, int(n), seed=100 + s) for s, n in enumerate(lens)}
    forced = g.make_forced_codes(FRAMES, batch, cfg, seed=8)
    uni = g.make_uniforms(FRAMES, batch, cfg, seed=9)
    smp = OSampling(temperature=0.8, top_p=0.8, ras_win=10, allow_eos=False)
    gsmp = Sampling(smp.temperature, smp.top_p, smp.ras_win, smp.allow_eos, smp.ras_temperature, smp.ras_top_p)

    # ---- GPU: all 64 sequences
    w = upload_weights(bits)
    max_ctx = int(lens.max()) + FRAMES + 8
    max_pages = sum(-(-(int(n) + FRAMES + 1) // cfg.page_tokens) for n in lens) + 8
    d = DualARDecoder(cfg, w, max_pages=max_pages, max_seqs=batch, max_ctx=max_ctx)
    pages = PageOracle(max_pages, cfg.page_tokens)
    for s, p in prompts.items():
        d.prefill(s, p)
        pages.append(s, len(p))
    states = {s: d.read_state(s) for s in sampled}
    slots = list(range(batch))
    frames = []
    for f in range(FRAMES):
        codes, status, slow, fast, draws = d.decode_frame_forced(slots, torch.from_numpy(uni[f]).cuda(), gsmp,
                                                                 torch.from_numpy(forced[f]).cuda())
        d.sync()
        assert d.last_launch_count() > 2, "batches above 2 run on the per-op path"
        codes, status = codes.cpu().numpy(), status.cpu().numpy()
        np.testing.assert_array_equal(codes, forced[f])
        np.testing.assert_array_equal(status, 0)
        frames.append((slow.cpu().numpy(), fast.cpu().numpy(), draws.cpu().numpy()))
        for s in slots:
            pages.append(s, 1)
    for s in slots:
        assert d.page_table(s) == pages.table[s], f"page table of slot {s}"
        assert d.slot_length(s) == len(prompts[s]) + FRAMES
    d.close()
    del w
    torch.cuda.empty_cache()

    # ---- oracle: the sampled sequences, one by one
    o = DualAROracle(cfg, bits, max_pos=max_ctx)
    samp = DrawStats()
    for s in sampled:
        seq = o.prefill(prompts[s])
        gh, gz = states[s]
        assert_logits_close(gh, seq.h_last, f"prefill hidden, slot {s}")
        assert_logits_close(gz, seq.z_last, f"prefill logits, slot {s}")
        for f, (slow, fast, draws) in enumerate(frames):
            hist = list(seq.history)
            n0, ras, _ = sample_q0(cfg, slow[s], smp, hist, float(uni[f, s, 0]), float(uni[f, s, 1]))
            samp.check(draws[s, 0], n0, smp.temperature, f"q0 draw f{f} slot {s}")
            samp.check(draws[s, 1], ras, smp.ras_temperature, f"ras draw f{f} slot {s}")
            for k in range(1, cfg.n_codebooks):
                rk = sample_top_p(fast[s, k - 1], np.arange(cfg.fast_vocab), smp.temperature, smp.top_p,
                                  float(uni[f, s, k + 1]))
                samp.check(draws[s, k + 2], rk, smp.temperature, f"q{k} draw f{f} slot {s}")
            r = o.decode_frame(seq, uni[f, s], smp, forced=forced[f, s])
            assert_logits_close(slow[s], r.slow_logits, f"slow logits f{f} slot {s}")
            assert_logits_close(fast[s], r.fast_logits, f"fast logits f{f} slot {s}")
    assert samp.compared > 0
    print(f"batch {batch}: sampler on GPU logits {samp.compared} compared / {samp.excluded} at a boundary")
