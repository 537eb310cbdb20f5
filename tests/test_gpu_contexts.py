"""Parity at the batch configurations' own context lengths, every row.

The one-layer, full-width model (S2-Pro layer shapes: dim 2560, 32/8 heads
of 128, FFN 9728, 4,096 semantic ids, N = 10) runs the batch workloads'
context lengths, so the decode attention is planned exactly as in the
full-size runs (the chunk plan depends on the contexts, the batch and the
SM count, not on the depth): batch 16 with contexts uniform in [512, 2048];
batch 64 with the batch-64 benchmark's contexts (uniform in [1024, 4096],
seed 3); batch 128 with the replacement workload's initial contexts (124
uniform in [2048, 4096] and 4 of 16,384, seed 4).  That takes the split-KV
attention to chunks of 2 to 48 pages and the 16K contexts through several
chunks each.

Every sequence is prefilled for real, then two teacher-forced frames run
for the whole batch (T 0.8, top-p 0.8, repetition-aware window 10,
<|im_end|> excluded).  For EVERY row the oracle (a spawn pool of workers)
replays the same prompt and frames, and the test checks:

- frame 0's slow logits (the prefill's) and the prefill's hidden state;
- frame 0's and frame 1's fast logits, frame 1's slow logits (the first
  decode position's attention over the whole context) and the state after
  frame 1 (the second one's), all within the tolerance;
- the page tables of all slots bit-exact against the page oracle;
- on a few rows, every GPU draw against the oracle sampler on the GPU's own
  logits (exact: the integer arithmetic of the draw is fixed).

At batch 128 eight sequences then finish: their slots are released and
restarted from queued prompts (prefilled), and a third frame runs for the
whole batch; the restarted rows are compared with fresh oracle runs.
"""
import numpy as np
import pytest

from dualar_inputs import generators as g
from dualar_inputs.config import S2PRO_L1
from oracle import PageOracle, Sampling as OSampling
from oracle import model as om
from oracle.sampler import sample_q0, sample_top_p
from oracle_pool import pool, run_sequence
from parity import DrawStats, assert_logits_close

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
torch = pytest.importorskip("torch")

FRAMES = 2
SMP = dict(temperature=0.8, top_p=0.8, ras_win=10, allow_eos=False)


def case_contexts(name: str) -> np.ndarray:
    if name == "b16":
        return g.make_lengths(16, 512, 2048, seed=2, stream="ctx_b16")
    if name == "b64":
        return g.make_lengths(64, 1024, 4096, seed=3, stream="ctx_b64")
    return np.asarray(g.make_replacement_workload(128, 4, 512, seed=4)["ctx"])


def _gpu_sampling():
    from dual_ar_tts_frame_gb300 import Sampling
    s = OSampling(**SMP)
    return Sampling(s.temperature, s.top_p, s.ras_win, s.allow_eos, s.ras_temperature, s.ras_top_p)


@pytest.mark.parametrize("name", ["b16", "b64", "b128"])
def test_every_row_matches_oracle_at_config_contexts(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dual_ar_tts_frame_gb300 import DualARDecoder, build, upload_weights
    build()
    cfg = S2PRO_L1
    ctx = case_contexts(name)
    b = ctx.size
    prompts = [g.make_prompt(cfg, int(n), seed=20_000 + s, stream=f"ctx_prompt_{name}") for s, n in enumerate(ctx)]
    forced = g.make_forced_codes(FRAMES + 1, b, cfg, seed=21)
    uni = g.make_uniforms(FRAMES + 1, b, cfg, seed=22)
    replaced, new_prompts = [], {}
    if name == "b128":
        wl = g.make_replacement_workload(128, 4, 512, seed=4)
        replaced = [int(s) for s in np.argsort(np.asarray(wl["finish"])[:124], kind="stable")[:8]]
        new_prompts = {s: g.make_prompt(cfg, int(wl["queue_ctx"][i]), seed=30_000 + i, stream="ctx_queue")
                       for i, s in enumerate(replaced)}
    max_ctx = max([int(ctx.max())] + [len(p) for p in new_prompts.values()]) + FRAMES + 8

    # ---- oracle, every row, in worker processes while the GPU runs
    workers = pool(cfg.name, max_pos=max_ctx + 8)
    jobs = [workers.apply_async(run_sequence, ({"prompt": prompts[s], "forced": forced[:FRAMES, s],
                                                "uniforms": uni[:FRAMES, s], "sampling": SMP},))
            for s in range(b)]
    rjobs = {s: workers.apply_async(run_sequence, ({"prompt": new_prompts[s], "forced": forced[FRAMES:, s],
                                                    "uniforms": uni[FRAMES:, s], "sampling": SMP},))
             for s in replaced}
    workers.close()

    try:
        # ---- GPU
        w = upload_weights(g.make_weights(cfg, seed=0))
        per = lambda n: -(-(int(n) + FRAMES + 2) // cfg.page_tokens)  # noqa: E731
        max_pages = sum(per(n) for n in ctx) + sum(per(len(p)) for p in new_prompts.values()) + 8
        d = DualARDecoder(cfg, w, max_pages=max_pages, max_seqs=b, max_ctx=max_ctx)
        pages = PageOracle(max_pages, cfg.page_tokens)
        for s in range(b):
            d.prefill(s, prompts[s])
            pages.append(s, len(prompts[s]))
        slots = list(range(b))
        gsmp = _gpu_sampling()
        frames = []
        for f in range(FRAMES):
            codes, status, slow, fast, draws = d.decode_frame_forced(slots, torch.from_numpy(uni[f]).cuda(), gsmp,
                                                                     torch.from_numpy(forced[f]).cuda())
            d.sync()
            assert d.last_launch_count() > 2, "batches above 2 run on the per-op path"
            np.testing.assert_array_equal(codes.cpu().numpy(), forced[f])
            np.testing.assert_array_equal(status.cpu().numpy(), 0)
            frames.append((slow.cpu().numpy(), fast.cpu().numpy(), draws.cpu().numpy()))
            for s in slots:
                pages.append(s, 1)
        end = [d.read_state(s) for s in slots]
        for s in slots:
            assert d.page_table(s) == pages.table[s], f"page table of slot {s}"
            assert d.slot_length(s) == len(prompts[s]) + FRAMES
        if replaced:
            # sequences finish: release, restart from the queue, decode once more
            for s in replaced:
                d.release(s)
                pages.release(s)
            for s in replaced:
                d.prefill(s, new_prompts[s])
                pages.append(s, len(new_prompts[s]))
            codes, status, slow3, fast3, _ = d.decode_frame_forced(slots, torch.from_numpy(uni[FRAMES]).cuda(),
                                                                   gsmp, torch.from_numpy(forced[FRAMES]).cuda())
            d.sync()
            np.testing.assert_array_equal(codes.cpu().numpy(), forced[FRAMES])
            np.testing.assert_array_equal(status.cpu().numpy(), 0)
            slow3, fast3 = slow3.cpu().numpy(), fast3.cpu().numpy()
            for s in slots:
                pages.append(s, 1)
                assert d.page_table(s) == pages.table[s], f"page table of slot {s} after replacement"
        d.close()
        del w
        torch.cuda.empty_cache()

        # ---- compare every row
        smp = OSampling(**SMP)
        samp = DrawStats()
        worst = [0.0, 0.0]
        for s in slots:
            r = jobs[s].get(timeout=1800)
            gh, gz = end[s]
            checks = [(frames[0][0][s], r["z0"], "slow logits f0 (prefill)"),
                      (frames[0][1][s], r["fast"][0], "fast logits f0"),
                      (frames[1][0][s], r["slow"][1], "slow logits f1"),
                      (frames[1][1][s], r["fast"][1], "fast logits f1"),
                      (gh, r["h_end"], "hidden after f1"),
                      (gz, r["z_end"], "logits after f1")]
            for got, ref, what in checks:
                e, rel = assert_logits_close(got, ref, f"{what}, slot {s} (context {ctx[s]})")
                worst = [max(worst[0], e), max(worst[1], rel)]
            if s in (0, b // 3, b - 1):
                hist = []
                for f, (slow, fast, draws) in enumerate(frames):
                    n0, ras, _ = sample_q0(cfg, slow[s], smp, hist, float(uni[f, s, 0]), float(uni[f, s, 1]))
                    samp.check(draws[s, 0], n0, smp.temperature, f"q0 draw f{f} slot {s}")
                    samp.check(draws[s, 1], ras, smp.ras_temperature, f"ras draw f{f} slot {s}")
                    for k in range(1, cfg.n_codebooks):
                        rk = sample_top_p(fast[s, k - 1], np.arange(cfg.fast_vocab), smp.temperature, smp.top_p,
                                          float(uni[f, s, k + 1]))
                        samp.check(draws[s, k + 2], rk, smp.temperature, f"q{k} draw f{f} slot {s}")
                    hist.append(int(forced[f, s, 0]))
        for s in replaced:
            r = rjobs[s].get(timeout=1800)
            assert_logits_close(slow3[s], r["z0"], f"slow logits of restarted slot {s}")
            assert_logits_close(fast3[s], r["fast"][0], f"fast logits of restarted slot {s}")
        assert samp.compared > 0
        print(f"{name}: {b} rows, contexts {int(ctx.min())}..{int(ctx.max())}; worst max abs {worst[0]:.3g}, "
              f"rel L2 {worst[1]:.3g}; {len(replaced)} restarted; draws {samp.compared} compared / "
              f"{samp.excluded} at a boundary")
    finally:
        workers.terminate()
        workers.join()


def test_rope_table_bit_exact_to_16k_positions():
    """The GPU's bf16 RoPE tables at head_dim 128 equal the oracle's bit for
    bit over 16,400 positions (the 16K contexts of the batch-128 workload)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dual_ar_tts_frame_gb300 import DualARDecoder, build, upload_weights
    build()
    cfg = S2PRO_L1
    w = upload_weights(g.make_weights(cfg, seed=0))
    n = 16_400
    d = DualARDecoder(cfg, w, max_pages=8, max_seqs=1, max_ctx=n)
    c, s = d.rope_table(n)
    d.close()
    oc, os_ = om.rope_table(n, cfg.head_dim, cfg.rope_base)
    np.testing.assert_array_equal(c, (oc.view(np.uint32) >> 16).astype(np.uint16))
    np.testing.assert_array_equal(s, (os_.view(np.uint32) >> 16).astype(np.uint16))
