"""Full-size parity: the S2-Pro-shaped model at batch 1 against the CPU oracle.

The decoder runs in the launch configuration the benchmark times: one slot,
the persistent frame kernel, with the benchmark's weights (seed 0), its
512-token prompt (seed 0), its uniforms (seed 1) and its sampling (T 0.8,
top-p 0.8, repetition-aware window 10, <|im_end|> excluded).  The oracle
computes the same frames one by one on the host:

- the state left by the prefill (final-normed hidden, restricted logits),
  and, printed beside it, the distance of the GPU's prefill logits from an
  oracle whose slow cache stays float32 instead of bf16;
- three sampled frames, then two greedy ones (T = 0, no resample),
  replayed in the oracle along the GPU's trajectory:
  slow and fast logits within the tolerance; every GPU draw equal to the
  oracle sampler's draw from the GPU's own logits (exact: the integer
  arithmetic of the draw is fixed); the committed codes equal to the
  oracle's own draws wherever those are stable under the measured logit
  difference (tests/parity.py: draw_decidable; for the greedy frames,
  wherever the oracle's top-1/top-2 gap exceeds max(0.1, 2 eps)).

The oracle needs ~30 GB of host memory and a minute or two of CPU time.
"""
import numpy as np
import pytest

from dualar_inputs import S2PRO
from dualar_inputs import generators as g
from oracle import DualAROracle, Sampling as OSampling
from oracle.sampler import sample_q0, sample_top_p
from parity import DrawStats, assert_logits_close, draw_decidable

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
torch = pytest.importorskip("torch")

PROMPT = 512
N_SAMPLED = 3
N_GREEDY = 2
N_FRAMES = N_SAMPLED + N_GREEDY


def test_s2pro_b1_prefill_sampled_and_greedy_frames_match_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dual_ar_tts_frame_gb300 import DualARDecoder, Sampling, build, upload_weights
    build()
    cfg = S2PRO
    bits = g.make_weights(cfg, seed=0)
    prompt = g.make_prompt(cfg, PROMPT, seed=0)
    uni = g.make_uniforms(N_FRAMES, 1, cfg, seed=1)
    sampled = OSampling(temperature=0.8, top_p=0.8, ras_win=10, allow_eos=False)
    greedy = OSampling(temperature=0.0, top_p=0.8, ras_win=0, allow_eos=False)
    plan = [sampled] * N_SAMPLED + [greedy] * N_GREEDY

    def gpu_sampling(o):
        return Sampling(o.temperature, o.top_p, o.ras_win, o.allow_eos, o.ras_temperature, o.ras_top_p)

    # ---- GPU: prefill, then sampled frames through the frame kernel
    w = upload_weights(bits)
    max_ctx = PROMPT + N_FRAMES + 8
    d = DualARDecoder(cfg, w, max_pages=2 * ((max_ctx + 63) // 64) + 2, max_seqs=2, max_ctx=max_ctx)
    d.prefill(0, prompt)
    gh, gz = d.read_state(0)
    frames = []
    for f in range(N_FRAMES):
        codes, status, slow, fast, draws = d.decode_frame_forced([0], torch.from_numpy(uni[f]).cuda(),
                                                                 gpu_sampling(plan[f]), None)
        d.sync()
        frames.append((codes.cpu().numpy()[0], int(status.cpu()[0]), slow.cpu().numpy()[0],
                       fast.cpu().numpy()[0], draws.cpu().numpy()[0]))
    assert d.last_launch_count() <= 2, "batch 1 must run as the persistent frame kernel"
    d.close()
    del w
    torch.cuda.empty_cache()

    # ---- oracle: the same prompt, then the GPU's trajectory
    o = DualAROracle(cfg, bits, max_pos=max_ctx)
    seq = o.prefill(prompt)
    assert_logits_close(gh, seq.h_last, "prefill hidden")
    assert_logits_close(gz, seq.z_last, "prefill logits")
    # What the bf16 slow-cache reading is worth: the same prefill with a
    # float32 cache, reported (not asserted) against the GPU.
    o.slow_kv_bf16 = False
    z32 = o.prefill(prompt).z_last
    o.slow_kv_bf16 = True
    d32 = np.asarray(gz, np.float64) - z32
    dbf = np.asarray(gz, np.float64) - seq.z_last
    print(f"prefill logits vs oracle: bf16 cache max abs {np.abs(dbf).max():.4g} rel L2 "
          f"{np.linalg.norm(dbf) / np.linalg.norm(seq.z_last):.3g}; float32 cache max abs "
          f"{np.abs(d32).max():.4g} rel L2 {np.linalg.norm(d32) / np.linalg.norm(z32):.3g}")
    stats = DrawStats()      # oracle logits, draws stable under the measured eps
    samp = DrawStats()       # oracle sampler on the GPU's own logits
    greedy_compared = 0
    for f, (codes, status, slow, fast, draws) in enumerate(frames):
        smp = plan[f]
        assert status == 0
        hist = list(seq.history)
        g0, gr, gch = sample_q0(cfg, slow, smp, hist, float(uni[f, 0, 0]), float(uni[f, 0, 1]))
        samp.check(draws[0], g0, smp.temperature, f"q0 draw f{f}")
        samp.check(draws[1], gr, smp.ras_temperature, f"ras draw f{f}")
        if draw_decidable(g0, smp.temperature) and draw_decidable(gr, smp.ras_temperature):
            assert draws[2] == gch and codes[0] == gch
        for k in range(1, cfg.n_codebooks):
            rk = sample_top_p(fast[k - 1], np.arange(cfg.fast_vocab), smp.temperature, smp.top_p,
                              float(uni[f, 0, k + 1]))
            samp.check(codes[k], rk, smp.temperature, f"q{k} draw f{f}")
        r = o.decode_frame(seq, uni[f, 0], smp, forced=codes)
        n0, ras, chosen = r.draws[0]
        assert_logits_close(slow, r.slow_logits, f"slow logits f{f}")
        assert_logits_close(fast, r.fast_logits, f"fast logits f{f}")
        eps0 = float(np.abs(slow - r.slow_logits).max())
        triggered = smp.ras_win > 0 and n0.index in hist[-smp.ras_win:]
        if draw_decidable(n0, smp.temperature, eps0) and (
                not triggered or draw_decidable(ras, smp.ras_temperature, eps0)):
            stats.compared += 1
            assert codes[0] == chosen, f"q0 f{f}: gpu {codes[0]} oracle {chosen}"
        else:
            stats.excluded += 1
        for k in range(1, cfg.n_codebooks):
            epsk = float(np.abs(fast[k - 1] - r.fast_logits[k - 1]).max())
            before = stats.compared
            stats.check(codes[k], r.draws[k], smp.temperature, f"q{k} f{f}", epsk)
            if smp.temperature <= 0:
                greedy_compared += stats.compared - before
    assert samp.compared > 0
    assert greedy_compared > 0
    print(f"full size: draws on oracle logits {stats.compared} compared / {stats.excluded} not stable; "
          f"sampler on GPU logits {samp.compared} compared / {samp.excluded} at a boundary")
