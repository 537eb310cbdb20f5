"""dualar_decode_frame_noalloc against dualar_decode_frame, through the C ABI.

The no-allocation call serves hosts that cannot let the library allocate
device memory once they are running (a fixed device budget handed over at
start-up, or the rest of the GPU already reserved by another framework).  It
must decode exactly what the ordinary call decodes: the same codes and the
same held logits and hidden state, call after call -- the fixed scratch array
it shares between calls has to be cleared and reused correctly.

This file is collected after the other parity files on purpose (only the
full-size 4-bit file comes later), so a run that stops at the first failure
has already run them.
"""
import numpy as np
import pytest

from dualar_inputs import TINY
from dualar_inputs import generators as g
from parity import assert_logits_close

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev_weights(tiny_bits):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dual_ar_tts_frame_gb300 import build, upload_weights
    build()
    return upload_weights(tiny_bits)


def test_noalloc_decode_matches_decode_frame(dev_weights):
    from dual_ar_tts_frame_gb300 import DualARDecoder, Sampling
    d = DualARDecoder(TINY, dev_weights, max_pages=32, max_seqs=4, max_ctx=512)
    # 150 positions: three split-KV chunks per KV head, so the attention
    # really goes through the partials and arrival counters in the fixed array
    prompt = g.make_prompt(TINY, 150, seed=31)
    d.prefill(0, prompt)      # decoded with dualar_decode_frame
    d.prefill(1, prompt)      # decoded with dualar_decode_frame_noalloc
    smp = Sampling(temperature=0.8, top_p=0.8, ras_win=10)
    uni = torch.from_numpy(g.make_uniforms(2, 1, TINY, seed=32)).cuda()
    codes_b = torch.empty((1, TINY.n_codebooks), dtype=torch.int32, device="cuda")
    status_b = torch.empty((1,), dtype=torch.int32, device="cuda")
    for call in range(2):     # two calls in a row share (and must clear) the array
        codes_a, status_a = d.decode_frame([0], uni[call], smp)
        d.decode_frame_noalloc([1], uni[call], smp, codes_b, status_b)
        d.sync()
        np.testing.assert_array_equal(codes_b.cpu().numpy(), codes_a.cpu().numpy())
        np.testing.assert_array_equal(status_b.cpu().numpy(), status_a.cpu().numpy())
        assert int(status_b.cpu()[0]) == 0
        ha, za = d.read_state(0)
        hb, zb = d.read_state(1)
        assert_logits_close(zb, za, f"held logits, call {call}")
        assert_logits_close(hb, ha, f"held hidden state, call {call}")
    d.close()


def test_noalloc_batch3_full_width_matches_decode_frame():
    """Three sequences at the full model width (one layer each of the slow
    and fast stacks), the largest batch the fixed array takes at that shape:
    the attention runs on the tensor cores with its partials and arrival
    counters in the array, over contexts of 11 to 46 pages (one page per
    split-KV chunk at this batch).  Two calls in a row against the ordinary
    call on copies of the same sequences."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dual_ar_tts_frame_gb300 import DualARDecoder, Sampling, build, upload_weights
    from dualar_inputs.config import S2PRO_L1
    build()
    cfg = S2PRO_L1
    w = upload_weights(g.make_weights(cfg, seed=0))
    lens = (700, 1500, 2900)
    d = DualARDecoder(cfg, w, max_pages=2 * sum(-(-(n + 4) // 64) for n in lens) + 4, max_seqs=6, max_ctx=3000)
    for i, n in enumerate(lens):
        p = g.make_prompt(cfg, n, seed=33 + i)
        d.prefill(i, p)          # decoded with dualar_decode_frame
        d.prefill(3 + i, p)      # decoded with dualar_decode_frame_noalloc
    smp = Sampling(temperature=0.8, top_p=0.8, ras_win=10, allow_eos=False)
    uni = torch.from_numpy(g.make_uniforms(2, 3, cfg, seed=36)).cuda()
    codes_b = torch.empty((3, cfg.n_codebooks), dtype=torch.int32, device="cuda")
    status_b = torch.empty((3,), dtype=torch.int32, device="cuda")
    for call in range(2):
        codes_a, status_a = d.decode_frame([0, 1, 2], uni[call], smp)
        d.decode_frame_noalloc([3, 4, 5], uni[call], smp, codes_b, status_b)
        d.sync()
        assert d.last_launch_count() > 2
        np.testing.assert_array_equal(codes_b.cpu().numpy(), codes_a.cpu().numpy())
        np.testing.assert_array_equal(status_b.cpu().numpy(), 0)
        for i in range(3):
            ha, za = d.read_state(i)
            hb, zb = d.read_state(3 + i)
            assert_logits_close(zb, za, f"held logits, row {i}, call {call}")
            assert_logits_close(hb, ha, f"held hidden state, row {i}, call {call}")
    d.close()


def test_noalloc_rejects_batches_beyond_the_array(dev_weights):
    from dual_ar_tts_frame_gb300 import DualARDecoder, Sampling
    from dual_ar_tts_frame_gb300._lib import DualARError
    d = DualARDecoder(TINY, dev_weights, max_pages=8, max_seqs=128, max_ctx=128)
    uni = torch.zeros((128, TINY.n_codebooks + 1), dtype=torch.float32, device="cuda")
    codes = torch.empty((128, TINY.n_codebooks), dtype=torch.int32, device="cuda")
    status = torch.empty((128,), dtype=torch.int32, device="cuda")
    with pytest.raises(DualARError) as e:
        d.decode_frame_noalloc(list(range(128)), uni, Sampling(), codes, status)
    assert e.value.code == -1 and "fixed array holds" in str(e.value)
    d.close()
