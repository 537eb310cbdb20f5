"""CPU oracle of the Dual-AR per-frame decode.

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and the CPU
baseline leg of bench.py may import this package.  It shares no code with
the CUDA library (dual_ar_tts_frame_gb300); both take their inputs from the
seeded generator in dualar_inputs.

Every function is pinned by a `-m "not gpu"` test against the pages'
figures, closed forms, brute force or library routines; see the module
docstrings for the passages each function follows.
"""
from .model import (DualAROracle, SeqState, Sampling, FrameResult, rmsnorm,  # noqa: F401
                    rope_table, apply_rope, gqa_attention, silu, block)
from .sampler import SampleResult, sample_top_p, sample_q0, q0_candidates  # noqa: F401
from .pages import PageOracle  # noqa: F401
