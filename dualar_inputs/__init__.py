"""Shapes and seeded synthetic inputs shared by the oracle and the CUDA path.

Nothing here computes any step of the Dual-AR decode."""
from .config import DualARConfig, TINY, S2PRO, CONFIGS, FRAMES_PER_AUDIO_SECOND  # noqa: F401
from . import generators  # noqa: F401
