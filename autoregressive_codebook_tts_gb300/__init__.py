"""GB300-native per-frame decode hot path for multi-codebook autoregressive TTS.

The compute path is a C-ABI shared library of hand-written CUDA kernels for sm_103a
(``csrc/``, declared in ``include/tts_decode.h``).  ``tts`` is its thin ctypes binding;
importing it loads the library and raises if it has not been built.  ``workloads``
draws the seeded synthetic inputs.
"""
__all__ = ["tts", "workloads"]
