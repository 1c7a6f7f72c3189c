"""GB300 lockstep frame step of a Moshi-class full-duplex speech model.

The compute path is the CUDA library ``libmfs.so`` (C ABI: include/mfs.h);
``full_duplex_speech_frame_gb300.mfs`` is its Python binding.
"""
from .build import build  # noqa: F401
