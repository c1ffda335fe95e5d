"""QuantWM 2-bit KV cache on GB300: CUDA kernels behind the libqwm C ABI.

`qwm` is the ctypes binding of the library (include/qwm.h); `build` compiles
it for sm_103a; `synth` draws the seeded synthetic workloads.
"""
from . import synth  # noqa: F401

__all__ = ["synth", "qwm", "build"]
