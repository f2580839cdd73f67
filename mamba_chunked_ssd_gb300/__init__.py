"""GB300 (sm_103a) Mamba-2 chunked SSD forward pass.

The compute lives in libmamba2ssd.so (CUDA kernels behind the C ABI declared
in include/mamba2_ssd.h); ``binding`` is its thin Python binding and
``synthetic`` draws seeded workload inputs.  Import ``binding`` explicitly:
this package module itself loads nothing so that CPU-only tools can use
``synthetic`` without the CUDA library.
"""
__all__ = ["binding", "synthetic", "build_lib"]
