"""GGUF Q4_0 / Q8_0 block-quantized matrix products on GB300 (sm_103a).

The compute lives in a C-ABI shared library (``libqmm.so``, built from
``csrc/`` by :func:`block_quantized_matmul_gguf_gb300.build.build_library`);
:mod:`block_quantized_matmul_gguf_gb300.qmm` is the thin ctypes binding with
the same entry-point names.  :mod:`block_quantized_matmul_gguf_gb300.synth`
draws the seeded synthetic inputs.  Importing the package loads nothing; the
binding raises if the CUDA library is missing.
"""
__all__ = ["qmm", "synth", "build"]
