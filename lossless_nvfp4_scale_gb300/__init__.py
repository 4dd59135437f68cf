"""GB300-native lossless CSF decoding of NVFP4 / MXFP4 MoE weight-scale planes.

Submodules:
  csf    -- Python binding of the C-ABI CUDA library (prepare, decode,
            paired decode); it raises if the compiled library is missing.
  synth  -- seeded synthetic scale stacks and routing prefixes.

Importing the package loads nothing; ``import lossless_nvfp4_scale_gb300.csf``
loads the CUDA library.
"""
__all__ = ["csf", "synth"]
