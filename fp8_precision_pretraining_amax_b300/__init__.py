"""Block-scaled FP8 linear layer for B300 (sm_103a).

  fp8bq   -- Python binding of the C ABI in include/fp8bq.h (libfp8bq.so):
             quantizers (row-wise 1x128, column-wise 128x1, weight 128x128)
             and the Fprop / Dgrad / Wgrad GEMMs on tcgen05 tensor cores
  linear  -- LinearFP8: one linear layer's forward/backward on that path
  synth   -- seeded synthetic inputs (no arithmetic of the method)
  build   -- nvcc build of libfp8bq.so

Importing `fp8bq` or `linear` loads the CUDA library and fails loudly if it
has not been built; `synth` and `build` do not need it.
"""
