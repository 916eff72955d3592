"""Block-wise masked-diffusion denoise step for GB300 (sm_103a).

The compute lives in the C-ABI library ``libbd.so`` (CUDA, built from
``csrc/``); ``bd`` is its thin ctypes binding.  ``workload`` draws the seeded
synthetic inputs.  Importing this package does not load the library; the
first call into ``bd`` does, and fails loudly if it has not been built.
"""
MASK = -1
