"""Sliding-window grouped-query attention for GB300 (sm_103a).

The compute path is the CUDA library ``libswa.so`` built from ``csrc/``;
``sliding_window_gqa_swa_gb300.swa`` is its thin ctypes binding and fails
loudly when the library is missing.  ``sliding_window_gqa_swa_gb300.synth``
holds the seeded input generators.  Importing the package itself loads
nothing.
"""
