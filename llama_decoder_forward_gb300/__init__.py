"""GB300-native pre-norm LLaMA decoder forward (SmolLM2-135M family).

The compute path lives in ``libsmol.so`` (hand-written sm_103a CUDA behind a
C ABI, declared in ``include/smol.h``).  ``smol`` is its thin ctypes binding;
``synth`` draws seeded synthetic workloads.  Importing this package does not
load the library: ``import llama_decoder_forward_gb300.smol`` does, and fails
loudly if it has not been built.
"""
