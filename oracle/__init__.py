"""Float64 CPU oracle of the LatentMoE layer forward: test infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline and
reference legs of ``bench.py`` may import this package. It shares no code
with the CUDA library and never imports it.
"""
