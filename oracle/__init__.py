"""CPU fp64 oracle of the routed MoE layer (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library shares no code with it.
"""
