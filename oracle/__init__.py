"""CPU oracle of the W4A16 routed-expert MoE layer (test infrastructure only).

Only tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.
"""
