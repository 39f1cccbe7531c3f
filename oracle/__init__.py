"""CPU oracle of the GDN hot path: test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The library never does.
"""
