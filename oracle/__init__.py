"""Plain CPU oracle of the KIVI hot path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline of ``bench.py`` may use it; the product path never does.
"""
