"""FP64 CPU oracle of the exact attention forward and backward passes -- test infrastructure.

Only the tests, ``__graft_entry__.smoke()`` and the CPU baseline leg of
``bench.py`` may import this package.  The CUDA path does not.
"""
