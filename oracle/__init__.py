"""fp64 CPU oracle for exact attention: TEST INFRASTRUCTURE ONLY.

Only tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
``--impl reference`` legs may import this package. It shares no code with the CUDA
path and imports nothing from it.
"""
