"""B300 (sm_103a) top-k Mixture-of-Experts layer forward behind a small C ABI.

``moe`` is the ctypes binding of ``include/moe.h``; ``synth`` makes seeded inputs;
``build`` compiles the library in-tree.
"""
