"""GB300-native forward pass of the complex-valued chunkwise SSD scan.

The compute path lives in ``libssdc.so`` (hand-written CUDA for sm_103a behind
a C ABI declared in ``include/ssdc.h``). ``ssdc`` is the thin ctypes binding;
``inputs`` draws the seeded synthetic workloads. Importing the package loads
nothing: the library is opened on first use, and a missing library is an error.
"""

__all__ = ["inputs", "ssdc"]
