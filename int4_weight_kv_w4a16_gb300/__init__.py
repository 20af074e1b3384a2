"""GB300 (sm_103a) INT4-weight / INT4-KV decode block.

The compute path is the C-ABI library ``libfutr.so`` built from ``csrc/``;
``futr`` is its thin ctypes binding.  Importing this package does not load the
library; ``futr.lib()`` does, and raises if it has not been built.
"""
__all__ = ["futr", "inputs"]
