"""GB300-native paged KV-cache decode attention.

``ops`` holds the thin Python binding of the C-ABI library ``libpagedkv.so``
(write new tokens into their slots, copy-on-write block copy, paged decode
attention); ``block_manager`` is the host-side allocator; ``workloads`` and
``scenarios`` build seeded synthetic inputs.  Importing the package does not
load the CUDA library; ``ops`` does, and fails loudly if it is missing.
"""

__all__ = ["ops", "block_manager", "workloads", "scenarios"]
