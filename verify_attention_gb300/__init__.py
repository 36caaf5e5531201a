"""GB300 FP8 paged KV cache: E4M3 insert and exact decode/verifier attention.

The compute path is the C-ABI library ``libfp8kv.so`` (hand-written CUDA for
sm_103a, ``csrc/``); ``fp8kv`` is its thin ctypes binding.  Importing this
package does not load the library; the first call does, and fails loudly if
it is missing.
"""
__all__ = ["fp8kv", "inputs"]
