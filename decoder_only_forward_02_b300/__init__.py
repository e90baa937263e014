"""B300 (sm_103a) forward pass of a nanochat-style decoder-only GPT behind a C ABI.

``binding.Model`` wraps ``nc_model_create`` / ``nc_forward`` of the in-tree ``libnc.so``;
``build.build()`` compiles it.  Importing this package does not load the library.
"""
__all__ = ["build", "binding"]
