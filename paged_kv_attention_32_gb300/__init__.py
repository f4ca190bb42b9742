"""GB300 (sm_103a) paged-KV decode attention and ragged causal prefill.

The compute path is the C-ABI library ``_lib/libpka.so`` (hand-written CUDA);
``api`` is its thin Python binding.  ``workloads`` draws seeded synthetic
inputs.  Importing the package does not load the library; the first API call
does, and raises if it is missing.
"""

__all__ = ["api", "workloads", "build"]
