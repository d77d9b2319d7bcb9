"""GB300-native decode-step MLA over a sequence-sharded latent KV cache.

The compute path is the CUDA library ``libmla_dcp.so`` (C ABI in
include/mla_dcp.h, built in-tree by ``build.build()``).  ``api`` binds it for
torch CUDA tensors; ``inputs`` draws seeded synthetic workloads.  Importing
this package does not import torch or load the library.
"""
__all__ = ["api", "inputs", "build"]
