"""MLA decode attention over a paged latent KV cache, for one GB300 (sm_103a).

The compute lives in a C-ABI CUDA library (csrc/, built into libmla_decode.so);
this package only marshals torch tensors into it.  See `ops` for the calls.
"""
