"""Sparse MLA attention over a paged latent KV cache, for one GB300 (sm_103a)."""
