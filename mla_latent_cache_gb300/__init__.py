"""Absorbed MLA decode over a paged latent KV cache, native to GB300 (sm_103a)."""
