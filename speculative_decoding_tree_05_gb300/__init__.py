"""DDTree verify attention over an MLA latent KV pool, as hand-written CUDA for sm_103a."""
