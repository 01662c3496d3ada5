"""fp64 CPU oracle of the latent routed-MoE layer (test infrastructure only)."""
