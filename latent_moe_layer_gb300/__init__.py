"""GB300-native forward of the Kimi K3 latent routed-MoE layer.

The CUDA library (``libk3moe.so``) is loaded lazily by ``latent_moe_layer_gb300.k3moe``
so that the seeded generator (``latent_moe_layer_gb300.synth``) can be imported on
machines without the built extension.
"""
