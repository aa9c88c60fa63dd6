"""Seeded synthetic inputs for the NVFP4 fused-MoE forward pass.

This package holds input preparation only: random draws, the model-load
NVFP4 quantisation of weights and activations, and routing draws.  None of
the forward pass itself (routing plan, GEMMs, SwiGLU, finalize) lives here.
Both the CUDA path and the CPU oracle consume what it produces.
"""
from .moe_inputs import (ACTIVATIONS, CONFIGS, MoEConfig, MoEInputs, activation_spec,  # noqa: F401
                         generate, generate_routing, route_tile_for)
