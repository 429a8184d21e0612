"""Seeded synthetic inputs for the NVFP4 W4A16 MoE layer.

This package is shared by the CPU oracle's tests and by the GPU path's tests and
benchmark.  It holds no arithmetic of the layer itself: it only draws random
activations, routing decisions and weights, and encodes the weights into the
NVFP4 storage format (E2M1 nibbles, E4M3 block scales, fp32 global scale) that
both sides then read byte for byte.
"""

from .gen import (CONFIGS, PROFILE_CONFIGS, LayerConfig, LayerInputs, config_by_name,  # noqa: F401
                  make_inputs, quantize_nvfp4)
