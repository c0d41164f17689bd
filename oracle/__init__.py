"""CPU fp64 oracle of the joint audio-video attention sub-block.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by
the benchmark's CPU-baseline leg, never by the CUDA library or its binding.
"""
from .h3_oracle import (MOD_AUDIO, MOD_TEXT, MOD_VIDEO, adaln_modulate,
                        attention, attention_varlen, block, block_rows, denoise_step,
                        gated_residual, gelu_tanh, mlp_block, sigma_to_t_h3,
                        layer_norm, linear, mrope, packed_layout, rope_angles,
                        rope_rotate_heads)

__all__ = ["MOD_TEXT", "MOD_VIDEO", "MOD_AUDIO", "packed_layout", "layer_norm",
           "adaln_modulate", "linear", "rope_angles", "rope_rotate_heads",
           "mrope", "attention", "attention_varlen", "gated_residual", "block", "block_rows",
           "denoise_step", "sigma_to_t_h3", "gelu_tanh", "mlp_block"]
