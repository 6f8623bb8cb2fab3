"""CPU oracle of the parameter-preparation stage.

TEST INFRASTRUCTURE ONLY. The plain, slow, obviously correct definition
the CUDA library is checked against; only tests/, the smoke check and the
benchmark's CPU-baseline leg import it. It shares no code with the product
library and never imports it.
"""
from .oracle import (OFFSET_AUTO, Model, build, e4m3_decode, e4m3_encode,
                     e4m3_encode_bits_range, quantize_element, quantize_tokens, tile_scale)

__all__ = ["OFFSET_AUTO", "Model", "build", "e4m3_decode", "e4m3_encode",
           "e4m3_encode_bits_range", "quantize_element", "quantize_tokens", "tile_scale"]
