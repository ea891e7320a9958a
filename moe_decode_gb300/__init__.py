"""GB300-native small-M MoE decode layer: a C-ABI CUDA library
(``libmoe_decode.so``) and its thin Python binding.

``moe_decode_gb300.api`` holds the binding (loads the compiled library and
fails loudly if it is missing); ``moe_decode_gb300.synth`` holds the seeded
synthetic-input generators. Importing the package itself loads nothing.
"""
