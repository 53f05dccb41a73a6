"""GB300-native W4A16 routed-expert MoE layer (compact INT4 experts, FP16 activations).

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
kernels (see include/moe_w4a16.h); ``moe_w4a16`` is its thin Python binding.
Importing this package does not load the library; the binding loads it on
first use and raises if it is missing.
"""
