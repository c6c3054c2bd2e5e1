"""VQ3 Hadamard-rotated vector-LUT MLP for one GB300 (sm_103a).

The compute path is the C-ABI library libvq3.so (include/vq3.h); the submodule
`bit_vector_lut_gb300.vq3` is its Python binding. Build the library with
`bit_vector_lut_gb300.build.build()`.
"""
