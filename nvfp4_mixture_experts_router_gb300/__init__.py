"""GB300-native NVFP4 Mixture-of-Experts layer forward.

The compute lives in libmoe_nvfp4.so (hand-written sm_103a CUDA kernels
behind a C ABI, see include/moe_nvfp4.h); ``api`` is its ctypes binding,
``synth`` the seeded synthetic inputs, ``build`` the in-tree nvcc build.
"""
__all__ = ["api", "synth", "build"]
