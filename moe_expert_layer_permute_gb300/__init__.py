"""GB300-native fused MoE expert layer (forward + backward) behind a C ABI.

The CUDA library (`libmoe_gb300.so`, built in-tree by `build.build()`) does every step of the
layer; `binding` marshals torch tensors and streams into its C entry points. Importing the package
does not load the library: `binding` loads it on import and raises if it is missing.
"""
__all__ = ["inputs", "build", "binding"]
