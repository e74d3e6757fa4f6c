"""GB300-native DeepSeek-V4 sparse MLA decode attention.

The compute path is the C-ABI library built from ``csrc/`` (CUDA kernels for
sm_103a); ``binding`` marshals torch tensors into that ABI.  Importing this
package does not load the shared library; the first call through
``binding`` does, and raises if it is missing.
"""
__all__ = ["binding", "workloads"]
