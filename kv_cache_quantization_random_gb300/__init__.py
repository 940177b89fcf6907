"""TurboQuant KV-cache compression and compressed-domain decode attention for GB300.

The compute lives in a C-ABI CUDA library (``csrc/``, built for sm_103a by
``build.py``); ``binding`` marshals PyTorch tensors into its calls.  There is
no CPU fallback: if the library is missing, the binding raises.
"""

__all__ = ["workloads"]
