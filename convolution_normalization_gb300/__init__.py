"""GB300-native fused convolution + normalization forward (sm_103a).

The compute path is the C-ABI library ``libconv_norm.so`` (see
``include/conv_norm.h``); ``binding`` is its thin ctypes binding.  Importing
``binding`` fails loudly when the library has not been built; build it with
``python -m convolution_normalization_gb300.build``.
"""
__all__ = ["binding", "build", "workloads"]
