"""GB300-native stride-1, pad-1 3x3 convolution: forward (fused bias + SiLU),
input gradient and weight gradient behind the C ABI of ``libconv3x3.so``.

``x3_convolution_gb300._lib`` holds the ctypes binding (same names as the C
entry points); ``x3_convolution_gb300.ops`` wraps it for torch tensors.
"""
from ._lib import (ACT_LRELU, ACT_NONE, ACT_SILU, DT_BF16, DT_F32, PATH_AUTO, PATH_SIMT, PATH_TENSOR,
                   Conv3x3Error, load)

__all__ = ["ACT_LRELU", "ACT_NONE", "ACT_SILU", "DT_BF16", "DT_F32", "PATH_AUTO", "PATH_SIMT", "PATH_TENSOR",
           "Conv3x3Error", "load"]
