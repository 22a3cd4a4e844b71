"""gemm_conv_chains_gb300: fused GEMM/conv operator chains for one GB300 (sm_103a).

The compute lives in libb2b.so (C ABI, include/b2b.h); this package is its thin binding:
``ops`` marshals torch tensors into the C calls, ``workloads`` draws the seeded synthetic
inputs, ``build`` compiles the library in-tree with nvcc.
"""
from .ops import (B2BError, b2b_conv_nhwc, b2b_gemm, conv_bias_act_nhwc, conv_relu_maxpool,
                  gemm_bias_act, get_device_error, maxpool2x2_nhwc, num_sms, pad_channels,
                  probe_timeout, set_wait_limit_ns, status_str, version)

__all__ = ["B2BError", "b2b_gemm", "b2b_conv_nhwc", "conv_relu_maxpool", "gemm_bias_act",
           "conv_bias_act_nhwc", "maxpool2x2_nhwc", "get_device_error", "num_sms",
           "pad_channels", "probe_timeout", "set_wait_limit_ns", "status_str", "version"]
