"""GB300-native hyper-connection (HC) residual mixing.

The compute path is libhcmix.so (hand-written sm_103a kernels behind a C ABI,
``include/hcmix.h``); ``binding`` is a thin ctypes layer over it.  The
library is loaded on first use and its absence raises -- there is no CPU or
PyTorch fallback.
"""
from .binding import (HcError, abi_version, hc_device_error, hc_launch_count, hc_mixes,
                      hc_mixes_pre, hc_mixes_pre_norm, hc_post, hc_post_mixes_pre, hc_pre,
                      hc_selftest_wait_timeout, hc_split_sinkhorn, hc_workspace_bytes, lib)

__all__ = ["HcError", "abi_version", "hc_device_error", "hc_launch_count", "hc_mixes",
           "hc_mixes_pre", "hc_mixes_pre_norm", "hc_post", "hc_post_mixes_pre", "hc_pre",
           "hc_selftest_wait_timeout", "hc_split_sinkhorn", "hc_workspace_bytes", "lib"]
