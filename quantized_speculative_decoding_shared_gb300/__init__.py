"""QSPEC hot path on GB300 (sm_103a): one shared INT4 weight set, a W4A4
draft linear, a W4A16 verify linear, an INT4 activation quantiser, greedy and
sampled verification, the KV overwrite, and draft-side sampling with the
draft statistics (confidence, entropy) -- CUDA kernels behind the C ABI in
include/qspec.h, bound here with ctypes.

Importing the package does not load the library; the first call does, and
raises if libqspec.so has not been built (``build.build()``).
"""
from .binding import (QspecError, draft_sample, draft_workspace, kv_overwrite, linear_w4a4,
                      linear_w4a4_bf16, linear_w4a16, load_library, pack_weights, quant_act_int4,
                      verify_greedy, verify_sample, verify_workspace)

__all__ = ["QspecError", "draft_sample", "draft_workspace", "kv_overwrite", "linear_w4a4", "linear_w4a4_bf16",
           "linear_w4a16", "load_library", "pack_weights", "quant_act_int4", "verify_greedy", "verify_sample",
           "verify_workspace"]
