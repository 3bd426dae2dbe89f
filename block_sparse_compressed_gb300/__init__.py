"""GB300-native Heavily Compressed Attention (HCA): forward and backward.

The computation lives in libhca.so (C ABI in include/hca.h, CUDA kernels for
sm_103a under csrc/); ``hca`` is its thin ctypes binding.
"""
from .hca import (HCAError, hca_attn_bwd, hca_attn_fwd, hca_query_tile_positions, hca_status_string,  # noqa: F401
                  hca_tile_map, hca_version, hca_visible_pairs, hca_workspace_size, hca_workspace_status)
