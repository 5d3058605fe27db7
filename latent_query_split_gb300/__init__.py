"""GB300-native (sm_103a) FLARE / FLARE++ split-KV token mixer.

The product is the C-ABI CUDA library declared in include/flare.h
(latent_query_split_gb300/_build/libflare.so, built by build.build()); this
package adds its thin Python binding (flare.py) and the seeded workload
generators (workloads.py).
"""
from .flare import (FlareError, flare_decode_fwd, flare_device_status, flare_encoder_bwd,
                    flare_encoder_fwd, flare_fwd, flare_lse_merge, flare_pp_fwd,
                    flare_version, flare_workspace_bytes, load_library, make_dims)

__all__ = ["FlareError", "flare_decode_fwd", "flare_device_status", "flare_encoder_bwd",
           "flare_encoder_fwd", "flare_fwd", "flare_lse_merge", "flare_pp_fwd", "flare_version",
           "flare_workspace_bytes", "load_library", "make_dims"]
