"""GB300-native Gated Residual (GR) read/write.

The C ABI (include/gr.h, libgr_gb300.so) holds the CUDA kernels; ``gr`` is its Python binding
(argument marshalling only) and ``workloads`` the seeded synthetic inputs.
"""
from . import gr  # noqa: F401
from .gr import (GRError, Params, load, pack_params, read, read_fixed_gates,  # noqa: F401
                 residual_add_ref, write, write_then_read, write_then_read_host)
