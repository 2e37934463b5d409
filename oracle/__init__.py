"""fp64 CPU oracle of the Gated Residual read/write (test infrastructure only).

Only the tests, the smoke check and the bench's CPU-baseline leg may import this package. The
product path (the CUDA library and its Python binding) never does, and the two share no code.

``gr_oracle.c`` holds the definition (per-token loops in fp64, OpenMP over tokens);
``dense.py`` holds a second, matrix-form formulation used to cross-check it on tiny sizes.
The functions here take numpy arrays of any float dtype, convert them exactly to float64, and
return float64 arrays.
"""
from .oracle import (build, chain, decompose, fp8_code_values, fp8_decode, fp8_encode, fp8_round_codes,
                     lib, num_threads, read, read_backward, read_fixed_gates, residual_add,
                     round_to_storage, set_num_threads, use_library, write, write_backward,
                     write_then_read, write_then_read_fp8)

__all__ = ["build", "chain", "decompose", "fp8_code_values", "fp8_decode", "fp8_encode", "fp8_round_codes",
           "lib", "num_threads", "read", "read_backward", "read_fixed_gates", "residual_add",
           "round_to_storage", "write_backward",
           "set_num_threads", "use_library", "write", "write_then_read", "write_then_read_fp8"]
