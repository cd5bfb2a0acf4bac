"""Walk-resident serial draft head for GB300 (sm_103a): C-ABI CUDA library plus a thin Python binding.

Import `speculative_decoding_serial_gb300.whead` for the binding; `build.build()` compiles the library.
"""
