"""GB300-native 1-bit (Q1_0) GEMV for LLM decode.

The compute path is the C-ABI shared library built from ``csrc/`` (declared in
``include/q1gemv.h``); ``decode_q1_gemv_gb300.binding`` marshals torch CUDA
tensors into it.  Submodules are imported on demand; the library is loaded on
first use, and when it is missing every call raises.
"""
