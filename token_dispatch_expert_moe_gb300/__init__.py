"""Single-GPU MoE layer for GB300 (sm_103a): the compute chain of a token-level
MoE dispatcher (route, drop, permute, SwiGLU grouped GEMM, un-permute and the
backward), as hand-written CUDA kernels behind the C ABI of libmoe.so.

`token_dispatch_expert_moe_gb300._lib` is the ctypes binding (one function per
C entry point); `token_dispatch_expert_moe_gb300.layer.MoELayer` strings the
calls together for a whole layer.
"""
__version__ = "0.1.0"
