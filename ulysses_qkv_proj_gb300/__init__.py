"""Ulysses QKV front end on one GB300: fused bf16 QKV projection + per-head
RMSNorm + RoPE + head-band scatter, and the head-chunk pack/merge kernels.

The compute lives in the C-ABI library `libqnre.so` (hand-written CUDA for
sm_103a).  `ulysses_qkv_proj_gb300.binding` marshals torch tensors into that
library's calls; the library is loaded on first use and a missing build is an
error, never a fallback.
"""
__all__ = ["binding", "workloads"]
