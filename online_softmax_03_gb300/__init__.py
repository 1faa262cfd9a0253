"""Exact scaled-dot-product attention forward for GB300 (sm_103a).

The compute path is the CUDA library built from csrc/ (libattn.so) behind
the C ABI declared in include/attn.h; `binding` marshals torch tensors into
that ABI.  Nothing here computes attention on the host.
"""
