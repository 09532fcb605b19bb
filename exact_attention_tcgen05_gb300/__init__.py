"""Exact scaled-dot-product attention for NVIDIA GB300 (sm_103a).

The compute path is the C-ABI library ``libattn.so`` built from ``csrc/``; the Python
functions in ``binding`` only marshal arguments to it. Importing this package does not
load the library; the first call does, and fails loudly if it was not built.
"""

__all__ = ["attn_fwd", "attn_bwd", "attention", "FlashAttentionFunction"]


def __getattr__(name):
    if name in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_bytes"):
        from . import binding
        return getattr(binding, name)
    if name in ("attention", "FlashAttentionFunction"):
        from . import autograd
        return getattr(autograd, name)
    raise AttributeError(name)
