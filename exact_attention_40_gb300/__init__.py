"""Exact fused scaled-dot-product attention for GB300 (sm_103a).

The compute lives in the C-ABI library ``libexattn.so`` (CUDA kernels under
``csrc/``); ``exattn`` is its thin ctypes binding.  Importing the package does
not load the library, so the input generator (``synth``) can be used on
hosts without a GPU; importing ``exattn`` loads it and fails loudly if it
has not been built.
"""

__all__ = ["exattn", "synth"]


def __getattr__(name):
    if name in ("attn_fwd", "attn_decode_paged", "attn_decode_workspace_bytes",
                "attn_get_device_status", "attn_status_string"):
        from . import exattn
        return getattr(exattn, name)
    raise AttributeError(name)
