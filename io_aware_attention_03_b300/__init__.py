"""Exact scaled-dot-product attention for one NVIDIA B300 (sm_103a).

The computation runs in the CUDA library ``libattn_b300.so`` (built from
``csrc/``) behind a C ABI declared in ``include/attn_b300.h``.  The Python
binding in :mod:`io_aware_attention_03_b300.attn` only marshals torch tensors
into that ABI; importing it loads the library and raises if it is missing.

Attribute access such as ``io_aware_attention_03_b300.attn_fwd`` loads the
binding lazily, so that :mod:`io_aware_attention_03_b300.inputs` (synthetic
inputs) can be imported on its own.
"""

_BINDING_NAMES = (
    "attn_fwd",
    "attn_fwd_fp8",
    "attn_bwd",
    "attn_bwd_workspace_size",
    "fp8_vt_stride",
    "attn_prefill_paged",
    "attn_decode",
    "attn_decode_fp8",
    "attn_decode_workspace_size",
    "attn_decode_noalloc",
    "attn_last_device_status",
    "attn_status_string",
    "AttnError",
)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import attn as _attn

        return getattr(_attn, name)
    raise AttributeError(name)
