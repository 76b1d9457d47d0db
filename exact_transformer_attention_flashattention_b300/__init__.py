"""Exact softmax attention for NVIDIA B300 (sm_103a).

Prefill (causal, sliding-window, non-causal) and split-KV decode with a
logsumexp tree combine, implemented as hand-written CUDA behind the C ABI of
include/b300attn.h.  The compute entry points are re-exported lazily from
``binding`` so that ``inputs`` can be imported on machines without the built
library; touching any entry point loads libb300attn.so and fails loudly if it
is missing.
"""

_BINDING = {
    "attn_fwd", "attn_fwd_varlen", "attn_fwd_paged", "attn_bwd", "attn_bwd_workspace_size",
    "attn_fp8_quantize", "attn_fwd_fp8", "attn_fp8_padded_len", "attn_fp8_workspace_size",
    "attn_decode_splitkv", "attn_decode_partials", "attn_decode_splitkv_noalloc",
    "attn_decode_splitkv_paged", "lse_tree_combine", "attn_decode_chunk",
    "attn_decode_workspace_size", "device_status", "selftest_bounded_wait", "last_error",
    "split_partials_view", "B300AttnError", "lib", "LIB_PATH",
}
_ALTERNATING = {"alternating_attention", "layer_groups"}

__all__ = sorted(_BINDING | _ALTERNATING)


def __getattr__(name):
    if name in _BINDING:
        from . import binding
        return getattr(binding, name)
    if name in _ALTERNATING:
        from . import alternating
        return getattr(alternating, name)
    raise AttributeError(name)
