"""Paged attention over a block-table KV cache, hand-written for sm_103a.

The compute lives in ``libpkv.so`` (C ABI, ``include/pkv.h``); this package is
its thin binding.  The library is loaded on first use and a missing or
unloadable library raises: there is no CPU fallback.
"""
_API = ("PkvError", "cascade_attention", "flash_attn_varlen_func",
        "merge_attn_states", "paged_attention_workspace_size",
        "reshape_and_cache_flash")


def __getattr__(name):
    if name in _API:
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
