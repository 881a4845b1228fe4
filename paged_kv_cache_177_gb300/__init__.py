"""GB300-native PagedAttention decode.

The compute path is the CUDA library ``libpagedkv.so`` (C ABI in
``include/pagedkv.h``), reached from Python through ``binding``:
``paged_decode_attention``, ``kv_append``, ``copy_blocks`` and the checks
around them.  ``block_manager`` and ``scheduler`` are the host-side paging and
continuous-batching logic that produce the calls' metadata; ``workloads``
draws seeded synthetic inputs.

The binding is imported on first use, so the host-side modules work on
machines without the library or a GPU.
"""
__version__ = "0.1.0"

_BINDING_NAMES = {
    "paged_decode_attention", "kv_append", "copy_blocks", "check_copy_pairs", "validate", "validate_slots",
    "swap_blocks", "check_swap_pairs", "paged_decode_attention_shared_prefix", "paged_prefill_attention",
    "paged_decode_step", "shared_prefix_workspace_bytes", "prefix_groups", "copy_blocks_layers", "kv_append_layers",
    "layer_pointers", "device_error", "workspace_bytes", "partition_tokens", "decode_launches", "decode_persistent",
    "status_string", "version", "PagedKVError",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
