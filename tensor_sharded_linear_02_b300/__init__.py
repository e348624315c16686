"""Tensor-parallel sharded linear layer and Megatron-style MLP block on one
B300 (sm_103a): a C-ABI CUDA library (``libtp_b300.so``) plus a thin ctypes
binding with the same entry-point names.

The binding is imported lazily so that importing ``inputs`` (the seeded
generator) does not load the CUDA library.
"""
__all__ = [
    "tp_column_linear", "tp_column_linear_grouped", "tp_row_linear",
    "tp_shard_reduce", "tp_shard_concat", "tp_shard_concat_grouped",
    "tp_mlp_block", "tp_mlp_block_workspace_size", "tp_mlp_block_static_ws",
    "tp_qkv_linear",
    "tp_column_linear_bias", "tp_row_linear_bias", "tp_mlp_block_bias",
    "tp_column_linear_backward", "tp_row_linear_backward", "tp_mlp_block_backward",
    "tp_mlp_block_backward_workspace_size",
    "tp_get_device_status",
    "tp_status_string", "TPError",
]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
