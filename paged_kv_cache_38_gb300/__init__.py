"""Paged KV-cache hot path for NVIDIA GB300 (sm_103a): a C-ABI CUDA library plus its binding.

The library (``libpa.so``, built from ``csrc/`` by ``build.build()``) implements paged decode
attention and the KV block movers; ``pa`` marshals torch tensors into its C entry points.
"""
from .pa import (PA_BF16, PA_ECUDA, PA_EINVAL, PA_ENOSPACE, PA_ERR_BLOCK_ID, PA_ERR_CTX_LEN,
                 PA_ERR_TIMEOUT, PA_EUNSUPPORTED, PA_F16, PA_FP8_E4M3, PA_OK,
                 PA_STATIC_WORKSPACE_BYTES, PA_SWAP_IN, PA_SWAP_OUT, PaError, lib,
                 make_decode_args, pa_copy_blocks, pa_decode, pa_decode_static_workspace,
                 pa_decode_workspace_size, pa_prefill, pa_swap_blocks, pa_testing_set_wait_limit,
                 pa_write_kv, pa_write_kv_fp8)

__all__ = [
    "PA_BF16", "PA_ECUDA", "PA_EINVAL", "PA_ENOSPACE", "PA_ERR_BLOCK_ID", "PA_ERR_CTX_LEN",
    "PA_ERR_TIMEOUT", "PA_EUNSUPPORTED", "PA_F16", "PA_FP8_E4M3", "PA_OK",
    "PA_STATIC_WORKSPACE_BYTES", "PA_SWAP_IN", "PA_SWAP_OUT", "PaError", "lib",
    "make_decode_args", "pa_copy_blocks", "pa_decode", "pa_decode_static_workspace",
    "pa_decode_workspace_size", "pa_prefill", "pa_swap_blocks", "pa_testing_set_wait_limit",
    "pa_write_kv", "pa_write_kv_fp8",
]
