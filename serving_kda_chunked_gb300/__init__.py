"""Kimi Delta Attention (KDA) on GB300: chunked prefill and batched decode.

The compute runs in hand-written CUDA kernels for sm_103a inside
``libkda.so``, behind the C ABI declared in ``include/kda.h``.  This package
is the thin Python binding over that library (argument marshalling only).
"""
from ._binding import (KDA_BF16, KDA_ERR_CUDA, KDA_ERR_INVALID_ARG,
                       KDA_ERR_TIMEOUT, KDA_ERR_TOO_LARGE, KDA_ERR_UNSUPPORTED, KDA_FP32, KDA_OK,
                       LIB_PATH, KdaError, abi_version, kda_decode_step,
                       kda_decode_step_pooled, kda_gdn_decode_step, kda_gdn_decode_step_pooled,
                       kda_gdn_prefill_chunked,
                       kda_noalloc_scratch_bytes, kda_prefill_check, kda_prefill_chunked,
                       kda_prefill_noalloc_check,
                       kda_prefill_chunked_host, kda_prefill_chunked_noalloc,
                       kda_prefill_host_workspace_size,
                       kda_prefill_workspace_size, load, status_string)

__all__ = ["kda_prefill_chunked", "kda_prefill_chunked_noalloc", "kda_noalloc_scratch_bytes",
           "kda_prefill_chunked_host", "kda_prefill_host_workspace_size",
           "kda_prefill_workspace_size", "kda_prefill_check", "kda_prefill_noalloc_check",
           "kda_decode_step", "kda_decode_step_pooled", "kda_gdn_prefill_chunked",
           "kda_gdn_decode_step", "kda_gdn_decode_step_pooled", "status_string",
           "abi_version", "load", "KdaError", "LIB_PATH", "KDA_OK",
           "KDA_ERR_INVALID_ARG", "KDA_ERR_UNSUPPORTED", "KDA_ERR_CUDA",
           "KDA_ERR_TIMEOUT", "KDA_ERR_TOO_LARGE", "KDA_BF16", "KDA_FP32"]
