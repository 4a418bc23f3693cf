"""GB300-native int8 ("C8") paged KV-cache store and dequant-gather.

The work is done by libkvc8 (hand-written sm_103a CUDA kernels behind the C ABI
in ``include/kvc8.h``); this package builds it and binds it with ctypes.
PyTorch only provides device memory and streams.
"""
from .binding import (DEV_BAD_BLOCK_ID, DEV_BAD_LENGTH, DEV_OK, DEV_OUT_ROW_RANGE,  # noqa: F401
                      DEV_POS_BEYOND_TABLE, ERR_CUDA, ERR_DEVICE_BOUNDS, ERR_INVALID_ARG,
                      ERR_UNSUPPORTED, ERR_WORKSPACE, OK, Geom, Kvc8Error,
                      declared_functions, kvc8_build_metadata, kvc8_dequant_gather,
                      kvc8_dequant_gather_noalloc, kvc8_dequant_gather_planned,
                      kvc8_gather_workspace_bytes, NOALLOC_MAX_SEQS,
                      kvc8_get_error, kvc8_status_str, kvc8_store, kvc8_version, load,
                      kvc8_store_bf16, kvc8_gather_bf16, kvc8_append_gather,
                      kvc8_build_append_metadata, kvc8_append_gather_planned,
                      kvc8_attention_workspace_bytes, kvc8_paged_decode_attention)
from .buildlib import build  # noqa: F401
