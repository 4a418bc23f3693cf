"""ctypes binding of libkvc8 (``include/kvc8.h``): argument marshalling only.

The functions carry the C names and argument order.  Tensor arguments may be
torch tensors (their ``data_ptr()`` is passed), plain integer addresses, or
None for NULL.  ``stream=None`` means torch's current CUDA stream.  A non-OK
status raises :class:`Kvc8Error`.  There is no fallback: if the library cannot
be built or loaded, importing the binding's functions fails loudly.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import buildlib as _build

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_CUDA = 3
ERR_DEVICE_BOUNDS = 4
ERR_WORKSPACE = 5

DEV_OK = 0
DEV_BAD_BLOCK_ID = 1
DEV_POS_BEYOND_TABLE = 2
DEV_OUT_ROW_RANGE = 3
DEV_BAD_LENGTH = 4

HEADER = os.path.join(_build.INCLUDE, "kvc8.h")


class Kvc8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_name(status)} ({status})")


class Geom(ctypes.Structure):
    """kvc8_geom."""
    _fields_ = [("num_seqs", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("quant_mode", ctypes.c_int32)]

    def __repr__(self):
        return "Geom(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


_lock = threading.Lock()
_lib = None


def declared_functions() -> list:
    """Names of the functions that include/kvc8.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc8_\w+)\s*\(", text)))


def configure(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the C signatures of kvc8.h on a loaded copy of the library."""
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    G = ctypes.POINTER(Geom)
    lib.kvc8_status_str.argtypes = [ctypes.c_int]
    lib.kvc8_status_str.restype = ctypes.c_char_p
    lib.kvc8_version.argtypes = []
    lib.kvc8_version.restype = i32
    lib.kvc8_store.argtypes = [G, i64, P, P, i64, i64, P, P, P, P, P, P, P, P, P]
    lib.kvc8_store.restype = ctypes.c_int
    lib.kvc8_gather_workspace_bytes.argtypes = [G]
    lib.kvc8_gather_workspace_bytes.restype = sz
    lib.kvc8_build_metadata.argtypes = [G, P, P, P, P, sz, P, P]
    lib.kvc8_build_metadata.restype = ctypes.c_int
    lib.kvc8_dequant_gather.argtypes = [G, P, P, P, P, P, P, P, P, P, i64, i64, i64, P, sz, P, P]
    lib.kvc8_dequant_gather.restype = ctypes.c_int
    lib.kvc8_dequant_gather_planned.argtypes = [G, P, P, P, P, P, P, P, P, i64, i64, i64, P, sz,
                                                P, P]
    lib.kvc8_dequant_gather_planned.restype = ctypes.c_int
    lib.kvc8_get_error.argtypes = [P, ctypes.POINTER(ctypes.c_int32), i32, P]
    lib.kvc8_get_error.restype = ctypes.c_int
    lib.kvc8_dequant_gather_noalloc.argtypes = [G, P, P, P, P, P, P, P, P, P, i64, i64, i64, P, P]
    lib.kvc8_dequant_gather_noalloc.restype = ctypes.c_int
    lib.kvc8_store_bf16.argtypes = [G, i64, P, P, i64, i64, P, P, P, P, P, P, P]
    lib.kvc8_store_bf16.restype = ctypes.c_int
    lib.kvc8_gather_bf16.argtypes = [G, P, P, P, P, P, P, P, i64, i64, i64, P, sz, P, P]
    lib.kvc8_gather_bf16.restype = ctypes.c_int
    lib.kvc8_attention_workspace_bytes.argtypes = [G, i32]
    lib.kvc8_attention_workspace_bytes.restype = sz
    lib.kvc8_paged_decode_attention.argtypes = [G, i32, P, i64, i64, P, P, P, P, P, P,
                                                ctypes.c_float, P, i64, i64, P, sz, P, P]
    lib.kvc8_paged_decode_attention.restype = ctypes.c_int
    lib.kvc8_append_gather.argtypes = [G, i64, P, P, i64, i64, P, P, P, P, P, P, P, P, P, P, i64,
                                       i64, i64, P, sz, P, P]
    lib.kvc8_append_gather.restype = ctypes.c_int
    lib.kvc8_build_append_metadata.argtypes = [G, P, P, P, P, P, sz, P, P]
    lib.kvc8_build_append_metadata.restype = ctypes.c_int
    lib.kvc8_append_gather_planned.argtypes = [G, i64, P, P, i64, i64, P, P, P, P, P, P, P, P, P,
                                               i64, i64, i64, P, sz, P, P]
    lib.kvc8_append_gather_planned.restype = ctypes.c_int
    return lib


def load(build_if_needed: bool = True) -> ctypes.CDLL:
    """Load libkvc8.so (building it with nvcc first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build() if build_if_needed else _build.LIB_PATH
        if not os.path.exists(path):
            raise ImportError(f"libkvc8 is not built ({path}); run dequant_kvc8_store_gb300/buildlib.py")
        _lib = configure(ctypes.CDLL(path))
        return _lib


def status_name(status: int) -> str:
    try:
        return load().kvc8_status_str(int(status)).decode()
    except Exception:  # while reporting a load failure
        return "status"


def _p(x):
    """Device/host address of a tensor, int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ok(status: int, where: str):
    if status != OK:
        raise Kvc8Error(status, where)


def kvc8_version() -> int:
    return int(load().kvc8_version())


def kvc8_status_str(status: int) -> str:
    return load().kvc8_status_str(int(status)).decode()


def kvc8_store(g: Geom, num_tokens, key_states, value_states, x_tok_stride, x_head_stride,
               key_cache, value_cache, key_scale, value_scale, block_table, cu_q_lens,
               context_kv_lens, dev_error=None, stream=None) -> None:
    st = load().kvc8_store(ctypes.byref(g), int(num_tokens), _p(key_states), _p(value_states),
                           int(x_tok_stride), int(x_head_stride), _p(key_cache),
                           _p(value_cache), _p(key_scale), _p(value_scale), _p(block_table),
                           _p(cu_q_lens), _p(context_kv_lens), _p(dev_error), _stream(stream))
    _ok(st, "kvc8_store")


def kvc8_gather_workspace_bytes(g: Geom) -> int:
    return int(load().kvc8_gather_workspace_bytes(ctypes.byref(g)))


def kvc8_build_metadata(g: Geom, context_lengths, context_seq_offset, offsets_out, workspace,
                        workspace_bytes, dev_error=None, stream=None) -> None:
    st = load().kvc8_build_metadata(ctypes.byref(g), _p(context_lengths), _p(context_seq_offset),
                                    _p(offsets_out), _p(workspace), int(workspace_bytes),
                                    _p(dev_error), _stream(stream))
    _ok(st, "kvc8_build_metadata")


def kvc8_dequant_gather(g: Geom, key_cache, value_cache, key_scale, value_scale, block_table,
                        context_lengths, context_seq_offset, key_out, value_out, out_rows,
                        out_tok_stride, out_head_stride, workspace, workspace_bytes,
                        dev_error=None, stream=None) -> None:
    st = load().kvc8_dequant_gather(ctypes.byref(g), _p(key_cache), _p(value_cache),
                                    _p(key_scale), _p(value_scale), _p(block_table),
                                    _p(context_lengths), _p(context_seq_offset), _p(key_out),
                                    _p(value_out), int(out_rows), int(out_tok_stride),
                                    int(out_head_stride), _p(workspace), int(workspace_bytes),
                                    _p(dev_error), _stream(stream))
    _ok(st, "kvc8_dequant_gather")


def kvc8_dequant_gather_planned(g: Geom, key_cache, value_cache, key_scale, value_scale,
                                block_table, context_lengths, key_out, value_out, out_rows,
                                out_tok_stride, out_head_stride, workspace, workspace_bytes,
                                dev_error=None, stream=None) -> None:
    st = load().kvc8_dequant_gather_planned(ctypes.byref(g), _p(key_cache), _p(value_cache),
                                            _p(key_scale), _p(value_scale), _p(block_table),
                                            _p(context_lengths), _p(key_out), _p(value_out),
                                            int(out_rows), int(out_tok_stride),
                                            int(out_head_stride), _p(workspace),
                                            int(workspace_bytes), _p(dev_error),
                                            _stream(stream))
    _ok(st, "kvc8_dequant_gather_planned")


NOALLOC_MAX_SEQS = 4096  # KVC8_NOALLOC_MAX_SEQS


def kvc8_dequant_gather_noalloc(g: Geom, key_cache, value_cache, key_scale, value_scale,
                                block_table, context_lengths, context_seq_offset, key_out,
                                value_out, out_rows, out_tok_stride, out_head_stride,
                                dev_error=None, stream=None) -> None:
    """kvc8_dequant_gather without a workspace, for callers that cannot allocate
    device memory: the plan lives in a fixed array inside the library (one per
    device, shared by all calls, at most NOALLOC_MAX_SEQS sequences).  Make the
    first call on a device before any stream capture; calls that overlap on the
    GPU race on the shared array."""
    st = load().kvc8_dequant_gather_noalloc(ctypes.byref(g), _p(key_cache), _p(value_cache),
                                            _p(key_scale), _p(value_scale), _p(block_table),
                                            _p(context_lengths), _p(context_seq_offset),
                                            _p(key_out), _p(value_out), int(out_rows),
                                            int(out_tok_stride), int(out_head_stride),
                                            _p(dev_error), _stream(stream))
    _ok(st, "kvc8_dequant_gather_noalloc")


def kvc8_store_bf16(g: Geom, num_tokens, key_states, value_states, x_tok_stride, x_head_stride,
                    key_cache, value_cache, block_table, cu_q_lens, context_kv_lens,
                    dev_error=None, stream=None) -> None:
    st = load().kvc8_store_bf16(ctypes.byref(g), int(num_tokens), _p(key_states),
                                _p(value_states), int(x_tok_stride), int(x_head_stride),
                                _p(key_cache), _p(value_cache), _p(block_table), _p(cu_q_lens),
                                _p(context_kv_lens), _p(dev_error), _stream(stream))
    _ok(st, "kvc8_store_bf16")


def kvc8_gather_bf16(g: Geom, key_cache, value_cache, block_table, context_lengths,
                     context_seq_offset, key_out, value_out, out_rows, out_tok_stride,
                     out_head_stride, workspace, workspace_bytes, dev_error=None,
                     stream=None) -> None:
    st = load().kvc8_gather_bf16(ctypes.byref(g), _p(key_cache), _p(value_cache),
                                 _p(block_table), _p(context_lengths), _p(context_seq_offset),
                                 _p(key_out), _p(value_out), int(out_rows), int(out_tok_stride),
                                 int(out_head_stride), _p(workspace), int(workspace_bytes),
                                 _p(dev_error), _stream(stream))
    _ok(st, "kvc8_gather_bf16")


def kvc8_append_gather(g: Geom, num_tokens, key_states, value_states, x_tok_stride,
                       x_head_stride, key_cache, value_cache, key_scale, value_scale, block_table,
                       cu_q_lens, context_kv_lens, context_seq_offset, key_out, value_out,
                       out_rows, out_tok_stride, out_head_stride, workspace, workspace_bytes,
                       dev_error=None, stream=None) -> None:
    st = load().kvc8_append_gather(
        ctypes.byref(g), int(num_tokens), _p(key_states), _p(value_states), int(x_tok_stride),
        int(x_head_stride), _p(key_cache), _p(value_cache), _p(key_scale), _p(value_scale),
        _p(block_table), _p(cu_q_lens), _p(context_kv_lens), _p(context_seq_offset),
        _p(key_out), _p(value_out), int(out_rows), int(out_tok_stride), int(out_head_stride),
        _p(workspace), int(workspace_bytes), _p(dev_error), _stream(stream))
    _ok(st, "kvc8_append_gather")


def kvc8_build_append_metadata(g: Geom, cu_q_lens, context_kv_lens, context_seq_offset,
                               offsets_out, workspace, workspace_bytes, dev_error=None,
                               stream=None) -> None:
    st = load().kvc8_build_append_metadata(
        ctypes.byref(g), _p(cu_q_lens), _p(context_kv_lens), _p(context_seq_offset),
        _p(offsets_out), _p(workspace), int(workspace_bytes), _p(dev_error), _stream(stream))
    _ok(st, "kvc8_build_append_metadata")


def kvc8_append_gather_planned(g: Geom, num_tokens, key_states, value_states, x_tok_stride,
                               x_head_stride, key_cache, value_cache, key_scale, value_scale,
                               block_table, cu_q_lens, context_kv_lens, key_out, value_out,
                               out_rows, out_tok_stride, out_head_stride, workspace,
                               workspace_bytes, dev_error=None, stream=None) -> None:
    st = load().kvc8_append_gather_planned(
        ctypes.byref(g), int(num_tokens), _p(key_states), _p(value_states), int(x_tok_stride),
        int(x_head_stride), _p(key_cache), _p(value_cache), _p(key_scale), _p(value_scale),
        _p(block_table), _p(cu_q_lens), _p(context_kv_lens), _p(key_out), _p(value_out),
        int(out_rows), int(out_tok_stride), int(out_head_stride), _p(workspace),
        int(workspace_bytes), _p(dev_error), _stream(stream))
    _ok(st, "kvc8_append_gather_planned")


def kvc8_attention_workspace_bytes(g: Geom, num_q_heads: int) -> int:
    return int(load().kvc8_attention_workspace_bytes(ctypes.byref(g), int(num_q_heads)))


def kvc8_paged_decode_attention(g: Geom, num_q_heads, query, q_seq_stride, q_head_stride,
                                key_cache, value_cache, key_scale, value_scale, block_table,
                                context_lengths, softmax_scale, out, out_seq_stride,
                                out_head_stride, workspace, workspace_bytes, dev_error=None,
                                stream=None) -> None:
    st = load().kvc8_paged_decode_attention(
        ctypes.byref(g), int(num_q_heads), _p(query), int(q_seq_stride), int(q_head_stride),
        _p(key_cache), _p(value_cache), _p(key_scale), _p(value_scale), _p(block_table),
        _p(context_lengths), float(softmax_scale), _p(out), int(out_seq_stride),
        int(out_head_stride), _p(workspace), int(workspace_bytes), _p(dev_error),
        _stream(stream))
    _ok(st, "kvc8_paged_decode_attention")


def kvc8_get_error(dev_error, reset: bool = False, stream=None) -> int:
    """Synchronise the stream and return the device error code (0 = none)."""
    code = ctypes.c_int32(0)
    st = load().kvc8_get_error(_p(dev_error), ctypes.byref(code), int(bool(reset)),
                               _stream(stream))
    if st not in (OK, ERR_DEVICE_BOUNDS):
        raise Kvc8Error(st, "kvc8_get_error")
    return int(code.value)
