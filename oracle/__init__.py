"""CPU oracle for the int8 (C8) paged KV-cache store and dequant-gather.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  The
product library never links, loads or calls it, and it shares no code with
the CUDA path: the arithmetic lives in ``kvc8_oracle.c`` (plain C, one IEEE
binary32 operation per step, built with ``-O2 -ffp-contract=off``), and this
module only marshals numpy arrays into it.

What it computes, and the page passages each step follows, is written out at
the top of ``kvc8_oracle.c``: mojo_opset pull request #379, "feat: [MLU] add
mlu experimental ops; fix post norm bug" (the review passes describing the
torch-native MojoStorePagedKVCacheC8 / MojoDequantFromPagedKVCache), with the
torch-native code as golden reference per the "Mojo Opset" README, section
"Backend Implementations / Torch native".

Pins (in ``tests/test_oracle_*.py``): hand-worked goldens under
``tests/golden/``, exact rational re-derivation of each rounding, invariants
(code range, the absmax element maps to +-127, |dequant(q) - x| <= s/2),
special cases (identity with s = 1, identity block table), a brute-force
placement model, and copies of the oracle with planted mistakes that the pins
must reject.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "kvc8_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkvc8_oracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra"]

OK = 0
ERR_ARG = 1
ERR_BOUNDS = 4


class OracleError(RuntimeError):
    pass


def compile_source(src_path: str, out_path: str) -> str:
    """Compile a C source of the oracle's form into a shared library (builds
    the oracle itself, and the copies with planted mistakes that the tests use
    to show the pins have teeth)."""
    os.makedirs(os.path.dirname(out_path) or ".", exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, src_path, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build/`` and return the path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)):
        return _LIB_PATH
    return compile_source(SOURCE, _LIB_PATH)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    """Contiguous array of exactly ``dtype`` (no silent conversion)."""
    if a is None:
        return None
    a = np.asarray(a)
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return np.ascontiguousarray(a)


def _check(rc, what):
    if rc != OK:
        raise OracleError(f"{what} returned {rc}")


class Oracle:
    """numpy front end of one compiled copy of ``kvc8_oracle.c``."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int, ctypes.c_int64
        lib.orc_quantize_rows.argtypes = [i32, i64, i32, i32, P, P, P, P]
        lib.orc_quantize_rows.restype = i32
        lib.orc_store.argtypes = [i32, i32, i64, i32, i32, i32, i32, i32,
                                  P, P, P, P, P, P, P, P, P]
        lib.orc_store.restype = i32
        lib.orc_exclusive_cumsum.argtypes = [i32, P, P]
        lib.orc_exclusive_cumsum.restype = None
        lib.orc_dequant_gather.argtypes = [i32, i32, i32, i32, i32, i32, i32,
                                           P, P, P, P, P, P, P, P, P,
                                           i64, i64, i64]
        lib.orc_dequant_gather.restype = i32
        lib.orc_quantize_value.argtypes = [ctypes.c_uint16, ctypes.c_float]
        lib.orc_quantize_value.restype = ctypes.c_int8
        lib.orc_dequantize_value.argtypes = [ctypes.c_int8, ctypes.c_float]
        lib.orc_dequantize_value.restype = ctypes.c_uint16
        lib.orc_round_to_bf16.argtypes = [ctypes.c_float]
        lib.orc_round_to_bf16.restype = ctypes.c_uint16
        lib.orc_row_scale_bf16.argtypes = [P, i32]
        lib.orc_row_scale_bf16.restype = ctypes.c_float
        lib.orc_store_bf16.argtypes = [i32, i64, i32, i32, i32, i32, i32, P, P, P, P, P, P, P]
        lib.orc_store_bf16.restype = i32
        lib.orc_gather_bf16.argtypes = [i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, P,
                                        i64, i64, i64]
        lib.orc_gather_bf16.restype = i32
        lib.orc_paged_decode_attention.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, P, P,
                                                   P, P, P, P, P, ctypes.c_double, P]
        lib.orc_paged_decode_attention.restype = i32
        self.lib = lib
        self.path = lib_path

    # ---- element-level steps ---------------------------------------------

    def quantize_value(self, x_bf16_bits: int, s) -> int:
        return int(self.lib.orc_quantize_value(int(x_bf16_bits), float(np.float32(s))))

    def dequantize_value(self, q: int, s) -> int:
        return int(self.lib.orc_dequantize_value(int(q), float(np.float32(s))))

    def round_to_bf16(self, f) -> int:
        return int(self.lib.orc_round_to_bf16(float(np.float32(f))))

    def row_scale(self, row_bf16_bits) -> np.float32:
        row = _c(row_bf16_bits, np.uint16)
        return np.float32(self.lib.orc_row_scale_bf16(_ptr(row), row.shape[-1]))

    # ---- row / tensor level ----------------------------------------------

    def quantize_rows(self, quant_mode: int, x_bits, static_scale=None):
        """x_bits uint16 [n][H][D] -> (codes int8 [n][H][D], scales fp32 [n][H] or None).

        static_scale: [H][D] for quant_mode 1, one scale per row [n][H] for
        quant_mode 2 (in the cache, the scale of the row's block)."""
        x = _c(x_bits, np.uint16)
        n, H, D = x.shape
        q = np.empty((n, H, D), np.int8)
        s = np.empty((n, H), np.float32) if quant_mode == 0 else None
        ss = _c(static_scale, np.float32) if quant_mode in (1, 2) else None
        _check(self.lib.orc_quantize_rows(quant_mode, n, H, D, _ptr(x), _ptr(ss),
                                          _ptr(q), _ptr(s)), "orc_quantize_rows")
        return q, s

    def store(self, quant_mode, k_bits, v_bits, k_cache, v_cache, k_scale, v_scale,
              block_table, cu_q_lens, context_kv_lens):
        """Store in place into the numpy caches (and quant_mode-0 scale caches).

        k_bits/v_bits uint16 [N][H][D]; caches int8 [NB][H][bs][D]; k_scale /
        v_scale fp32 [NB][H][bs] (quant_mode 0, written), [H][D] (quant_mode
        1, read) or [NB][H] (quant_mode 2, read); block_table int32 [B][MB];
        cu_q_lens int32 [B+1] or None;
        context_kv_lens int32 [B].  Outputs must be C-contiguous.
        """
        for a in (k_cache, v_cache, k_scale, v_scale):
            if not a.flags.c_contiguous:
                raise ValueError("output arrays must be C-contiguous")
        if k_cache.dtype != np.int8 or v_cache.dtype != np.int8:
            raise TypeError("caches must be int8")
        if k_scale.dtype != np.float32 or v_scale.dtype != np.float32:
            raise TypeError("scales must be float32")
        k, v = _c(k_bits, np.uint16), _c(v_bits, np.uint16)
        bt = _c(block_table, np.int32)
        cu = _c(cu_q_lens, np.int32)
        ctx = _c(context_kv_lens, np.int32)
        NB, H, bs, D = k_cache.shape
        B, MB = bt.shape
        N = k.shape[0]
        _check(self.lib.orc_store(quant_mode, B, N, H, D, bs, NB, MB, _ptr(k), _ptr(v),
                                  _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                  _ptr(bt), _ptr(cu), _ptr(ctx)), "orc_store")

    def exclusive_cumsum(self, lens):
        lens = _c(lens, np.int32)
        out = np.empty(lens.shape[0], np.int64)
        self.lib.orc_exclusive_cumsum(lens.shape[0], _ptr(lens), _ptr(out))
        return out

    def dequant_gather(self, quant_mode, k_cache, v_cache, k_scale, v_scale, block_table,
                       context_lengths, context_seq_offset=None, k_out=None, v_out=None,
                       out_rows=None):
        """Gather + dequantise into bf16 bits; returns (k_out, v_out) uint16 [rows][H][D].

        Passed-in outputs must be C-contiguous uint16 [rows][H][D]; rows that
        no sequence covers keep their contents.
        """
        kc, vc = _c(k_cache, np.int8), _c(v_cache, np.int8)
        ks, vs = _c(k_scale, np.float32), _c(v_scale, np.float32)
        bt = _c(block_table, np.int32)
        ctx = _c(context_lengths, np.int32)
        off = _c(context_seq_offset, np.int64)
        NB, H, bs, D = kc.shape
        B, MB = bt.shape
        if k_out is None:
            rows = int(out_rows if out_rows is not None else int(ctx.astype(np.int64).sum()))
            k_out = np.zeros((rows, H, D), np.uint16)
            v_out = np.zeros((rows, H, D), np.uint16)
        for a in (k_out, v_out):
            if not a.flags.c_contiguous or a.dtype != np.uint16:
                raise ValueError("outputs must be C-contiguous uint16")
        rows = k_out.shape[0]
        _check(self.lib.orc_dequant_gather(quant_mode, B, H, D, bs, NB, MB, _ptr(kc), _ptr(vc),
                                           _ptr(ks), _ptr(vs), _ptr(bt), _ptr(ctx), _ptr(off),
                                           _ptr(k_out), _ptr(v_out), rows, H * D, D),
               "orc_dequant_gather")
        return k_out, v_out

    def store_bf16(self, k_bits, v_bits, k_cache, v_cache, block_table, cu_q_lens,
                   context_kv_lens):
        """bf16 store (no quantisation) into uint16 caches [NB][H][bs][D], in place."""
        for a in (k_cache, v_cache):
            if not a.flags.c_contiguous or a.dtype != np.uint16:
                raise ValueError("caches must be C-contiguous uint16")
        k, v = _c(k_bits, np.uint16), _c(v_bits, np.uint16)
        bt = _c(block_table, np.int32)
        cu = _c(cu_q_lens, np.int32)
        ctx = _c(context_kv_lens, np.int32)
        NB, H, bs, D = k_cache.shape
        B, MB = bt.shape
        _check(self.lib.orc_store_bf16(B, k.shape[0], H, D, bs, NB, MB, _ptr(k), _ptr(v),
                                       _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(cu),
                                       _ptr(ctx)), "orc_store_bf16")

    def gather_bf16(self, k_cache, v_cache, block_table, context_lengths,
                    context_seq_offset=None, k_out=None, v_out=None, out_rows=None):
        """Gather of a bf16 cache; returns (k_out, v_out) uint16 [rows][H][D]."""
        kc, vc = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
        bt = _c(block_table, np.int32)
        ctx = _c(context_lengths, np.int32)
        off = _c(context_seq_offset, np.int64)
        NB, H, bs, D = kc.shape
        B, MB = bt.shape
        if k_out is None:
            rows = int(out_rows if out_rows is not None else int(ctx.astype(np.int64).sum()))
            k_out = np.zeros((rows, H, D), np.uint16)
            v_out = np.zeros((rows, H, D), np.uint16)
        rows = k_out.shape[0]
        _check(self.lib.orc_gather_bf16(B, H, D, bs, NB, MB, _ptr(kc), _ptr(vc), _ptr(bt),
                                        _ptr(ctx), _ptr(off), _ptr(k_out), _ptr(v_out), rows,
                                        H * D, D), "orc_gather_bf16")
        return k_out, v_out

    def paged_decode_attention(self, quant_mode, query_bits, k_cache, v_cache, k_scale, v_scale,
                               block_table, context_lengths, softmax_scale):
        """Decode attention of query_bits (bf16 bits [B][Hq][D]) over the paged
        int8 cache; returns the unrounded fp64 output [B][Hq][D]."""
        qb = _c(query_bits, np.uint16)
        kc, vc = _c(k_cache, np.int8), _c(v_cache, np.int8)
        ks, vs = _c(k_scale, np.float32), _c(v_scale, np.float32)
        bt = _c(block_table, np.int32)
        ctx = _c(context_lengths, np.int32)
        NB, H, bs, D = kc.shape
        B, MB = bt.shape
        hq = qb.shape[1]
        if hq % H != 0 or qb.shape != (B, hq, D):
            raise ValueError("query must be [B][G*H][D]")
        out = np.empty((B, hq, D), np.float64)
        _check(self.lib.orc_paged_decode_attention(quant_mode, B, H, hq // H, D, bs, NB, MB,
                                                   _ptr(qb), _ptr(kc), _ptr(vc), _ptr(ks),
                                                   _ptr(vs), _ptr(bt), _ptr(ctx),
                                                   float(softmax_scale), _ptr(out)),
               "orc_paged_decode_attention")
        return out


_lock = threading.Lock()
_default = None


def default() -> Oracle:
    """The oracle built from ``kvc8_oracle.c`` as committed."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def __getattr__(name):
    # module-level shortcuts: oracle.store(...), oracle.dequant_gather(...), ...
    if name in {"quantize_value", "dequantize_value", "round_to_bf16", "row_scale",
                "quantize_rows", "store", "exclusive_cumsum", "dequant_gather",
                "store_bf16", "gather_bf16", "paged_decode_attention"}:
        return getattr(default(), name)
    raise AttributeError(name)
