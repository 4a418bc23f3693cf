"""The allocation-free dequant-gather (kvc8_dequant_gather_noalloc).

Some callers cannot allocate device memory where they gather -- a plugin inside
a runtime that owns all device memory, or a serving loop that must not
allocate once running -- so they cannot pass the workspace that
kvc8_dequant_gather needs.  The no-alloc entry point keeps that scratch in a
fixed array inside the library instead.  These tests check, through the C ABI,
that it returns exactly what the oracle's gather and the workspace entry point
return, in every scale mode, on calls in a row with different batches (so a
plan left over from an earlier call would show), and that it refuses what the
workspace entry point refuses, plus batches beyond its fixed size.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import dequant_kvc8_store_gb300 as kv
from dequant_kvc8_store_gb300 import workloads as W
from dequant_kvc8_store_gb300.device import DeviceBatch

FILL = 0xFFFF  # the bf16 NaN no dequantised value can be: rows left unwritten show


def _check_against_oracle_and_workspace_gather(w, offsets=None, layout="dense", pad=0):
    d = DeviceBatch(w, offsets=offsets, out_layout=layout, out_pad_rows=pad, fill_out=FILL)
    d.gather()  # the entry point with a caller workspace
    assert d.error_code() == 0
    want_ws = d.host_outputs()
    d.k_out.view(torch.int16).fill_(-1)
    d.v_out.view(torch.int16).fill_(-1)
    ko = d.k_out
    kv.kvc8_dequant_gather_noalloc(d.g, d.k_cache, d.v_cache, d.k_scale, d.v_scale,
                                   d.block_table, d.context_lengths, d.offsets, ko, d.v_out,
                                   d.out_rows, ko.stride(0), ko.stride(1), d.dev_error)
    got = d.host_outputs()
    assert d.error_code() == 0
    H, D = w.kv_heads, w.head_dim
    want_k = np.full((d.out_rows, H, D), FILL, np.uint16)
    want_v = np.full((d.out_rows, H, D), FILL, np.uint16)
    oracle.dequant_gather(w.quant_mode, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                          w.block_table, w.context_lengths,
                          None if offsets is None else np.asarray(offsets, np.int64),
                          want_k, want_v)
    # tolerance: none (0 ULP), as for every gather comparison in this suite
    assert np.array_equal(got[0], want_k) and np.array_equal(got[1], want_v)
    assert np.array_equal(got[0], want_ws[0]) and np.array_equal(got[1], want_ws[1])


@pytest.mark.gpu
def test_noalloc_gather_matches_oracle_and_workspace_gather_in_a_row():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    kv.load()
    rng = np.random.default_rng(404)
    # set-up call: nothing to gather, but the device's array is looked up
    g0 = kv.Geom(0, 2, 64, 16, 8, 4, 0)
    assert kv.load().kvc8_dequant_gather_noalloc(ctypes.byref(g0), *([None] * 7), None, None,
                                                 0, 0, 0, None, None) == kv.OK
    first = W.make_workload("noalloc-a", q_lens=np.zeros(300, np.int64),
                            ctx_before=rng.integers(0, 600, size=300), kv_heads=2,
                            head_dim=64, block_size=16, num_blocks=300 * 38, quant_mode=0,
                            seed=404, with_store=False)
    second = W.make_workload("noalloc-b", q_lens=np.zeros(5, np.int64),
                             ctx_before=[129, 1, 0, 640, 77], kv_heads=8, head_dim=128,
                             block_size=64, num_blocks=60, quant_mode=1, seed=405,
                             with_store=False)
    third = W.make_workload("noalloc-c", q_lens=np.zeros(7, np.int64),
                            ctx_before=[33, 0, 250, 1, 16, 17, 99], kv_heads=4, head_dim=128,
                            block_size=16, num_blocks=120, quant_mode=2, seed=406,
                            with_store=False)
    _check_against_oracle_and_workspace_gather(first)
    lens = second.context_lengths.astype(np.int64)
    offsets = np.concatenate([[3], 3 + np.cumsum(lens + 2)[:-1]])
    _check_against_oracle_and_workspace_gather(second, offsets=offsets, layout="head_major",
                                               pad=5)
    _check_against_oracle_and_workspace_gather(third)
    _check_against_oracle_and_workspace_gather(first)  # the first batch again, after the others


def test_noalloc_gather_refuses_batches_beyond_its_scratch():
    g = kv.Geom(kv.NOALLOC_MAX_SEQS + 1, 8, 128, 16, 64, 8, 0)
    fake = 1 << 20  # never dereferenced: the size check comes first
    st = kv.load().kvc8_dequant_gather_noalloc(ctypes.byref(g), *([fake] * 6), None, fake, fake,
                                               10, 1024, 128, None, None)
    assert st == kv.ERR_UNSUPPORTED


def test_noalloc_gather_refuses_what_the_workspace_gather_refuses():
    """Geometry checks are shared with kvc8_dequant_gather: a block table whose
    num_seqs x max_blocks_per_seq leaves int32, a bad scale mode, a head_dim
    that is not a multiple of 16.  Nothing is dereferenced or enqueued."""
    lib = kv.load()
    fake = 1 << 20
    for geom, want in [((4096, 8, 128, 16, 64, 1 << 20, 0), kv.ERR_UNSUPPORTED),
                       ((4, 8, 128, 16, 64, 8, 3), kv.ERR_INVALID_ARG),
                       ((4, 8, 120, 16, 64, 8, 0), kv.ERR_INVALID_ARG)]:
        g = kv.Geom(*geom)
        st_noalloc = lib.kvc8_dequant_gather_noalloc(ctypes.byref(g), *([fake] * 6), None, fake,
                                                     fake, 10, 1024, 128, None, None)
        st_ws = lib.kvc8_dequant_gather(ctypes.byref(g), *([fake] * 6), None, fake, fake, 10,
                                        1024, 128, fake, 1 << 30, None, None)
        assert st_noalloc == want and st_ws == want, (geom, st_noalloc, st_ws)
