"""The allocation-free dequant-gather (kvc8_dequant_gather_noalloc).

Some callers cannot allocate device memory where they gather -- a plugin inside
a runtime that owns all device memory, or a serving loop that must not
allocate once running -- so they cannot pass the workspace that
kvc8_dequant_gather needs.  The no-alloc entry point keeps that scratch in a
fixed array inside the library instead.  These tests check, through the C ABI,
that it returns exactly what the workspace entry point returns, on two calls in
a row with different batches (so a plan left over from the first call would
show), and that batches beyond its fixed size are refused.
"""
import ctypes

import numpy as np
import pytest
import torch

import dequant_kvc8_store_gb300 as kv
from dequant_kvc8_store_gb300 import workloads as W
from dequant_kvc8_store_gb300.device import DeviceBatch


def _compare_with_workspace_gather(w, offsets=None, layout="dense"):
    d = DeviceBatch(w, offsets=offsets, out_layout=layout, fill_out=0xFFFF)
    d.gather()  # the entry point with a caller workspace
    want_k, want_v = d.host_outputs()
    d.k_out.view(torch.int16).fill_(-1)
    d.v_out.view(torch.int16).fill_(-1)
    ko = d.k_out
    kv.kvc8_dequant_gather_noalloc(d.g, d.k_cache, d.v_cache, d.k_scale, d.v_scale,
                                   d.block_table, d.context_lengths, d.offsets, ko, d.v_out,
                                   d.out_rows, ko.stride(0), ko.stride(1), d.dev_error)
    got_k, got_v = d.host_outputs()
    assert d.error_code() == 0
    # tolerance: none (0 ULP), as for every gather comparison in this suite
    assert np.array_equal(got_k, want_k)
    assert np.array_equal(got_v, want_v)


@pytest.mark.gpu
def test_noalloc_gather_matches_workspace_gather_twice():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    rng = np.random.default_rng(404)
    first = W.make_workload("noalloc-a", q_lens=np.zeros(300, np.int64),
                            ctx_before=rng.integers(0, 600, size=300), kv_heads=2,
                            head_dim=64, block_size=16, num_blocks=300 * 38, quant_mode=0,
                            seed=404, with_store=False)
    second = W.make_workload("noalloc-b", q_lens=np.zeros(5, np.int64),
                             ctx_before=[129, 1, 0, 640, 77], kv_heads=8, head_dim=128,
                             block_size=64, num_blocks=60, quant_mode=1, seed=405,
                             with_store=False)
    _compare_with_workspace_gather(first)
    lens = second.context_lengths.astype(np.int64)
    offsets = np.concatenate([[3], 3 + np.cumsum(lens + 2)[:-1]])
    _compare_with_workspace_gather(second, offsets=offsets, layout="head_major")


def test_noalloc_gather_refuses_batches_beyond_its_scratch():
    g = kv.Geom(kv.NOALLOC_MAX_SEQS + 1, 8, 128, 16, 64, 8, 0)
    fake = 1 << 20  # never dereferenced: the size check comes first
    st = kv.load().kvc8_dequant_gather_noalloc(ctypes.byref(g), *([fake] * 6), None, fake, fake,
                                               10, 1024, 128, None, None)
    assert st == kv.ERR_UNSUPPORTED
