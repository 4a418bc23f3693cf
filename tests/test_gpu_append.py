"""The fused append + gather (kvc8_append_gather) on the GPU against the oracle.

By definition the fused call equals kvc8_store followed by kvc8_dequant_gather
of the whole context, so the expected values are the oracle's store and then
the oracle's gather with context_lengths = cached + new tokens.  Every
comparison is exact: the whole pool after the call, and every output row,
including rows that no sequence covers.
"""
import numpy as np
import pytest
import torch

import oracle
import dequant_kvc8_store_gb300 as kv
from dequant_kvc8_store_gb300 import workloads as W
from dequant_kvc8_store_gb300.device import DeviceBatch
from test_gpu_parity import (SMALL, _assert_bits_equal, _assert_pool_equal, _oracle_store,
                             _random_geometry)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kv.load()
    yield
    torch.cuda.synchronize()


def check_fused(w, *, offsets=None, out_layout="dense", out_pad_rows=0, fill=0xFFFF,
                planned=False, stream=None):
    d = DeviceBatch(w, offsets=offsets, out_layout=out_layout, out_pad_rows=out_pad_rows,
                    fill_out=fill)
    if planned:
        d.build_append_metadata(stream=stream)
        d.append_gather_planned(stream)
    else:
        d.append_gather(stream)
    assert d.error_code() == 0
    want_pool = _oracle_store(w)
    _assert_pool_equal(d.host_caches(), want_pool)
    kc, vc, ks, vs = want_pool
    H, D = w.kv_heads, w.head_dim
    ko = np.full((d.out_rows, H, D), fill, np.uint16)
    vo = np.full((d.out_rows, H, D), fill, np.uint16)
    oracle.dequant_gather(w.quant_mode, kc, vc, ks, vs, w.block_table, w.context_lengths,
                          None if offsets is None else np.asarray(offsets, np.int64), ko, vo)
    gk, gv = d.host_outputs()
    _assert_bits_equal(gk, ko, "k_out")
    _assert_bits_equal(gv, vo, "v_out")
    return d


@pytest.mark.parametrize("i", range(len(SMALL)))
def test_fused_small_ragged(i):
    w = W.make_workload(f"fused{i}", seed=250 + i, **SMALL[i])
    check_fused(w)


@pytest.mark.parametrize("i", range(48))
def test_fused_random_geometries(i):
    # the parity file's seeded random problems, through the fused call (its
    # long appends take the store + plan + gather route)
    w = W.make_workload(f"frand{i}", seed=600 + i, **_random_geometry(1000 + i))
    check_fused(w)


def test_fused_decode_shapes():
    # one new token per sequence, with and without cu_q_lens, across block edges
    ctx = [0, 1, 15, 16, 17, 31, 32, 100, 127, 128, 129, 300]
    for null_cu in (False, True):
        for mode in (0, 1):
            w = W.make_workload(f"fdec{null_cu}{mode}", q_lens=np.ones(len(ctx), np.int64),
                                ctx_before=ctx, kv_heads=8, head_dim=128, block_size=16,
                                num_blocks=len(ctx) * 20, quant_mode=mode, seed=270 + mode,
                                decode_null_cu=null_cu)
            check_fused(w)


def test_fused_strided_padded_output_and_given_offsets():
    w = W.make_workload("fpad", q_lens=[13, 1, 70], ctx_before=[3, 40, 0], kv_heads=4,
                        head_dim=64, block_size=16, num_blocks=32, quant_mode=0, seed=271)
    lens = w.context_lengths.astype(np.int64)
    offsets = np.concatenate([[2], 2 + np.cumsum(lens + np.array([5, 0, 9]))[:-1]])
    check_fused(w, offsets=offsets, out_layout="head_major", out_pad_rows=7)
    check_fused(w, offsets=offsets, out_layout="dense", out_pad_rows=3, planned=True)
    check_fused(w, out_layout="head_major")


def test_fused_gather_only_and_side_stream():
    w = W.make_workload("fgo", q_lens=[0, 0, 0], ctx_before=[129, 1, 640], kv_heads=8,
                        head_dim=128, block_size=64, num_blocks=30, quant_mode=1, seed=272,
                        with_store=False)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        check_fused(w, stream=s)
    check_fused(w)


def test_fused_planned_metadata_shared_by_two_layers():
    """One plan, two layers: each layer has its own pool and new rows."""
    kw = dict(q_lens=[1, 1, 40, 1], ctx_before=[63, 64, 7, 500], kv_heads=8, head_dim=128,
              block_size=64, num_blocks=64, quant_mode=0)
    layer0 = W.make_workload("layer0", seed=273, **kw)
    layer1 = W.make_workload("layer1", seed=274, **kw)
    d0, d1 = DeviceBatch(layer0, fill_out=0xFFFF), DeviceBatch(layer1, fill_out=0xFFFF)
    off = torch.full((layer0.num_seqs,), -1, dtype=torch.int64, device="cuda")
    d0.build_append_metadata(offsets_out=off)
    d1.workspace = d0.workspace  # the layers run one after the other on one stream
    d0.append_gather_planned()
    d1.append_gather_planned()
    assert d0.error_code() == 0 and d1.error_code() == 0
    assert np.array_equal(off.cpu().numpy(), oracle.exclusive_cumsum(layer0.context_lengths))
    for w, d in ((layer0, d0), (layer1, d1)):
        want_pool = _oracle_store(w)
        _assert_pool_equal(d.host_caches(), want_pool)
        ko, vo = oracle.dequant_gather(w.quant_mode, *want_pool, w.block_table,
                                       w.context_lengths)
        gk, gv = d.host_outputs()
        _assert_bits_equal(gk, ko, "k_out")
        _assert_bits_equal(gv, vo, "v_out")


def test_fused_matches_separate_calls_bit_for_bit():
    w = W.make_workload("fsep", q_lens=[200, 1, 129, 1], ctx_before=[0, 300, 127, 5],
                        kv_heads=4, head_dim=128, block_size=128, num_blocks=24, quant_mode=0,
                        seed=275, outlier_channels=4)
    a = DeviceBatch(w, fill_out=0)
    a.store()
    a.gather()
    b = DeviceBatch(w, fill_out=0)
    b.append_gather()
    assert a.error_code() == 0 and b.error_code() == 0
    for x, y in zip(a.host_caches(), b.host_caches()):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    for x, y in zip(a.host_outputs(), b.host_outputs()):
        assert np.array_equal(x, y)


def test_fused_reports_short_output_and_stores_anyway():
    w = W.make_workload("fshort", q_lens=[1, 1], ctx_before=[20, 5], kv_heads=2, head_dim=64,
                        block_size=16, num_blocks=8, quant_mode=0, seed=276)
    d = DeviceBatch(w, fill_out=0)
    d.out_rows -= 1  # the last sequence's new row (output row 26) falls outside
    d.append_gather()
    assert d.error_code(reset=True) == kv.DEV_OUT_ROW_RANGE
    _assert_pool_equal(d.host_caches(), _oracle_store(w))


def _check_fused_full_size(w):
    """One fused call on a full-size batch: the whole pool, and every element
    of the output (each sequence's cached rows and its appended rows) against
    the oracle's store followed by its gather."""
    d = DeviceBatch(w, fill_out=0xFFFF)
    d.append_gather()
    assert d.error_code() == 0
    oracle.store(w.quant_mode, w.k_states, w.v_states, w.k_cache, w.v_cache, w.k_scale,
                 w.v_scale, w.block_table, w.cu_q_lens, w.context_kv_lens)
    _assert_pool_equal(d.host_caches(), (w.k_cache, w.v_cache, w.k_scale, w.v_scale))
    ko, vo = oracle.dequant_gather(w.quant_mode, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                                   w.block_table, w.context_lengths)
    gk, gv = d.host_outputs()
    _assert_bits_equal(gk, ko, "k_out")
    del gk, ko
    _assert_bits_equal(gv, vo, "v_out")


def test_fused_full_size_decode():
    """The decode batch at full size through the fused kernel (256 appended
    tokens, 1.13 M gathered positions)."""
    _check_fused_full_size(W.decode())


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_fused_long_append_takes_store_then_gather(mode):
    """More than 16 384 appended rows: the call runs the store kernel, a plan
    over cached + new positions and the gather; same bits as the oracle."""
    w = W.make_workload(f"flong{mode}", q_lens=[700, 500, 1, 0], ctx_before=[30, 0, 900, 64],
                        kv_heads=8, head_dim=128, block_size=64, num_blocks=4 * 16 + 4,
                        quant_mode=mode, seed=280 + mode)
    assert w.num_tokens * 2 * w.kv_heads > 16384
    check_fused(w)
    lens = w.context_lengths.astype(np.int64)
    offsets = np.concatenate([[5], 5 + np.cumsum(lens + 3)[:-1]])
    check_fused(w, offsets=offsets, out_layout="head_major", out_pad_rows=4)


def test_fused_long_decode_append_and_small_workspace():
    """1100 single-token sequences (cu_q_lens NULL) take the long path; with a
    workspace that only holds the plan the call stays on the fused kernel."""
    rng = np.random.default_rng(290)
    ctx = rng.integers(0, 300, size=1100)
    w = W.make_workload("flongdec", q_lens=np.ones(1100, np.int64), ctx_before=ctx, kv_heads=8,
                        head_dim=64, block_size=64, num_blocks=1100 * 5, quant_mode=0,
                        seed=290, decode_null_cu=True)
    check_fused(w)
    d = DeviceBatch(w, fill_out=0xFFFF)
    spans_bytes = (4 * w.num_seqs + 255) // 256 * 256
    d.ws_bytes = kv.kvc8_gather_workspace_bytes(d.g) - spans_bytes  # the plan alone
    d.append_gather()
    assert d.error_code() == 0
    want_pool = _oracle_store(w)
    _assert_pool_equal(d.host_caches(), want_pool)
    ko, vo = oracle.dequant_gather(w.quant_mode, *want_pool, w.block_table, w.context_lengths)
    gk, gv = d.host_outputs()
    _assert_bits_equal(gk, ko, "k_out")
    _assert_bits_equal(gv, vo, "v_out")


@pytest.mark.parametrize("make", [W.prefill, W.mixed], ids=["prefill", "mixed"])
def test_fused_full_size_long_append(make):
    """The prefill and mixed batches through the fused call (more than 16 384
    appended rows: store, span plan, gather)."""
    w = make()
    assert w.num_tokens * 2 * w.kv_heads > 16384
    _check_fused_full_size(w)
