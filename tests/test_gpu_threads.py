"""libkvc8 called from two host threads at once, each on its own stream.

The library keeps small per-device caches of launch facts (SM count, CTAs per
SM of each kernel variant) in atomic words.  Here two threads store and gather
their own batches concurrently -- with geometries that give the same kernel
variants different shared-memory sizes, so the cached entries keep changing
under each other -- and every result is compared with the oracle, bit for bit.
The ctypes calls release the GIL, so the two threads' host code really runs at
the same time.
"""
import threading

import numpy as np
import pytest
import torch

import oracle
import dequant_kvc8_store_gb300 as kv
from dequant_kvc8_store_gb300 import workloads as W
from dequant_kvc8_store_gb300.device import DeviceBatch
from test_gpu_parity import _assert_bits_equal, _assert_pool_equal, _oracle_store

pytestmark = pytest.mark.gpu


def _batches(tag, seed):
    out = []
    for i, (H, D, mode) in enumerate([(8, 128, 0), (4, 64, 1), (2, 128, 1), (8, 64, 2),
                                       (6, 128, 1)]):
        out.append(W.make_workload(f"{tag}{i}", q_lens=[40, 1, 77, 5], ctx_before=[0, 30, 9, 64],
                                   kv_heads=H, head_dim=D, block_size=16, num_blocks=40,
                                   quant_mode=mode, seed=seed + i))
    return out


def test_two_host_threads_two_streams():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kv.load()
    work = {0: _batches("thr-a", 600), 1: _batches("thr-b", 700)}
    done = {0: [], 1: []}
    errors = []
    start = threading.Barrier(2)

    def run(k):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            batches = [DeviceBatch(w, fill_out=0xFFFF) for w in work[k]]
            torch.cuda.synchronize()
            start.wait()
            for _ in range(3):  # the same calls again: the results must not change
                for d in batches:
                    d.store(s)  # stores into a pool already holding the batch: same bits
                    d.gather(s)
            s.synchronize()
            done[k] = batches
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(k,)) for k in (0, 1)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for k in (0, 1):
        for w, d in zip(work[k], done[k]):
            assert d.error_code() == 0
            want_pool = _oracle_store(w)
            _assert_pool_equal(d.host_caches(), want_pool)
            ko, vo = oracle.dequant_gather(w.quant_mode, *want_pool, w.block_table,
                                           w.context_lengths)
            gk, gv = d.host_outputs()
            _assert_bits_equal(gk, ko, "k_out")
            _assert_bits_equal(gv, vo, "v_out")
