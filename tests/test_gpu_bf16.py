"""The bf16 paged KV cache (no quantisation) on the GPU against the oracle.

kvc8_store_bf16 and kvc8_gather_bf16 move bf16 rows without changing them, so
every comparison is exact: the whole pool after the store (stray writes show)
and every output row, including rows the gather must leave untouched.  The
prior pool contents are seeded random bits, so a row that is not written keeps
a value that no written row can match by chance.
"""
import numpy as np
import pytest
import torch

import oracle
import dequant_kvc8_store_gb300 as kv
from dequant_kvc8_store_gb300 import workloads as W
from test_gpu_parity import _random_geometry

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kv.load()
    yield
    torch.cuda.synchronize()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _bits(t):
    return t.cpu().numpy().view(np.uint16)


def _pool(w, seed):
    rng = np.random.default_rng([seed, 16])
    shape = (w.num_blocks, w.kv_heads, w.block_size, w.head_dim)
    return (rng.integers(0, 1 << 16, size=shape, dtype=np.uint16),
            rng.integers(0, 1 << 16, size=shape, dtype=np.uint16))


def _assert_equal(got, want, name):
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        raise AssertionError(f"{name}: {len(bad)} mismatches, first at {bad[:5].tolist()}")


def check_bf16(w, *, x_pad=0, head_major_in=False, offsets=None, head_major_out=False,
               out_pad_rows=0, fill=0xFFFF, stream=None):
    """Store w's new tokens into a bf16 pool and gather every sequence back."""
    H, D = w.kv_heads, w.head_dim
    g = kv.Geom(w.num_seqs, H, D, w.block_size, w.num_blocks, w.max_blocks_per_seq, 0)
    kc0, vc0 = _pool(w, w.seed)
    kc, vc = _dev(kc0.view(np.int16)), _dev(vc0.view(np.int16))
    bt = _dev(w.block_table)
    ctx = _dev(w.context_kv_lens)
    lens = _dev(w.context_lengths)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    N = w.num_tokens
    if N:
        def states(x):
            x = torch.from_numpy(x.view(np.int16))
            if head_major_in:  # [H][N][D + x_pad] storage, viewed as [N][H][D]
                full = torch.zeros((H, N, D + x_pad), dtype=torch.int16)
                full[:, :, :D] = x.transpose(0, 1)
                return full.cuda().transpose(0, 1)[:, :, :D]
            full = torch.zeros((N, H, D + x_pad), dtype=torch.int16)
            full[:, :, :D] = x
            return full.cuda()[:, :, :D]
        kx, vx = states(w.k_states), states(w.v_states)
        assert kx.stride() == vx.stride() and kx.stride(2) == 1
        cu = None if w.cu_q_lens is None else _dev(w.cu_q_lens)
        kv.kvc8_store_bf16(g, N, kx, vx, kx.stride(0), kx.stride(1), kc, vc, bt, cu, ctx, err,
                           stream)
    rows = (w.total_context if offsets is None
            else int(max([o + l for o, l in zip(offsets, w.context_lengths)] + [0])))
    rows += out_pad_rows
    fill16 = fill - 65536 if fill > 32767 else fill

    def out():
        if head_major_out:  # [H][rows][D] storage viewed as [rows][H][D]
            return torch.full((H, rows, D), fill16, dtype=torch.int16,
                              device="cuda").transpose(0, 1)
        return torch.full((rows, H, D), fill16, dtype=torch.int16, device="cuda")
    ko, vo = out(), out()
    ws = torch.empty(kv.kvc8_gather_workspace_bytes(g), dtype=torch.uint8, device="cuda")
    off_d = None if offsets is None else _dev(np.asarray(offsets, np.int64))
    kv.kvc8_gather_bf16(g, kc, vc, bt, lens, off_d, ko, vo, rows, ko.stride(0), ko.stride(1), ws,
                        ws.numel(), err, stream)
    assert kv.kvc8_get_error(err, stream=stream) == 0

    want_k, want_v = kc0.copy(), vc0.copy()
    if N:
        oracle.store_bf16(w.k_states, w.v_states, want_k, want_v, w.block_table,
                          w.cu_q_lens if w.cu_q_lens is not None else np.arange(N + 1, dtype=np.int32),
                          w.context_kv_lens)
    _assert_equal(_bits(kc), want_k, "k_cache")
    _assert_equal(_bits(vc), want_v, "v_cache")
    ok = np.full((rows, H, D), fill, np.uint16)
    ov = np.full((rows, H, D), fill, np.uint16)
    oracle.gather_bf16(want_k, want_v, w.block_table, w.context_lengths,
                       None if offsets is None else np.asarray(offsets, np.int64), ok, ov)
    _assert_equal(_bits(ko.contiguous()), ok, "k_out")
    _assert_equal(_bits(vo.contiguous()), ov, "v_out")


SMALL = [
    dict(q_lens=[0, 1, 17, 40, 3], ctx_before=[0, 5, 16, 30, 0], kv_heads=2, head_dim=64,
         block_size=16, num_blocks=40),
    dict(q_lens=[200, 1, 129], ctx_before=[0, 300, 127], kv_heads=4, head_dim=128,
         block_size=128, num_blocks=16),
    dict(q_lens=[3, 2, 5], ctx_before=[2, 0, 1], kv_heads=1, head_dim=16, block_size=1,
         num_blocks=40),
    dict(q_lens=[33, 7], ctx_before=[5, 60], kv_heads=3, head_dim=48, block_size=8,
         num_blocks=40),
    dict(q_lens=[70, 0, 1], ctx_before=[10, 0, 95], kv_heads=2, head_dim=256, block_size=32,
         num_blocks=24),
    dict(q_lens=[70, 5], ctx_before=[10, 33], kv_heads=5, head_dim=80, block_size=16,
         num_blocks=30),
    dict(q_lens=[1] * 7, ctx_before=[0, 1, 15, 16, 17, 100, 63], kv_heads=8, head_dim=128,
         block_size=16, num_blocks=64, decode_null_cu=True),
    dict(q_lens=[300, 1, 1, 650], ctx_before=[0, 4000, 31, 700], kv_heads=8, head_dim=128,
         block_size=64, num_blocks=300),
    # a token's rows above the 8 chunks a lane keeps in flight (2*16*256/8 = 1024 chunks)
    dict(q_lens=[41, 1, 70], ctx_before=[0, 9, 31], kv_heads=16, head_dim=256,
         block_size=16, num_blocks=40),
]


@pytest.mark.parametrize("i", range(len(SMALL)))
def test_bf16_small_ragged(i):
    w = W.make_workload(f"bf16small{i}", seed=150 + i, quant_mode=0, **SMALL[i])
    check_bf16(w)


@pytest.mark.parametrize("i", range(32))
def test_bf16_random_geometries(i):
    # the parity file's seeded random problems (scales unused by this path)
    g = _random_geometry(2000 + i)
    g["quant_mode"] = 0
    w = W.make_workload(f"bf16rand{i}", seed=700 + i, **g)
    check_bf16(w)


def test_bf16_strided_inputs_and_outputs():
    w = W.make_workload("bf16strided", q_lens=[45, 0, 130, 2], ctx_before=[3, 64, 0, 17],
                        kv_heads=4, head_dim=96, block_size=32, num_blocks=40, quant_mode=0,
                        seed=170)
    check_bf16(w, x_pad=8, head_major_in=True, head_major_out=True, out_pad_rows=5)
    lens = w.context_lengths.astype(np.int64)
    offsets = np.concatenate([[7], 7 + np.cumsum(lens + 3)[:-1]])
    check_bf16(w, x_pad=24, offsets=offsets, out_pad_rows=2)


def test_bf16_side_stream_and_gather_only():
    w = W.make_workload("bf16side", q_lens=[0, 0, 0], ctx_before=[129, 1, 640], kv_heads=8,
                        head_dim=128, block_size=64, num_blocks=30, quant_mode=0, seed=171,
                        with_store=False)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        check_bf16(w, stream=s)
    check_bf16(w)


def test_bf16_empty_calls_are_noops():
    g = kv.Geom(0, 2, 64, 16, 4, 2, 0)
    kv.kvc8_store_bf16(g, 0, None, None, 0, 0, None, None, None, None, None)
    kv.kvc8_gather_bf16(g, None, None, None, None, None, None, None, 0, 0, 0, None, 0)
    w = W.make_workload("bf16zero", q_lens=[0, 0], ctx_before=[0, 0], kv_heads=2, head_dim=64,
                        block_size=16, num_blocks=4, quant_mode=0, seed=172, with_store=False)
    check_bf16(w, out_pad_rows=4, fill=0x1234)


def test_bf16_store_reports_bad_block_and_skips_it():
    w = W.make_workload("bf16bad", q_lens=[5, 3], ctx_before=[0, 0], kv_heads=2, head_dim=64,
                        block_size=16, num_blocks=8, quant_mode=0, seed=173)
    H, D = w.kv_heads, w.head_dim
    g = kv.Geom(w.num_seqs, H, D, w.block_size, w.num_blocks, w.max_blocks_per_seq, 0)
    bt = w.block_table.copy()
    bt[1, 0] = w.num_blocks  # out of the pool
    kc0, vc0 = _pool(w, 173)
    kc, vc = _dev(kc0.view(np.int16)), _dev(vc0.view(np.int16))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kx = _dev(w.k_states.view(np.int16))
    vx = _dev(w.v_states.view(np.int16))
    kv.kvc8_store_bf16(g, w.num_tokens, kx, vx, H * D, D, kc, vc, _dev(bt), _dev(w.cu_q_lens),
                       _dev(w.context_kv_lens), err)
    assert kv.kvc8_get_error(err, reset=True) == kv.DEV_BAD_BLOCK_ID
    # sequence 0 is stored as usual; sequence 1 writes nothing
    want_k, want_v = kc0.copy(), vc0.copy()
    oracle.store_bf16(w.k_states[:5], w.v_states[:5], want_k, want_v, bt[:1],
                      w.cu_q_lens[:2], w.context_kv_lens[:1])
    _assert_equal(_bits(kc), want_k, "k_cache")
    _assert_equal(_bits(vc), want_v, "v_cache")


def test_bf16_gather_reports_short_output():
    w = W.make_workload("bf16short", q_lens=[0, 0], ctx_before=[40, 17], kv_heads=2,
                        head_dim=64, block_size=16, num_blocks=8, quant_mode=0, seed=174,
                        with_store=False)
    H, D = w.kv_heads, w.head_dim
    g = kv.Geom(w.num_seqs, H, D, w.block_size, w.num_blocks, w.max_blocks_per_seq, 0)
    kc0, vc0 = _pool(w, 174)
    kc, vc = _dev(kc0.view(np.int16)), _dev(vc0.view(np.int16))
    rows = w.total_context - 1
    ko = torch.zeros((rows, H, D), dtype=torch.int16, device="cuda")
    vo = torch.zeros_like(ko)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(kv.kvc8_gather_workspace_bytes(g), dtype=torch.uint8, device="cuda")
    kv.kvc8_gather_bf16(g, kc, vc, _dev(w.block_table), _dev(w.context_lengths), None, ko, vo,
                        rows, H * D, D, ws, ws.numel(), err)
    assert kv.kvc8_get_error(err, reset=True) == kv.DEV_OUT_ROW_RANGE
    # Sequence 1's second tile (its row 16, output row 56) does not fit and is
    # skipped whole; every tile before it fits and is gathered.
    ok = np.zeros((rows + 1, H, D), np.uint16)
    ov = np.zeros((rows + 1, H, D), np.uint16)
    oracle.gather_bf16(kc0, vc0, w.block_table, w.context_lengths, None, ok, ov)
    _assert_equal(_bits(ko), ok[:rows], "k_out")
    _assert_equal(_bits(vo), ov[:rows], "v_out")


def test_bf16_full_size_prefill():
    check_bf16(W.prefill())


def test_bf16_decode_shaped():
    """256 single-token sequences (no cu_q_lens), contexts up to 1024 tokens."""
    rng = np.random.default_rng(175)
    ctx = rng.integers(0, 1024, size=256)
    w = W.make_workload("bf16decode", q_lens=np.ones(256, np.int64), ctx_before=ctx, kv_heads=8,
                        head_dim=128, block_size=128, num_blocks=256 * 9, quant_mode=0,
                        seed=175, decode_null_cu=True)
    check_bf16(w)
