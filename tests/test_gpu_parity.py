"""libkvc8 on the GPU against the CPU oracle, bit for bit.

Every comparison is exact: int8 codes, fp32 scales (as bit patterns), page
placement (the whole pool, so stray writes show), untouched output rows, and
the dequantised bf16 output (0 ULP).  Inputs come from the seeded generators
in ``dequant_kvc8_store_gb300.workloads``; expected values come only from the
oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import dequant_kvc8_store_gb300 as kv
from dequant_kvc8_store_gb300 import workloads as W
from dequant_kvc8_store_gb300.device import DeviceBatch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kv.load()
    yield
    torch.cuda.synchronize()


def _oracle_store(w):
    """Run the oracle's store on copies of the pool; returns the expected pool."""
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    ks, vs = w.k_scale.copy(), w.v_scale.copy()
    if w.has_store:
        oracle.store(w.quant_mode, w.k_states, w.v_states, kc, vc, ks, vs, w.block_table,
                     w.cu_q_lens, w.context_kv_lens)
    return kc, vc, ks, vs


def _assert_pool_equal(got, want):
    for g_, w_, name in zip(got, want, ("k_cache", "v_cache", "k_scale", "v_scale")):
        if g_.dtype == np.float32:
            g_, w_ = g_.view(np.uint32), w_.view(np.uint32)
        if not np.array_equal(g_, w_):
            bad = np.argwhere(g_ != w_)
            raise AssertionError(f"{name}: {len(bad)} mismatches, first at {bad[:5].tolist()}")


def _assert_bits_equal(got, want, name):
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i = tuple(bad[0])
        raise AssertionError(f"{name}: {len(bad)} mismatches, first at {bad[:5].tolist()}: "
                             f"got {got[i]:#06x} want {want[i]:#06x}")


def check_full(w, *, offsets=None, out_layout="dense", out_pad_rows=0, fill=0xFFFF,
               planned=False, stream=None):
    d = DeviceBatch(w, offsets=offsets, out_layout=out_layout, out_pad_rows=out_pad_rows,
                    fill_out=fill)
    d.store(stream)
    if planned:
        d.build_metadata(stream=stream)
        d.gather_planned(stream)
    else:
        d.gather(stream)
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


# ---- the tiny round trip and a sweep of small ragged problems -----------------------

def test_tiny_round_trip():
    check_full(W.tiny())


SMALL = [
    dict(q_lens=[0, 1, 17, 40, 3], ctx_before=[0, 5, 16, 30, 0], kv_heads=2, head_dim=64,
         block_size=16, num_blocks=40, quant_mode=0),
    dict(q_lens=[200, 1, 129], ctx_before=[0, 300, 127], kv_heads=4, head_dim=128,
         block_size=128, num_blocks=16, quant_mode=1),
    dict(q_lens=[3, 2, 5], ctx_before=[2, 0, 1], kv_heads=1, head_dim=16, block_size=1,
         num_blocks=40, quant_mode=0),
    dict(q_lens=[33, 7], ctx_before=[5, 60], kv_heads=3, head_dim=48, block_size=8,
         num_blocks=40, quant_mode=0),
    dict(q_lens=[33, 7], ctx_before=[5, 60], kv_heads=3, head_dim=48, block_size=8,
         num_blocks=40, quant_mode=1),
    dict(q_lens=[70, 0, 1], ctx_before=[10, 0, 95], kv_heads=2, head_dim=256, block_size=32,
         num_blocks=24, quant_mode=0),
    dict(q_lens=[70, 5], ctx_before=[10, 33], kv_heads=5, head_dim=80, block_size=16,
         num_blocks=30, quant_mode=1),
    dict(q_lens=[1] * 7, ctx_before=[0, 1, 15, 16, 17, 100, 63], kv_heads=8, head_dim=128,
         block_size=16, num_blocks=64, quant_mode=0, decode_null_cu=True),
    dict(q_lens=[300, 1, 1, 650], ctx_before=[0, 4000, 31, 700], kv_heads=8, head_dim=128,
         block_size=64, num_blocks=300, quant_mode=1),
    dict(q_lens=[129, 255, 1], ctx_before=[0, 1, 1023], kv_heads=8, head_dim=128,
         block_size=128, num_blocks=40, quant_mode=0, outlier_channels=4),
    # K and V rows of a token above 4 KB (the unstaged store path)
    dict(q_lens=[77, 3, 140], ctx_before=[5, 0, 60], kv_heads=16, head_dim=128,
         block_size=32, num_blocks=30, quant_mode=0),
    dict(q_lens=[41, 1, 70], ctx_before=[0, 9, 31], kv_heads=12, head_dim=256,
         block_size=16, num_blocks=40, quant_mode=1),
    # one static scale per (block, kv head)
    dict(q_lens=[0, 1, 17, 40, 3], ctx_before=[0, 5, 16, 30, 0], kv_heads=2, head_dim=64,
         block_size=16, num_blocks=40, quant_mode=2),
    dict(q_lens=[33, 7], ctx_before=[5, 60], kv_heads=3, head_dim=48, block_size=8,
         num_blocks=40, quant_mode=2),
    dict(q_lens=[1] * 7, ctx_before=[0, 1, 15, 16, 17, 100, 63], kv_heads=8, head_dim=128,
         block_size=16, num_blocks=64, quant_mode=2, decode_null_cu=True),
    dict(q_lens=[77, 3, 140], ctx_before=[5, 0, 60], kv_heads=16, head_dim=128,
         block_size=32, num_blocks=30, quant_mode=2, block_scale_range=(0.002, 0.5)),
    # odd block size: the small dynamic-scale gather keeps whole tiles
    dict(q_lens=[20, 1, 9], ctx_before=[6, 13, 0], kv_heads=4, head_dim=64, block_size=7,
         num_blocks=24, quant_mode=0),
    # static per-channel scales on kv_heads x head_dim = 8448 channels (each
    # lane keeps its channels' quantities in registers: no table size limit)
    dict(q_lens=[20, 7], ctx_before=[3, 40], kv_heads=33, head_dim=256, block_size=16,
         num_blocks=12, quant_mode=1),
    # one 16-channel lane per row: 30 of a warp's 32 lanes idle
    dict(q_lens=[9, 1, 30], ctx_before=[0, 7, 2], kv_heads=1, head_dim=16, block_size=4,
         num_blocks=24, quant_mode=1),
    dict(q_lens=[9, 1, 30], ctx_before=[0, 7, 2], kv_heads=1, head_dim=16, block_size=4,
         num_blocks=24, quant_mode=2),
    # 64 kv heads of 256 channels: a token spans 64 warps, eight CTAs
    dict(q_lens=[5, 1, 9], ctx_before=[0, 3, 17], kv_heads=64, head_dim=256, block_size=16,
         num_blocks=8, quant_mode=0),
    dict(q_lens=[5, 1, 9], ctx_before=[0, 3, 17], kv_heads=64, head_dim=256, block_size=16,
         num_blocks=8, quant_mode=1),
]


@pytest.mark.parametrize("i", range(len(SMALL)))
def test_small_ragged(i):
    w = W.make_workload(f"small{i}", seed=50 + i, **SMALL[i])
    check_full(w)


def _random_geometry(i):
    """Seeded small problem i: head_dim any multiple of 16 up to 256, 1-16 kv
    heads, block sizes from 1 to 128 (odd ones included), 1-39 sequences
    with ragged new and cached lengths on three scales, all three scale
    modes, and the decode form (cu_q_lens = None) now and then."""
    rng = np.random.default_rng([4242, i])
    D = 16 * int(rng.integers(1, 17))
    H = int(rng.integers(1, 17))
    bs = int(rng.choice([1, 2, 3, 5, 7, 8, 16, 17, 31, 32, 48, 64, 96, 128]))
    B = int(rng.integers(1, 40))
    mode = int(rng.integers(0, 3))
    decode = bool(rng.random() < 0.2)
    q = np.ones(B, np.int64) if decode else rng.integers(0, int(rng.choice([3, 40, 300])), size=B)
    ctx = rng.integers(0, int(rng.choice([5, 100, 1000])), size=B)
    mb = int(((ctx + q + bs - 1) // bs).max())
    return dict(q_lens=q, ctx_before=ctx, kv_heads=H, head_dim=D, block_size=bs,
                num_blocks=max(B * max(mb, 1) + int(rng.integers(0, 9)), 1), quant_mode=mode,
                decode_null_cu=decode)


@pytest.mark.parametrize("i", range(96))
def test_random_geometries(i):
    w = W.make_workload(f"rand{i}", seed=300 + i, **_random_geometry(i))
    check_full(w)


@pytest.mark.parametrize("mode", [0, 1])
def test_many_sequences(mode):
    """1 500 sequences: more than the gather keeps of the tile table in shared
    memory (it searches the plan in global memory)."""
    rng = np.random.default_rng(90 + mode)
    B = 1500
    ctx = rng.integers(0, 40, size=B)
    q = rng.integers(0, 3, size=B)
    w = W.make_workload(f"many{mode}", q_lens=q, ctx_before=ctx, kv_heads=2, head_dim=64,
                        block_size=16, num_blocks=B * 3 + 8, quant_mode=mode, seed=90 + mode)
    check_full(w)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_strided_input_states(mode):
    """New K/V rows read through token and head strides wider than the
    rows (a view into a larger buffer, as from a fused projection)."""
    w = W.make_workload(f"xstride{mode}", q_lens=[37, 1, 90], ctx_before=[5, 18, 0], kv_heads=4,
                        head_dim=96, block_size=16, num_blocks=40, quant_mode=mode, seed=95 + mode)
    d = DeviceBatch(w, fill_out=0xFFFF)
    N, H, D = w.num_tokens, w.kv_heads, w.head_dim
    for name in ("k_states", "v_states"):
        x = getattr(d, name)
        big = torch.full((N, H + 1, D + 24), 0x7F80, dtype=x.dtype, device=x.device)
        big[:, :H, :D] = x
        setattr(d, name, big[:, :H, :D])
    assert d.k_states.stride() == ((H + 1) * (D + 24), D + 24, 1)
    d.store()
    d.gather()
    assert d.error_code() == 0
    want_pool = _oracle_store(w)
    _assert_pool_equal(d.host_caches(), want_pool)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_pool_declared_beyond_2_31_rows(mode):
    """A pool declared with more than 2^31 rows (num_blocks * kv_heads *
    block_size) makes the store index cache rows in 64 bits.  Only the first
    blocks are allocated, and the block table names only those."""
    w = W.make_workload(f"rows64_{mode}", q_lens=[37, 1, 50], ctx_before=[3, 20, 0], kv_heads=2,
                        head_dim=64, block_size=16, num_blocks=40, quant_mode=mode,
                        seed=120 + mode)
    d = DeviceBatch(w, fill_out=0xFFFF)
    d.g.num_blocks = 1 << 27
    assert d.g.num_blocks * w.kv_heads * w.block_size > 2**31 - 1
    d.store()
    d.gather()
    assert d.error_code() == 0
    want_pool = _oracle_store(w)
    _assert_pool_equal(d.host_caches(), want_pool)
    kc, vc, ks, vs = want_pool
    ko = np.full((d.out_rows, w.kv_heads, w.head_dim), 0xFFFF, np.uint16)
    vo = ko.copy()
    oracle.dequant_gather(w.quant_mode, kc, vc, ks, vs, w.block_table, w.context_lengths, None,
                          ko, vo)
    gk, gv = d.host_outputs()
    _assert_bits_equal(gk, ko, "k_out")
    _assert_bits_equal(gv, vo, "v_out")


def test_strided_padded_output_and_given_offsets():
    w = W.make_workload("pad", q_lens=[13, 1, 70], ctx_before=[3, 40, 0], kv_heads=4,
                        head_dim=64, block_size=16, num_blocks=32, quant_mode=0, seed=71)
    lens = w.context_lengths.astype(np.int64)
    pads = np.array([5, 0, 9])
    offsets = np.concatenate([[2], 2 + np.cumsum(lens + pads)[:-1]])
    check_full(w, offsets=offsets, out_layout="head_major", out_pad_rows=7)
    check_full(w, offsets=offsets, out_layout="dense", out_pad_rows=3)
    check_full(w, out_layout="head_major")


def test_planned_gather_and_metadata_offsets():
    w = W.make_workload("plan", q_lens=[13, 1, 70, 0], ctx_before=[3, 40, 0, 9], kv_heads=2,
                        head_dim=64, block_size=16, num_blocks=40, quant_mode=1, seed=72)
    check_full(w, planned=True)
    d = DeviceBatch(w)
    off = torch.full((w.num_seqs,), -7, dtype=torch.int64, device="cuda")
    d.build_metadata(offsets_out=off)
    torch.cuda.synchronize()
    assert np.array_equal(off.cpu().numpy(), oracle.exclusive_cumsum(w.context_lengths))


def test_side_stream_and_repeat_calls():
    w = W.make_workload("stream", q_lens=[40, 9], ctx_before=[7, 0], kv_heads=2, head_dim=64,
                        block_size=16, num_blocks=16, quant_mode=0, seed=73)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d = check_full(w, stream=s)
        first = d.host_outputs()
        d.gather(s)  # a second gather over the same cache gives the same bits
        s.synchronize()
        second = d.host_outputs()
    assert np.array_equal(first[0], second[0]) and np.array_equal(first[1], second[1])


def test_empty_calls_are_noops():
    w = W.make_workload("empty", q_lens=[0, 0], ctx_before=[0, 0], kv_heads=2, head_dim=64,
                        block_size=16, num_blocks=8, quant_mode=0, seed=74)
    d = DeviceBatch(w, out_pad_rows=4, fill_out=0x1234)
    before = d.host_caches()
    d.store()
    d.gather()
    assert d.error_code() == 0
    _assert_pool_equal(d.host_caches(), before)
    assert np.all(d.host_outputs()[0] == 0x1234)
    g0 = kv.Geom(0, 2, 64, 16, 8, 4, 0)
    kv.kvc8_dequant_gather(g0, d.k_cache, d.v_cache, d.k_scale, d.v_scale, d.block_table,
                           d.context_lengths, None, d.k_out, d.v_out, 0, 128, 64,
                           d.workspace, d.ws_bytes, d.dev_error)


# ---- inputs that drive the exact-division path -------------------------------------

def _set_states(w, k, v):
    w.k_states = k
    w.v_states = v
    return w


def _f32_to_bits(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_exact_ties_everywhere_dynamic():
    """amax = 127 * 2^e and x = (j + 1/2) * 2^e: every quotient is an exact tie
    (s = 2^e exactly), so every element takes the exact IEEE path."""
    rng = np.random.default_rng(80)
    w = W.make_workload("ties0", q_lens=[64, 33], ctx_before=[0, 5], kv_heads=4, head_dim=128,
                        block_size=32, num_blocks=16, quant_mode=0, seed=80)
    N, H, D = w.num_tokens, w.kv_heads, w.head_dim
    def gen():
        e = rng.integers(-20, 10, size=(N, H, 1)).astype(np.float32)
        j = rng.integers(-127, 127, size=(N, H, D)).astype(np.float32)
        x = (j + 0.5) * np.exp2(e)
        x[:, :, 0] = 127 * np.exp2(e[:, :, 0])
        return _f32_to_bits(x)
    check_full(_set_states(w, gen(), gen()))


def test_exact_ties_tiny_scales_dynamic():
    """Exact ties on rows whose scale 2^e straddles 2^-100: above it the
    flagged groups are recomputed in registers from one exact remainder, below
    it they take the division; amax down to 2^-106 keeps every value normal."""
    rng = np.random.default_rng(82)
    w = W.make_workload("ties_tiny", q_lens=[48, 17], ctx_before=[3, 0], kv_heads=4, head_dim=128,
                        block_size=16, num_blocks=16, quant_mode=0, seed=82)
    N, H, D = w.num_tokens, w.kv_heads, w.head_dim
    def gen():
        e = rng.integers(-113, -90, size=(N, H, 1)).astype(np.float32)
        j = rng.integers(-127, 127, size=(N, H, D)).astype(np.float32)
        x = (j + 0.5) * np.exp2(e)
        x[:, :, 0] = 127 * np.exp2(e[:, :, 0])
        x[:, :, 1::2] = np.round(x[:, :, 1::2] / np.exp2(e)) * np.exp2(e)  # half the values off the ties
        return _f32_to_bits(x)
    check_full(_set_states(w, gen(), gen()))


def test_reciprocal_traps_and_special_rows_dynamic():
    """Rows whose entries sit at amax/2 (quotients within 2e-6 of 63.5, where
    x * (1/s) and x / s round differently), all-zero rows, and rows of bf16
    subnormals (scale below the reciprocal fast-path range)."""
    rng = np.random.default_rng(81)
    w = W.make_workload("traps", q_lens=[40, 24], ctx_before=[1, 0], kv_heads=4, head_dim=64,
                        block_size=16, num_blocks=16, quant_mode=0, seed=81)
    N, H, D = w.num_tokens, w.kv_heads, w.head_dim
    def gen():
        amax = rng.integers(0x3F80, 0x4300, size=(N, H, 1)).astype(np.uint16)
        x = np.broadcast_to(amax - 0x0080, (N, H, D)).copy()  # amax / 2
        x[:, :, ::3] |= 0x8000
        x[:, :, 0] = amax[:, :, 0]
        x[:, :, 5:9] = (amax - 0x0100)  # amax / 4
        x[::7, 1, :] = 0                 # all-zero rows
        x[::5, 2, :] = rng.integers(1, 0x0080, size=(len(range(0, N, 5)), D)) | \
            (rng.integers(0, 2, size=(len(range(0, N, 5)), D)) << 15)  # subnormals
        return x.astype(np.uint16)
    check_full(_set_states(w, gen(), gen()))


def test_static_scales_extremes():
    """Static scales: exact ties (s = 2^e, x = (j + 1/2) s), saturation both
    ways, zero scales, huge and tiny scales outside the reciprocal range."""
    rng = np.random.default_rng(82)
    w = W.make_workload("static", q_lens=[50, 14], ctx_before=[0, 3], kv_heads=2, head_dim=128,
                        block_size=16, num_blocks=16, quant_mode=1, seed=82)
    N, H, D = w.num_tokens, w.kv_heads, w.head_dim
    e = rng.integers(-10, 4, size=(H, D)).astype(np.float32)
    s = np.exp2(e).astype(np.float32)
    s[0, 0:4] = 0.0
    s[0, 4:8] = np.float32(1e-38)    # below 2^-120: exact path
    s[0, 8:12] = np.float32(3e38)    # above 2^120: exact path
    s[1, 0:8] = np.float32(1e-30)    # reciprocal 1e30: saturates on the fast path
    s[1, 8:16] = np.float32(0.0049)  # saturating for N(0,1)
    def gen():
        j = rng.integers(-130, 130, size=(N, H, D)).astype(np.float32)
        with np.errstate(over="ignore"):  # (j + 1/2) * 3e38 overflows to inf on purpose
            x = (j + 0.5) * s[None]
        x[:, :, 16:32] = rng.standard_normal((N, H, 16)).astype(np.float32) * 50
        x[:, 0, 8:12] = rng.standard_normal((N, 4)).astype(np.float32) * np.float32(1e30)
        return _f32_to_bits(x)
    w.k_scale = s
    w.v_scale = (s * np.float32(0.5)).astype(np.float32)
    check_full(_set_states(w, gen(), gen()))


def test_block_scales_extremes():
    """Per-block scales: exact ties against each token's block scale (s = 2^e,
    x = (j + 1/2) s), saturation, zero scales, and scales whose reciprocal leaves
    the normal range."""
    rng = np.random.default_rng(83)
    w = W.make_workload("block", q_lens=[50, 14, 30], ctx_before=[0, 3, 17], kv_heads=2,
                        head_dim=128, block_size=16, num_blocks=24, quant_mode=2, seed=83)
    N, H, D = w.num_tokens, w.kv_heads, w.head_dim
    NB = w.num_blocks
    s = np.exp2(rng.integers(-10, 4, size=(NB, H))).astype(np.float32)
    s[0::6, 0] = 0.0
    s[1::6, 1] = np.float32(1e-38)   # below 2^-120: exact path
    s[2::6, 0] = np.float32(3e38)    # above 2^120: exact path
    s[3::6, 1] = np.float32(1e-30)   # reciprocal 1e30: saturates on the fast path
    s[4::6, 0] = np.float32(0.0049)  # saturating for N(0,1) x 50
    # the block each new token lands in
    tok_blk = np.empty(N, np.int64)
    t = 0
    for b, q in enumerate(w.q_lens()):
        for i in range(int(q)):
            pos = int(w.context_kv_lens[b]) + i
            tok_blk[t] = w.block_table[b][pos // w.block_size]
            t += 1
    def gen(scale):
        j = rng.integers(-130, 130, size=(N, H, D)).astype(np.float64)
        x = (j + 0.5) * scale[tok_blk][:, :, None].astype(np.float64)
        x[:, :, 16:32] = rng.standard_normal((N, H, 16)) * 50
        return _f32_to_bits(np.clip(x, -1e38, 1e38))  # finite inputs only
    w.k_scale = s
    w.v_scale = (s * np.float32(0.5)).astype(np.float32)
    check_full(_set_states(w, gen(w.k_scale), gen(w.v_scale)))


def test_subnormal_scales_in_gather():
    """Mode-0 scale caches with subnormal and zero scales (prefilled, not
    stored): fp32 products that are subnormal must round to bf16 like the
    oracle's bit-level rounding."""
    w = W.make_workload("subn", q_lens=[0, 0], ctx_before=[40, 17], kv_heads=2, head_dim=64,
                        block_size=16, num_blocks=8, quant_mode=0, seed=83, with_store=False)
    rng = np.random.default_rng(83)
    sc = w.k_scale
    sc.reshape(-1)[::3] = np.float32(1e-40)
    sc.reshape(-1)[1::7] = np.float32(2.5e-39)
    sc.reshape(-1)[2::11] = 0.0
    w.v_scale.reshape(-1)[::2] = np.float32(np.finfo(np.float32).tiny)
    check_full(w)


# ---- device-side bounds reporting --------------------------------------------------

def test_store_reports_bad_block_and_skips_it():
    w = W.make_workload("badblk", q_lens=[5, 9, 4], ctx_before=[2, 0, 1], kv_heads=2,
                        head_dim=64, block_size=8, num_blocks=12, quant_mode=0, seed=90)
    w.block_table[2, 0] = w.num_blocks + 3  # the last sequence points outside the pool
    d = DeviceBatch(w)
    d.store()
    assert d.error_code() == kv.DEV_BAD_BLOCK_ID
    # expected: the oracle's store of the first two sequences only
    kc, vc, ks, vs = w.k_cache.copy(), w.v_cache.copy(), w.k_scale.copy(), w.v_scale.copy()
    n_ok = int(w.cu_q_lens[2])
    oracle.store(0, w.k_states[:n_ok], w.v_states[:n_ok], kc, vc, ks, vs, w.block_table[:2],
                 w.cu_q_lens[:3], w.context_kv_lens[:2])
    _assert_pool_equal(d.host_caches(), (kc, vc, ks, vs))


def test_store_reports_position_beyond_table():
    w = W.make_workload("beyond", q_lens=[3, 3], ctx_before=[0, 0], kv_heads=1, head_dim=16,
                        block_size=4, num_blocks=8, quant_mode=0, seed=91,
                        max_blocks_per_seq=2)
    w.context_kv_lens[1] = 6  # positions 6, 7 fit; 8 would need a third block
    d = DeviceBatch(w)
    d.store()
    assert d.error_code() == kv.DEV_POS_BEYOND_TABLE


def test_gather_reports_short_output_and_negative_length():
    w = W.make_workload("short", q_lens=[0, 0], ctx_before=[20, 30], kv_heads=2, head_dim=32,
                        block_size=8, num_blocks=16, quant_mode=1, seed=92, with_store=False)
    d = DeviceBatch(w, fill_out=0xFFFF)
    kv.kvc8_dequant_gather(d.g, d.k_cache, d.v_cache, d.k_scale, d.v_scale, d.block_table,
                           d.context_lengths, None, d.k_out, d.v_out, 25, d.k_out.stride(0),
                           d.k_out.stride(1), d.workspace, d.ws_bytes, d.dev_error)
    assert d.error_code(reset=True) == kv.DEV_OUT_ROW_RANGE
    # the first sequence (rows 0..19) is complete and exact
    ko = np.full((50, 2, 32), 0xFFFF, np.uint16)
    vo = ko.copy()
    oracle.dequant_gather(1, w.k_cache, w.v_cache, w.k_scale, w.v_scale, w.block_table[:1],
                          w.context_lengths[:1], None, ko, vo)
    gk, gv = d.host_outputs()
    _assert_bits_equal(gk[:20], ko[:20], "k_out")
    d.context_lengths[1] = -4
    d.gather()
    assert d.error_code(reset=True) == kv.DEV_BAD_LENGTH


# ---- full-size workloads, in the launch configuration the benchmark times -----------

def _check_full_size(w):
    """Store + gather of a full-size batch: the whole pool after the store and
    every output element after the gather, bit for bit against the oracle
    (its gather runs at about 2 GB/s on one core, a few seconds even for the
    6.5 GB long-context batch)."""
    d = DeviceBatch(w, fill_out=0xFFFF)
    d.store()
    d.gather()
    assert d.error_code() == 0
    # store: the whole pool after the oracle's store (in place on the host arrays)
    if w.has_store:
        oracle.store(w.quant_mode, w.k_states, w.v_states, w.k_cache, w.v_cache, w.k_scale,
                     w.v_scale, w.block_table, w.cu_q_lens, w.context_kv_lens)
    _assert_pool_equal(d.host_caches(), (w.k_cache, w.v_cache, w.k_scale, w.v_scale))
    # gather: every output row and element (the output was filled with the
    # bf16 NaN 0xFFFF, which no dequantised value can be)
    ko, vo = oracle.dequant_gather(w.quant_mode, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                                   w.block_table, w.context_lengths)
    gk, gv = d.host_outputs()
    _assert_bits_equal(gk, ko, "k_out")
    del gk, ko
    _assert_bits_equal(gv, vo, "v_out")
    return d


def test_full_prefill():
    _check_full_size(W.prefill())


@pytest.mark.parametrize("null_cu", [False, True])
def test_full_decode(null_cu):
    _check_full_size(W.decode(decode_null_cu=null_cu))


def test_full_mixed():
    _check_full_size(W.mixed())


def test_full_longctx():
    _check_full_size(W.longctx())


def test_full_prefill_block():
    _check_full_size(W.prefill_block())
