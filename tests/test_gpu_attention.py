"""Paged decode attention over the int8 cache (kvc8_paged_decode_attention)
against the oracle.

The oracle computes the exact attention of the bf16 query over the bf16 rows
the dequant-gather produces, in fp64.  The kernel multiplies bf16 operands on
the tensor cores with fp32 accumulation, rounds the softmax weights to bf16
(and normalises by the sum of the rounded weights) and rounds the output to
bf16.  So each output is a weighted average of the V' rows whose weights are
off by a relative 2^-8 at most (bf16 rounding 2^-9, exp2 approximation and
fp32 score error well below that); such an average moves by at most
2 * 2^-8 * max_p |V'[p][d]|, and the output rounding adds 2^-9 |out|.  The
tolerance per element is therefore 2^-7 * max_p |V'[p][d]| + 2^-8 |out|.
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


def _query(rng, B, HQ, D):
    x = rng.standard_normal((B, HQ, D)).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)  # bf16 bits (truncated)


def _bf16_to_f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def run_attention(w, group, scale, rng, q_layout="dense", out_layout="dense", d=None):
    d = d or DeviceBatch(w)
    H, D, B = w.kv_heads, w.head_dim, w.num_seqs
    HQ = H * group
    qb = _query(rng, B, HQ, D)
    qt = torch.from_numpy(qb.view(np.int16))
    if q_layout == "head_major":  # [HQ][B][D] storage viewed as [B][HQ][D]
        q = qt.transpose(0, 1).contiguous().cuda().transpose(0, 1)
    else:
        q = qt.cuda()
    if out_layout == "head_major":
        out = torch.full((HQ, B, D), -1, dtype=torch.int16, device="cuda").transpose(0, 1)
    else:
        out = torch.full((B, HQ, D), -1, dtype=torch.int16, device="cuda")
    ws_bytes = kv.kvc8_attention_workspace_bytes(d.g, HQ)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    kv.kvc8_paged_decode_attention(d.g, HQ, q, q.stride(0), q.stride(1), d.k_cache, d.v_cache,
                                   d.k_scale, d.v_scale, d.block_table, d.context_lengths, scale,
                                   out, out.stride(0), out.stride(1), ws, ws_bytes, d.dev_error)
    return qb, out.contiguous().cpu().numpy().view(np.uint16), d


def check_attention(w, group, scale, qb, got, seqs=None):
    """Compare the bf16 output with the fp64 oracle on sequences `seqs`."""
    seqs = np.arange(w.num_seqs) if seqs is None else np.asarray(seqs)
    H, D = w.kv_heads, w.head_dim
    bt = w.block_table[seqs]
    lens = w.context_lengths[seqs]
    want = oracle.paged_decode_attention(w.quant_mode, qb[seqs], w.k_cache, w.v_cache, w.k_scale,
                                         w.v_scale, bt, lens, scale)
    got_f = _bf16_to_f32(got[seqs]).astype(np.float64)
    # max_p |V'[p][d]| per (sequence, kv head, channel), from the oracle's gather
    _, vo = oracle.dequant_gather(w.quant_mode, w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                                  bt, lens)
    vf = np.abs(_bf16_to_f32(vo).astype(np.float64))
    off = np.concatenate([[0], np.cumsum(lens.astype(np.int64))])
    for i in range(len(seqs)):
        if lens[i] == 0:
            assert not got_f[i].any(), "empty context must give zeros"
            continue
        vmax = np.repeat(vf[off[i]:off[i + 1]].max(axis=0), group, axis=0)  # [HQ][D]
        tol = 2.0 ** -7 * vmax + 2.0 ** -8 * np.abs(want[i]) + 1e-30
        err = np.abs(got_f[i] - want[i])
        bad = np.argwhere(err > tol)
        assert len(bad) == 0, (f"sequence {seqs[i]}: {len(bad)} outputs beyond tolerance, first "
                               f"{bad[:3].tolist()}: got {got_f[i][tuple(bad[0])]}, want "
                               f"{want[i][tuple(bad[0])]}, tol {tol[tuple(bad[0])]}")


CASES = [
    # lens cross 16-position pieces, blocks and the 2048-position splits
    dict(lens=[0, 1, 15, 16, 300], H=2, G=4, D=128, bs=16, mode=0),
    dict(lens=[3000, 1, 1024, 1025, 2048], H=4, G=8, D=64, bs=32, mode=0),
    dict(lens=[77, 513, 1], H=2, G=1, D=128, bs=64, mode=1),
    dict(lens=[129, 2100, 64], H=3, G=3, D=128, bs=128, mode=2),
    dict(lens=[1000, 31, 4097], H=8, G=2, D=64, bs=16, mode=1),
    dict(lens=[5, 2500], H=1, G=8, D=128, bs=256, mode=2),
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_attention_small(i):
    c = CASES[i]
    lens = np.asarray(c["lens"], np.int64)
    mb = int(((lens + c["bs"] - 1) // c["bs"]).max()) or 1
    w = W.make_workload(f"att{i}", q_lens=np.zeros(len(lens), np.int64), ctx_before=lens,
                        kv_heads=c["H"], head_dim=c["D"], block_size=c["bs"],
                        num_blocks=len(lens) * mb + 3, quant_mode=c["mode"], seed=300 + i,
                        with_store=False)
    rng = np.random.default_rng(400 + i)
    scale = 1.0 / np.sqrt(c["D"])
    qb, got, d = run_attention(w, c["G"], scale, rng)
    assert d.error_code() == 0
    check_attention(w, c["G"], scale, qb, got)


def _random_case(i):
    """Seeded problem i: head_dim 64 or 128, block sizes 16 to 256, 1-8 kv
    heads with groups of 1-8 query heads, all scale modes, 1-24 sequences
    whose lengths run from 0 past several 2048-position splits."""
    rng = np.random.default_rng([5150, i])
    top = int(rng.choice([40, 600, 9000]))
    return dict(lens=rng.integers(0, top, size=int(rng.integers(1, 25))),
                H=int(rng.integers(1, 9)), G=int(rng.integers(1, 9)),
                D=int(rng.choice([64, 128])), bs=int(rng.choice([16, 32, 48, 64, 128, 256])),
                mode=int(rng.integers(0, 3)))


@pytest.mark.parametrize("i", range(24))
def test_attention_random(i):
    c = _random_case(i)
    lens = np.asarray(c["lens"], np.int64)
    mb = int(((lens + c["bs"] - 1) // c["bs"]).max()) or 1
    w = W.make_workload(f"attr{i}", q_lens=np.zeros(len(lens), np.int64), ctx_before=lens,
                        kv_heads=c["H"], head_dim=c["D"], block_size=c["bs"],
                        num_blocks=len(lens) * mb + 3, quant_mode=c["mode"], seed=900 + i,
                        with_store=False)
    rng = np.random.default_rng(950 + i)
    scale = 1.0 / np.sqrt(c["D"])
    qb, got, d = run_attention(w, c["G"], scale, rng)
    assert d.error_code() == 0
    check_attention(w, c["G"], scale, qb, got)


def test_attention_strided_and_peaked():
    w = W.make_workload("attstr", q_lens=np.zeros(3, np.int64), ctx_before=[700, 2, 1500],
                        kv_heads=4, head_dim=128, block_size=64, num_blocks=80, quant_mode=0,
                        seed=310, with_store=False)
    rng = np.random.default_rng(410)
    for scale in (0.088, 3.0):  # 3.0: one position carries nearly all the weight
        qb, got, d = run_attention(w, 4, scale, rng, q_layout="head_major",
                                   out_layout="head_major")
        assert d.error_code() == 0
        check_attention(w, 4, scale, qb, got)


def test_attention_after_store():
    """Attention over a cache the store has just written (the decode step's order)."""
    w = W.make_workload("attstore", q_lens=[1, 1, 1, 1], ctx_before=[0, 17, 1023, 2000],
                        kv_heads=8, head_dim=128, block_size=16, num_blocks=4 * 130,
                        quant_mode=0, seed=311, decode_null_cu=True)
    d = DeviceBatch(w)
    d.store()
    oracle.store(w.quant_mode, w.k_states, w.v_states, w.k_cache, w.v_cache, w.k_scale,
                 w.v_scale, w.block_table, w.cu_q_lens, w.context_kv_lens)
    rng = np.random.default_rng(411)
    qb, got, d = run_attention(w, 4, 0.088, rng, d=d)
    assert d.error_code() == 0
    check_attention(w, 4, 0.088, qb, got)


def test_attention_reports_bad_block():
    w = W.make_workload("attbad", q_lens=np.zeros(2, np.int64), ctx_before=[40, 40],
                        kv_heads=2, head_dim=64, block_size=16, num_blocks=8, quant_mode=0,
                        seed=312, with_store=False)
    w.block_table = w.block_table.copy()
    w.block_table[1, 1] = 1000
    rng = np.random.default_rng(412)
    qb, got, d = run_attention(w, 2, 0.125, rng)
    assert d.error_code(reset=True) == kv.DEV_BAD_BLOCK_ID
    check_attention(w, 2, 0.125, qb, got, seqs=[0])  # the other sequence is intact


def test_attention_full_size_decode():
    """The decode batch (256 sequences, contexts up to 8192, 32 query heads on
    8 kv heads) at full size, every sequence and output element checked
    against the oracle."""
    w = W.decode()
    oracle.store(w.quant_mode, w.k_states, w.v_states, w.k_cache, w.v_cache, w.k_scale,
                 w.v_scale, w.block_table, w.cu_q_lens, w.context_kv_lens)
    d = DeviceBatch(w)  # the pool after the store
    rng = np.random.default_rng(413)
    qb, got, d = run_attention(w, 4, 1.0 / np.sqrt(128), rng, d=d)
    assert d.error_code() == 0
    check_attention(w, 4, 1.0 / np.sqrt(128), qb, got)
    assert not np.any(got == 0xFFFF)
