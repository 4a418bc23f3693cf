"""Seeded synthetic inputs for the int8 paged KV-cache store and dequant-gather.

This module only draws inputs.  It holds none of the store's or the gather's
arithmetic, and both the CUDA library's tests and the CPU oracle's tests take
their inputs from it (the oracle never imports it; the tests hand the same
arrays to both sides).

Every array is drawn on the host with numpy PCG64 streams seeded from
(seed, stream id, chunk id), so the values are the same on any machine and
for any thread count.  bf16 values are drawn as fp32 and rounded to bf16 by
torch's CPU conversion (round to nearest even).

Named workloads (the shapes of the paged-cache workloads in the method's
description, all synthetic):

* ``tiny``      batch 2, new-token counts {5, 19} stored after {3, 0} cached
                tokens, 2 kv heads, head_dim 64, block 16, 8-block pool,
                dynamic per-token scales; K/V ~ N(0, 1).
* ``prefill``   batch 16, prompts U{512..4096} into an empty cache, 8 kv
                heads, head_dim 128, block 128, 1024-block pool; N(0, 1) with
                4 outlier channels per head (fixed over tokens, drawn
                separately for K and V) multiplied by 20 before bf16 rounding;
                dynamic scales.
* ``decode``    batch 256, one new token each, cached context U{1..8192},
                8 x 128, block 128, 18000-block pool; dynamic scales.
* ``mixed``     64 sequences, exactly 32 decode (1 token) and 32 chunks of
                U{256..2048} tokens (seeded assignment), cached context
                U{0..16384}, 8 x 128, block 64, 20480-block pool; static
                per-(head, channel) scales U[0.005, 0.05].
* ``longctx``   8 x 131072 cached tokens, 8 x 128, block 128, 8192-block
                pool, gather only; codes uniform on [-127, 127], dynamic
                scales U[0.01, 0.1].

Before a store, the whole pool holds seeded codes uniform on [-127, 127] and
(dynamic mode) scales U[0.01, 0.1], so cached context and untouched slots are
defined.  Block tables are seeded permutations of the pool, one row per
sequence, so no block is shared between sequences.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np
import torch

_CHUNK = 1 << 25  # elements per independently seeded chunk

# stream ids, so that each array of a workload draws from its own stream
_S_META, _S_K, _S_V, _S_KC, _S_VC, _S_KS, _S_VS, _S_OUT = range(8)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _chunked(n: int, dtype, seed: int, stream: int, draw) -> np.ndarray:
    """Fill an array of n elements chunk by chunk; chunk c draws from the PCG64
    stream seeded by (seed, stream, c), so the result is thread-count free."""
    out = np.empty(n, dtype)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def work(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        rng = np.random.default_rng([seed, stream, c])
        out[lo:hi] = draw(rng, hi - lo)

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def _draw_codes(rng, m):
    # raw bytes are uniform on [-128, 127]; the byte -128 is redrawn uniformly
    # on [-127, 127], which leaves every code exactly uniform on [-127, 127].
    raw = rng.bit_generator.random_raw((m + 7) // 8).view(np.int8)[:m].copy()
    idx = np.flatnonzero(raw == -128)
    raw[idx] = rng.integers(-127, 128, size=idx.size, dtype=np.int8)
    return raw


def random_codes(n: int, seed: int, stream: int) -> np.ndarray:
    return _chunked(n, np.int8, seed, stream, _draw_codes)


def random_uniform_f32(n: int, lo: float, hi: float, seed: int, stream: int) -> np.ndarray:
    return _chunked(n, np.float32, seed, stream,
                    lambda rng, m: rng.uniform(lo, hi, size=m).astype(np.float32))


def random_normal_f32(n: int, seed: int, stream: int) -> np.ndarray:
    return _chunked(n, np.float32, seed, stream,
                    lambda rng, m: rng.standard_normal(m, dtype=np.float32))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (torch CPU conversion, nearest even); returns uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Workload:
    """One store (+ gather) problem.  All arrays are host numpy arrays.

    k_states, v_states : uint16 (bf16 bits) [num_tokens][H][D]   (None: gather only)
    k_cache, v_cache   : int8 [NB][H][bs][D]      pool contents before the store
    k_scale, v_scale   : fp32 [NB][H][bs] (quant_mode 0) or [H][D] (quant_mode 1)
    block_table        : int32 [B][MB]
    cu_q_lens          : int32 [B + 1] or None (decode: one token per sequence)
    context_kv_lens    : int32 [B]   tokens cached before the store
    context_lengths    : int32 [B]   tokens cached after the store (gather lengths)
    """
    name: str
    quant_mode: int
    kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    block_table: np.ndarray
    context_kv_lens: np.ndarray
    context_lengths: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    k_scale: np.ndarray
    v_scale: np.ndarray
    cu_q_lens: Optional[np.ndarray] = None
    k_states: Optional[np.ndarray] = None
    v_states: Optional[np.ndarray] = None
    seed: int = 0

    @property
    def num_seqs(self) -> int:
        return int(self.block_table.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def num_tokens(self) -> int:
        return 0 if self.k_states is None else int(self.k_states.shape[0])

    @property
    def total_context(self) -> int:
        return int(self.context_lengths.astype(np.int64).sum())

    @property
    def has_store(self) -> bool:
        return self.k_states is not None

    def q_lens(self) -> np.ndarray:
        if self.cu_q_lens is None:
            return np.ones(self.num_seqs, np.int32)
        return np.diff(self.cu_q_lens).astype(np.int32)


def make_workload(name: str, *, q_lens, ctx_before, kv_heads: int, head_dim: int,
                  block_size: int, num_blocks: int, quant_mode: int, seed: int,
                  max_blocks_per_seq: Optional[int] = None, decode_null_cu: bool = False,
                  outlier_channels: int = 0, outlier_gain: float = 20.0,
                  static_scale_range=(0.005, 0.05), pool_scale_range=(0.01, 0.1),
                  block_scale_range=(0.01, 0.1),
                  gather_only: bool = False, with_store: bool = True) -> Workload:
    """General seeded workload.

    q_lens / ctx_before: per-sequence new-token counts and cached-token counts.
    decode_null_cu: pass cu_q_lens = None (every q_len must be 1).
    gather_only: no new tokens; the gather reads ctx_before tokens.
    """
    q_lens = np.asarray(q_lens, np.int64)
    ctx_before = np.asarray(ctx_before, np.int64)
    B = int(ctx_before.shape[0])
    if gather_only or not with_store:
        q_lens = np.zeros(B, np.int64)
    ctx_after = ctx_before + q_lens
    need = int(((ctx_after + block_size - 1) // block_size).max()) if B else 0
    MB = int(max_blocks_per_seq if max_blocks_per_seq is not None else max(need, 1))
    if need > MB:
        raise ValueError("max_blocks_per_seq too small for the contexts")
    if B * MB > num_blocks:
        raise ValueError("pool too small for one distinct row of blocks per sequence")
    meta = np.random.default_rng([seed, _S_META])
    perm = meta.permutation(num_blocks).astype(np.int32)
    block_table = np.ascontiguousarray(perm[:B * MB].reshape(B, MB))
    H, D = kv_heads, head_dim
    pool = num_blocks * H * block_size * D
    k_cache = random_codes(pool, seed, _S_KC).reshape(num_blocks, H, block_size, D)
    v_cache = random_codes(pool, seed, _S_VC).reshape(num_blocks, H, block_size, D)
    if quant_mode == 0:
        lo, hi = pool_scale_range
        n_sc = num_blocks * H * block_size
        k_scale = random_uniform_f32(n_sc, lo, hi, seed, _S_KS).reshape(num_blocks, H, block_size)
        v_scale = random_uniform_f32(n_sc, lo, hi, seed, _S_VS).reshape(num_blocks, H, block_size)
    elif quant_mode == 1:
        lo, hi = static_scale_range
        k_scale = random_uniform_f32(H * D, lo, hi, seed, _S_KS).reshape(H, D)
        v_scale = random_uniform_f32(H * D, lo, hi, seed, _S_VS).reshape(H, D)
    elif quant_mode == 2:
        lo, hi = block_scale_range
        k_scale = random_uniform_f32(num_blocks * H, lo, hi, seed, _S_KS).reshape(num_blocks, H)
        v_scale = random_uniform_f32(num_blocks * H, lo, hi, seed, _S_VS).reshape(num_blocks, H)
    else:
        raise ValueError("quant_mode must be 0, 1 or 2")
    k_states = v_states = cu = None
    if not gather_only and with_store:
        N = int(q_lens.sum())
        if decode_null_cu:
            if not np.all(q_lens == 1):
                raise ValueError("cu_q_lens = None needs one token per sequence")
        else:
            cu = np.zeros(B + 1, np.int32)
            cu[1:] = np.cumsum(q_lens)
        ks, vs = [], []
        for stream, sink in ((_S_K, ks), (_S_V, vs)):
            x = random_normal_f32(N * H * D, seed, stream).reshape(N, H, D)
            if outlier_channels:
                ch_rng = np.random.default_rng([seed, stream, 1 << 20])
                for h in range(H):
                    ch = ch_rng.choice(D, size=outlier_channels, replace=False)
                    x[:, h, ch] *= np.float32(outlier_gain)
            sink.append(f32_to_bf16_bits(x).reshape(N, H, D))
        k_states, v_states = ks[0], vs[0]
    return Workload(name=name, quant_mode=quant_mode, kv_heads=H, head_dim=D,
                    block_size=block_size, num_blocks=num_blocks, block_table=block_table,
                    context_kv_lens=ctx_before.astype(np.int32),
                    context_lengths=ctx_after.astype(np.int32),
                    k_cache=k_cache, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale,
                    cu_q_lens=cu, k_states=k_states, v_states=v_states, seed=seed)


# ---- the five named workloads ------------------------------------------------

def tiny(seed: int = 1000) -> Workload:
    return make_workload("tiny", q_lens=[5, 19], ctx_before=[3, 0], kv_heads=2, head_dim=64,
                         block_size=16, num_blocks=8, max_blocks_per_seq=4, quant_mode=0,
                         seed=seed)


def prefill(seed: int = 1001) -> Workload:
    rng = np.random.default_rng([seed, 99])
    q = rng.integers(512, 4096, size=16, endpoint=True)
    return make_workload("prefill", q_lens=q, ctx_before=np.zeros(16, np.int64), kv_heads=8,
                         head_dim=128, block_size=128, num_blocks=1024, max_blocks_per_seq=32,
                         quant_mode=0, seed=seed, outlier_channels=4)


def decode(seed: int = 1002, decode_null_cu: bool = False) -> Workload:
    rng = np.random.default_rng([seed, 99])
    ctx = rng.integers(1, 8192, size=256, endpoint=True)
    return make_workload("decode", q_lens=np.ones(256, np.int64), ctx_before=ctx, kv_heads=8,
                         head_dim=128, block_size=128, num_blocks=18000, max_blocks_per_seq=65,
                         quant_mode=0, seed=seed, decode_null_cu=decode_null_cu)


def mixed(seed: int = 1003) -> Workload:
    rng = np.random.default_rng([seed, 99])
    is_chunk = np.zeros(64, bool)
    is_chunk[rng.permutation(64)[:32]] = True
    q = np.where(is_chunk, rng.integers(256, 2048, size=64, endpoint=True), 1)
    ctx = rng.integers(0, 16384, size=64, endpoint=True)
    return make_workload("mixed", q_lens=q, ctx_before=ctx, kv_heads=8, head_dim=128,
                         block_size=64, num_blocks=20480, max_blocks_per_seq=288,
                         quant_mode=1, seed=seed)


def longctx(seed: int = 1004) -> Workload:
    return make_workload("longctx", q_lens=np.zeros(8, np.int64),
                         ctx_before=np.full(8, 131072, np.int64), kv_heads=8, head_dim=128,
                         block_size=128, num_blocks=8192, max_blocks_per_seq=1024,
                         quant_mode=0, seed=seed, gather_only=True)


def prefill_block(seed: int = 1005) -> Workload:
    """The prefill batch with one static scale per (block, kv head)."""
    rng = np.random.default_rng([seed, 99])
    q = rng.integers(512, 4096, size=16, endpoint=True)
    return make_workload("prefill_block", q_lens=q, ctx_before=np.zeros(16, np.int64),
                         kv_heads=8, head_dim=128, block_size=128, num_blocks=1024,
                         max_blocks_per_seq=32, quant_mode=2, seed=seed, outlier_channels=4)


def decode_small(seed: int = 1006) -> Workload:
    """The decode batch cut to 64 sequences (about 2 GB on the device): the
    size for detailed profiles of the decode kernels."""
    rng = np.random.default_rng([seed, 99])
    ctx = rng.integers(1, 8192, size=64, endpoint=True)
    return make_workload("decode_small", q_lens=np.ones(64, np.int64), ctx_before=ctx,
                         kv_heads=8, head_dim=128, block_size=128, num_blocks=64 * 65,
                         max_blocks_per_seq=65, quant_mode=0, seed=seed)


def mixed_small(seed: int = 1007) -> Workload:
    """The chunked-prefill mix with cached contexts cut to U[0, 1024] and a
    pool to match (about 1 GB on the device): the size for detailed profiles
    of the static-scale store."""
    rng = np.random.default_rng([seed, 99])
    is_chunk = np.zeros(64, bool)
    is_chunk[rng.permutation(64)[:32]] = True
    q = np.where(is_chunk, rng.integers(256, 2048, size=64, endpoint=True), 1)
    ctx = rng.integers(0, 1024, size=64, endpoint=True)
    return make_workload("mixed_small", q_lens=q, ctx_before=ctx, kv_heads=8, head_dim=128,
                         block_size=64, num_blocks=64 * 52, max_blocks_per_seq=52,
                         quant_mode=1, seed=seed)


NAMED = {"tiny": tiny, "prefill": prefill, "decode": decode, "mixed": mixed,
         "longctx": longctx, "prefill_block": prefill_block, "decode_small": decode_small,
         "mixed_small": mixed_small}


def algorithmic_bytes(w: Workload) -> dict:
    """Algorithmic HBM bytes of one store and one gather (K and V together).

    store : read the bf16 rows, write the int8 rows (+ one fp32 scale per row in
            quant_mode 0; the static table in quant_mode 1 is read once, 2*H*D*4).
    gather: read the int8 rows (+ one fp32 scale per row in quant_mode 0, or the
            static table once), write the bf16 rows.
    Index metadata (block table, lengths) is left out (< 0.1%).
    """
    H, D = w.kv_heads, w.head_dim
    rows_store = 2 * H * w.num_tokens
    rows_gather = 2 * H * w.total_context
    table = 2 * H * D * 4 if w.quant_mode == 1 else 0
    per_row_scale = 4 if w.quant_mode == 0 else 0
    store = rows_store * (2 * D + D + per_row_scale) + (table if w.num_tokens else 0)
    gather = rows_gather * (D + per_row_scale + 2 * D) + (table if w.total_context else 0)
    if w.quant_mode == 2:  # one 4-byte scale per (block, head) that the op touches
        store += 4 * 2 * H * _blocks_touched(w, new_only=True)
        gather += 4 * 2 * H * _blocks_touched(w, new_only=False)
    return {"store": int(store), "gather": int(gather)}


def _blocks_touched(w: Workload, new_only: bool) -> int:
    """Logical blocks that hold the new tokens (new_only) or any gathered
    position, summed over sequences."""
    bs = w.block_size
    end = w.context_lengths.astype(np.int64)
    start = w.context_kv_lens.astype(np.int64) if new_only else np.zeros_like(end)
    has = end > start
    first = start // bs
    last = (end - 1) // bs
    return int(np.where(has, last - first + 1, 0).sum())


def algorithmic_bytes_bf16(w: Workload) -> dict:
    """Algorithmic HBM bytes of one store and one gather of the bf16 cache (no
    quantisation): every row is read once and written once, 2*D bytes each way."""
    H, D = w.kv_heads, w.head_dim
    return {"store": int(2 * H * w.num_tokens * 4 * D),
            "gather": int(2 * H * w.total_context * 4 * D)}


def algorithmic_bytes_fused(w: Workload) -> dict:
    """Algorithmic HBM bytes of one fused append + gather (K and V together):
    the store's bytes for the new tokens, the gather's bytes for the cached
    positions, and the bf16 output rows of the new tokens (written once, never
    read back from the cache)."""
    H, D = w.kv_heads, w.head_dim
    table = 2 * H * D * 4 if w.quant_mode == 1 else 0
    per_row_scale = 4 if w.quant_mode == 0 else 0
    cached = 2 * H * int(w.context_kv_lens.astype(np.int64).sum())
    new = 2 * H * w.num_tokens
    total = new * (2 * D + D + per_row_scale + 2 * D) + cached * (D + per_row_scale + 2 * D)
    return {"store": 0, "gather": int(total + table)}


def algorithmic_bytes_attention(w: Workload, group: int) -> dict:
    """Algorithmic HBM bytes of one paged decode attention (int8 path): every
    cached K and V code of every gathered position once, their scales, the
    query read and the bf16 output written."""
    H, D = w.kv_heads, w.head_dim
    rows = 2 * H * w.total_context
    scales = (rows * 4 if w.quant_mode == 0 else 2 * H * D * 4 if w.quant_mode == 1
              else 4 * 2 * H * _blocks_touched(w, new_only=False))
    q_out = 2 * w.num_seqs * H * group * D * 2
    return {"store": 0, "gather": int(rows * D + scales + q_out)}
