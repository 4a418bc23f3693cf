"""Device-resident buffers for one store + gather problem, and the calls that
run it through libkvc8.  Marshalling only: every step of the store and the
gather runs in the library's kernels; torch allocates the memory and supplies
the stream.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B
from .workloads import Workload


def _bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class DeviceBatch:
    """Holds a Workload on the GPU.

    out_layout: "dense" -> outputs [rows][H][D];
                "head_major" -> outputs stored [H][rows][D] and viewed as
                [rows][H][D] (a transposed, strided view, as the pages' tests
                pass with context_strided);
    out_pad_rows: extra output rows after the last sequence (not written).
    offsets: optional int64 [B] caller-given context_seq_offset.
    """

    def __init__(self, w: Workload, device="cuda", out_layout="dense", out_pad_rows=0,
                 offsets=None, fill_out=None, pin=False):
        self.w = w
        self.device = torch.device(device)
        dev = self.device
        self.g = B.Geom(w.num_seqs, w.kv_heads, w.head_dim, w.block_size, w.num_blocks,
                        w.max_blocks_per_seq, w.quant_mode)
        H, D = w.kv_heads, w.head_dim
        to = (lambda t: t.pin_memory()) if pin else (lambda t: t)
        self.k_states = self.v_states = None
        if w.has_store:
            self.k_states = _bf16(w.k_states).to(dev)
            self.v_states = _bf16(w.v_states).to(dev)
        self.k_cache = torch.from_numpy(w.k_cache).to(dev)
        self.v_cache = torch.from_numpy(w.v_cache).to(dev)
        self.k_scale = torch.from_numpy(w.k_scale).to(dev)
        self.v_scale = torch.from_numpy(w.v_scale).to(dev)
        self.block_table = torch.from_numpy(w.block_table).to(dev)
        self.cu_q_lens = None if w.cu_q_lens is None else torch.from_numpy(w.cu_q_lens).to(dev)
        self.context_kv_lens = torch.from_numpy(w.context_kv_lens).to(dev)
        self.context_lengths = torch.from_numpy(w.context_lengths).to(dev)
        self.offsets = None
        if offsets is not None:
            self.offsets = torch.from_numpy(np.asarray(offsets, np.int64)).to(dev)
            rows = int(max(int(o) + int(l) for o, l in zip(offsets, w.context_lengths))) if w.num_seqs else 0
        else:
            rows = w.total_context
        self.out_rows = rows + out_pad_rows
        if out_layout == "dense":
            self.k_out = torch.empty((self.out_rows, H, D), dtype=torch.bfloat16, device=dev)
            self.v_out = torch.empty((self.out_rows, H, D), dtype=torch.bfloat16, device=dev)
        elif out_layout == "head_major":
            self.k_out = torch.empty((H, self.out_rows, D), dtype=torch.bfloat16,
                                     device=dev).transpose(0, 1)
            self.v_out = torch.empty((H, self.out_rows, D), dtype=torch.bfloat16,
                                     device=dev).transpose(0, 1)
        else:
            raise ValueError(out_layout)
        if fill_out is not None:
            self.k_out.view(torch.int16).fill_(np.int16(np.uint16(fill_out).view(np.int16)))
            self.v_out.view(torch.int16).fill_(np.int16(np.uint16(fill_out).view(np.int16)))
        self.ws_bytes = B.kvc8_gather_workspace_bytes(self.g)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.dev_error = torch.zeros(1, dtype=torch.int32, device=dev)
        del to

    # ---- the calls ------------------------------------------------------------

    def store(self, stream=None):
        if self.k_states is None:
            return
        ks = self.k_states
        B.kvc8_store(self.g, ks.shape[0], ks, self.v_states, ks.stride(0), ks.stride(1),
                     self.k_cache, self.v_cache, self.k_scale, self.v_scale, self.block_table,
                     self.cu_q_lens, self.context_kv_lens, self.dev_error, stream)

    def gather(self, stream=None):
        ko = self.k_out
        B.kvc8_dequant_gather(self.g, self.k_cache, self.v_cache, self.k_scale, self.v_scale,
                              self.block_table, self.context_lengths, self.offsets, ko,
                              self.v_out, self.out_rows, ko.stride(0), ko.stride(1),
                              self.workspace, self.ws_bytes, self.dev_error, stream)

    def build_metadata(self, offsets_out=None, stream=None):
        B.kvc8_build_metadata(self.g, self.context_lengths, self.offsets, offsets_out,
                              self.workspace, self.ws_bytes, self.dev_error, stream)

    def gather_planned(self, stream=None):
        ko = self.k_out
        B.kvc8_dequant_gather_planned(self.g, self.k_cache, self.v_cache, self.k_scale,
                                      self.v_scale, self.block_table, self.context_lengths, ko,
                                      self.v_out, self.out_rows, ko.stride(0), ko.stride(1),
                                      self.workspace, self.ws_bytes, self.dev_error, stream)

    def _append_operands(self):
        ks = self.k_states
        if ks is None:  # nothing to append: every sequence gets zero new tokens
            if getattr(self, "_zero_cu", None) is None:
                self._zero_cu = torch.zeros(self.w.num_seqs + 1, dtype=torch.int32,
                                            device=self.device)
            return 0, None, None, 0, 0, self._zero_cu
        return ks.shape[0], ks, self.v_states, ks.stride(0), ks.stride(1), self.cu_q_lens

    def append_gather(self, stream=None):
        """The store and the gather of the whole context in one pass (plan +
        one fused launch)."""
        n, ks, vs, ts, hs, cu = self._append_operands()
        ko = self.k_out
        B.kvc8_append_gather(self.g, n, ks, vs, ts, hs, self.k_cache, self.v_cache, self.k_scale,
                             self.v_scale, self.block_table, cu, self.context_kv_lens,
                             self.offsets, ko, self.v_out, self.out_rows, ko.stride(0),
                             ko.stride(1), self.workspace, self.ws_bytes, self.dev_error, stream)

    def build_append_metadata(self, offsets_out=None, stream=None):
        _, _, _, _, _, cu = self._append_operands()
        B.kvc8_build_append_metadata(self.g, cu, self.context_kv_lens, self.offsets, offsets_out,
                                     self.workspace, self.ws_bytes, self.dev_error, stream)

    def append_gather_planned(self, stream=None):
        n, ks, vs, ts, hs, cu = self._append_operands()
        ko = self.k_out
        B.kvc8_append_gather_planned(self.g, n, ks, vs, ts, hs, self.k_cache, self.v_cache,
                                     self.k_scale, self.v_scale, self.block_table, cu,
                                     self.context_kv_lens, ko, self.v_out, self.out_rows,
                                     ko.stride(0), ko.stride(1), self.workspace, self.ws_bytes,
                                     self.dev_error, stream)

    def error_code(self, reset=False) -> int:
        return B.kvc8_get_error(self.dev_error, reset=reset)

    # ---- host copies ------------------------------------------------------------

    def host_caches(self):
        return (self.k_cache.cpu().numpy(), self.v_cache.cpu().numpy(),
                self.k_scale.cpu().numpy(), self.v_scale.cpu().numpy())

    def host_outputs(self):
        return bf16_bits(self.k_out), bf16_bits(self.v_out)


class Bf16Batch:
    """Holds a Workload's tokens, metadata and a bf16 page pool [NB][H][bs][D]
    (no quantisation) on the GPU, for kvc8_store_bf16 / kvc8_gather_bf16.  The
    pool starts as seeded random bits; outputs are dense [rows][H][D]."""

    def __init__(self, w: Workload, device="cuda", seed=0):
        self.w = w
        dev = self.device = torch.device(device)
        self.g = B.Geom(w.num_seqs, w.kv_heads, w.head_dim, w.block_size, w.num_blocks,
                        w.max_blocks_per_seq, 0)
        H, D = w.kv_heads, w.head_dim
        self.k_states = self.v_states = None
        if w.has_store:
            self.k_states = _bf16(w.k_states).to(dev)
            self.v_states = _bf16(w.v_states).to(dev)
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed)
        shape = (w.num_blocks, H, w.block_size, D)
        self.k_cache = torch.randint(-32768, 32768, shape, dtype=torch.int16, device=dev,
                                     generator=gen).view(torch.bfloat16)
        self.v_cache = torch.randint(-32768, 32768, shape, dtype=torch.int16, device=dev,
                                     generator=gen).view(torch.bfloat16)
        self.block_table = torch.from_numpy(w.block_table).to(dev)
        self.cu_q_lens = None if w.cu_q_lens is None else torch.from_numpy(w.cu_q_lens).to(dev)
        self.context_kv_lens = torch.from_numpy(w.context_kv_lens).to(dev)
        self.context_lengths = torch.from_numpy(w.context_lengths).to(dev)
        self.out_rows = w.total_context
        self.k_out = torch.empty((self.out_rows, H, D), dtype=torch.bfloat16, device=dev)
        self.v_out = torch.empty((self.out_rows, H, D), dtype=torch.bfloat16, device=dev)
        self.ws_bytes = B.kvc8_gather_workspace_bytes(self.g)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.dev_error = torch.zeros(1, dtype=torch.int32, device=dev)

    def store(self, stream=None):
        if self.k_states is None:
            return
        ks = self.k_states
        B.kvc8_store_bf16(self.g, ks.shape[0], ks, self.v_states, ks.stride(0), ks.stride(1),
                          self.k_cache, self.v_cache, self.block_table, self.cu_q_lens,
                          self.context_kv_lens, self.dev_error, stream)

    def gather(self, stream=None):
        ko = self.k_out
        B.kvc8_gather_bf16(self.g, self.k_cache, self.v_cache, self.block_table,
                           self.context_lengths, None, ko, self.v_out, self.out_rows,
                           ko.stride(0), ko.stride(1), self.workspace, self.ws_bytes,
                           self.dev_error, stream)

    def error_code(self, reset=False) -> int:
        return B.kvc8_get_error(self.dev_error, reset=reset)


class DecodeAttention:
    """One decode query per sequence (num_q_heads = group * kv_heads, seeded
    N(0, 1) bf16) attending over a DeviceBatch's int8 cache through
    kvc8_paged_decode_attention; output bf16 [B][num_q_heads][D]."""

    def __init__(self, d: DeviceBatch, group: int, seed: int = 0, softmax_scale=None):
        self.d = d
        w = d.w
        self.num_q_heads = w.kv_heads * group
        rng = np.random.default_rng([seed, 77])
        x = rng.standard_normal((w.num_seqs, self.num_q_heads, w.head_dim)).astype(np.float32)
        self.q_bits = (x.view(np.uint32) >> 16).astype(np.uint16)
        self.query = _bf16(self.q_bits).to(d.device)
        self.out = torch.empty_like(self.query)
        self.scale = float(softmax_scale if softmax_scale is not None else w.head_dim ** -0.5)
        self.ws_bytes = B.kvc8_attention_workspace_bytes(d.g, self.num_q_heads)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=d.device)

    def __call__(self, stream=None):
        d, q, o = self.d, self.query, self.out
        B.kvc8_paged_decode_attention(d.g, self.num_q_heads, q, q.stride(0), q.stride(1),
                                      d.k_cache, d.v_cache, d.k_scale, d.v_scale,
                                      d.block_table, d.context_lengths, self.scale, o,
                                      o.stride(0), o.stride(1), self.workspace, self.ws_bytes,
                                      d.dev_error, stream)
