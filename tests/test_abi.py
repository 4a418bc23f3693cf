"""The C ABI library on the CPU: it builds, loads, exports every function the
header declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes

import pytest

import dequant_kvc8_store_gb300 as kv
from dequant_kvc8_store_gb300 import binding as B


@pytest.fixture(scope="module")
def lib():
    return kv.load()


def test_every_declared_function_is_exported(lib):
    names = B.declared_functions()
    assert {"kvc8_store", "kvc8_dequant_gather", "kvc8_build_metadata",
            "kvc8_dequant_gather_planned", "kvc8_gather_workspace_bytes",
            "kvc8_get_error", "kvc8_status_str", "kvc8_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in kvc8.h but not exported"


def test_status_strings_and_version(lib):
    assert kv.kvc8_status_str(kv.OK) == "ok"
    assert "argument" in kv.kvc8_status_str(kv.ERR_INVALID_ARG)
    assert "workspace" in kv.kvc8_status_str(kv.ERR_WORKSPACE)
    assert kv.kvc8_status_str(99) == "unknown status"
    assert kv.kvc8_version() >= 10000


def test_workspace_bytes_grows_with_batch():
    g = kv.Geom(1, 8, 128, 128, 1024, 32, 0)
    a = kv.kvc8_gather_workspace_bytes(g)
    g.num_seqs = 100000
    b = kv.kvc8_gather_workspace_bytes(g)
    assert a >= 256 and a % 256 == 0 and b % 256 == 0
    assert b >= 100000 * 8 + 100001 * 4


FAKE = 1 << 20  # an aligned, never-dereferenced address: checks fail before any launch


def _store(g, n=4, **kw):
    args = dict(key_states=FAKE, value_states=FAKE, x_tok_stride=g.kv_heads * g.head_dim,
                x_head_stride=g.head_dim, key_cache=FAKE, value_cache=FAKE, key_scale=FAKE,
                value_scale=FAKE, block_table=FAKE, cu_q_lens=FAKE, context_kv_lens=FAKE)
    args.update(kw)
    return kv.load().kvc8_store(ctypes.byref(g), n, args["key_states"], args["value_states"],
                                args["x_tok_stride"], args["x_head_stride"], args["key_cache"],
                                args["value_cache"], args["key_scale"], args["value_scale"],
                                args["block_table"], args["cu_q_lens"], args["context_kv_lens"],
                                None, None)


def test_store_rejects_bad_geometry():
    ok = dict(num_seqs=2, kv_heads=8, head_dim=128, block_size=16, num_blocks=64,
              max_blocks_per_seq=8, quant_mode=0)
    for field, bad, want in [("head_dim", 24, kv.ERR_INVALID_ARG), ("head_dim", 8, kv.ERR_INVALID_ARG),
                             ("head_dim", 512, kv.ERR_UNSUPPORTED),
                             ("quant_mode", 3, kv.ERR_INVALID_ARG),
                             ("kv_heads", 0, kv.ERR_INVALID_ARG),
                             ("block_size", 0, kv.ERR_INVALID_ARG),
                             ("num_blocks", 0, kv.ERR_INVALID_ARG),
                             ("max_blocks_per_seq", 0, kv.ERR_INVALID_ARG),
                             ("num_seqs", -1, kv.ERR_INVALID_ARG)]:
        g = kv.Geom(**{**ok, field: bad})
        assert _store(g) == want, (field, bad)
    assert kv.load().kvc8_store(None, 1, *([FAKE] * 2), 8, 8, *([FAKE] * 7), None, None) == \
        kv.ERR_INVALID_ARG


def test_store_rejects_bad_pointers_and_strides():
    g = kv.Geom(2, 8, 128, 16, 64, 8, 0)
    for name in ("key_states", "value_states", "key_cache", "value_cache", "key_scale",
                 "value_scale", "block_table", "context_kv_lens"):
        assert _store(g, **{name: None}) == kv.ERR_INVALID_ARG, name
    assert _store(g, x_tok_stride=1028) == kv.ERR_INVALID_ARG
    assert _store(g, x_head_stride=-128) == kv.ERR_INVALID_ARG
    assert _store(g, key_states=FAKE + 2) == kv.ERR_INVALID_ARG
    assert _store(g, key_scale=FAKE + 4) == kv.ERR_INVALID_ARG
    # decode form (cu_q_lens NULL) needs one token per sequence
    assert _store(g, n=3, cu_q_lens=None) == kv.ERR_INVALID_ARG
    assert _store(g, n=-1) == kv.ERR_INVALID_ARG
    # nothing to store is a no-op, whatever the pointers
    assert _store(g, n=0, key_states=None) == kv.OK


def _gather(g, fn="kvc8_dequant_gather", **kw):
    a = dict(kc=FAKE, vc=FAKE, ks=FAKE, vs=FAKE, bt=FAKE, lens=FAKE, off=None, ko=FAKE, vo=FAKE,
             rows=10, ts=g.kv_heads * g.head_dim, hs=g.head_dim, ws=FAKE, wsb=1 << 20)
    a.update(kw)
    lib = kv.load()
    if fn == "kvc8_dequant_gather":
        return lib.kvc8_dequant_gather(ctypes.byref(g), a["kc"], a["vc"], a["ks"], a["vs"],
                                       a["bt"], a["lens"], a["off"], a["ko"], a["vo"], a["rows"],
                                       a["ts"], a["hs"], a["ws"], a["wsb"], None, None)
    return lib.kvc8_dequant_gather_planned(ctypes.byref(g), a["kc"], a["vc"], a["ks"], a["vs"],
                                           a["bt"], a["lens"], a["ko"], a["vo"], a["rows"],
                                           a["ts"], a["hs"], a["ws"], a["wsb"], None, None)


@pytest.mark.parametrize("fn", ["kvc8_dequant_gather", "kvc8_dequant_gather_planned"])
def test_gather_rejects_bad_arguments(fn):
    g = kv.Geom(2, 8, 128, 16, 64, 8, 0)
    for name in ("kc", "vc", "ks", "vs", "bt", "lens", "ko", "vo"):
        assert _gather(g, fn, **{name: None}) == kv.ERR_INVALID_ARG, name
    assert _gather(g, fn, rows=-1) == kv.ERR_INVALID_ARG
    assert _gather(g, fn, ts=1020) == kv.ERR_INVALID_ARG
    assert _gather(g, fn, hs=4) == kv.ERR_INVALID_ARG
    assert _gather(g, fn, ko=FAKE + 8) == kv.ERR_INVALID_ARG
    assert _gather(g, fn, ws=None) == kv.ERR_WORKSPACE
    assert _gather(g, fn, ws=FAKE + 16) == kv.ERR_WORKSPACE
    assert _gather(g, fn, wsb=16) == kv.ERR_WORKSPACE
    g0 = kv.Geom(0, 8, 128, 16, 64, 8, 0)
    assert _gather(g0, fn, kc=None) == kv.OK  # empty batch: no-op


def test_build_metadata_rejects_bad_arguments():
    g = kv.Geom(2, 8, 128, 16, 64, 8, 0)
    lib = kv.load()
    assert lib.kvc8_build_metadata(ctypes.byref(g), None, None, None, FAKE, 1 << 20, None,
                                   None) == kv.ERR_INVALID_ARG
    assert lib.kvc8_build_metadata(ctypes.byref(g), FAKE, None, None, FAKE, 8, None,
                                   None) == kv.ERR_WORKSPACE


def test_get_error_rejects_null():
    code = ctypes.c_int32()
    assert kv.load().kvc8_get_error(None, ctypes.byref(code), 0, None) == kv.ERR_INVALID_ARG


def _store_bf16(g, n=4, **kw):
    a = dict(ks=FAKE, vs=FAKE, ts=g.kv_heads * g.head_dim, hs=g.head_dim, kc=FAKE, vc=FAKE,
             bt=FAKE, cu=FAKE, ctx=FAKE)
    a.update(kw)
    return kv.load().kvc8_store_bf16(ctypes.byref(g), n, a["ks"], a["vs"], a["ts"], a["hs"],
                                     a["kc"], a["vc"], a["bt"], a["cu"], a["ctx"], None, None)


def _gather_bf16(g, **kw):
    a = dict(kc=FAKE, vc=FAKE, bt=FAKE, lens=FAKE, off=None, ko=FAKE, vo=FAKE, rows=10,
             ts=g.kv_heads * g.head_dim, hs=g.head_dim, ws=FAKE, wsb=1 << 20)
    a.update(kw)
    return kv.load().kvc8_gather_bf16(ctypes.byref(g), a["kc"], a["vc"], a["bt"], a["lens"],
                                      a["off"], a["ko"], a["vo"], a["rows"], a["ts"], a["hs"],
                                      a["ws"], a["wsb"], None, None)


def test_bf16_store_and_gather_reject_bad_arguments():
    g = kv.Geom(2, 8, 128, 16, 64, 8, 0)
    for name in ("ks", "vs", "kc", "vc", "bt", "ctx"):
        assert _store_bf16(g, **{name: None}) == kv.ERR_INVALID_ARG, name
    assert _store_bf16(g, ts=1028) == kv.ERR_INVALID_ARG
    assert _store_bf16(g, kc=FAKE + 2) == kv.ERR_INVALID_ARG
    assert _store_bf16(g, n=3, cu=None) == kv.ERR_INVALID_ARG
    assert _store_bf16(g, n=-1) == kv.ERR_INVALID_ARG
    assert _store_bf16(g, n=1 << 31) == kv.ERR_UNSUPPORTED
    assert _store_bf16(g, n=0, ks=None) == kv.OK
    # the quantisation mode is not used: any value is accepted
    assert _store_bf16(kv.Geom(2, 8, 128, 16, 64, 8, 7), n=0) == kv.OK
    assert _store_bf16(kv.Geom(2, 8, 24, 16, 64, 8, 0)) == kv.ERR_INVALID_ARG
    for name in ("kc", "vc", "bt", "lens", "ko", "vo"):
        assert _gather_bf16(g, **{name: None}) == kv.ERR_INVALID_ARG, name
    assert _gather_bf16(g, rows=-1) == kv.ERR_INVALID_ARG
    assert _gather_bf16(g, hs=4) == kv.ERR_INVALID_ARG
    assert _gather_bf16(g, vo=FAKE + 8) == kv.ERR_INVALID_ARG
    assert _gather_bf16(g, ws=None) == kv.ERR_WORKSPACE
    assert _gather_bf16(g, wsb=16) == kv.ERR_WORKSPACE
    assert _gather_bf16(kv.Geom(0, 8, 128, 16, 64, 8, 0), kc=None) == kv.OK


def _append(g, fn="kvc8_append_gather", n=2, **kw):
    a = dict(ks=FAKE, vs=FAKE, ts=g.kv_heads * g.head_dim, hs=g.head_dim, kc=FAKE, vc=FAKE,
             ksc=FAKE, vsc=FAKE, bt=FAKE, cu=FAKE, ctx=FAKE, off=None, ko=FAKE, vo=FAKE, rows=10,
             ots=g.kv_heads * g.head_dim, ohs=g.head_dim, ws=FAKE, wsb=1 << 20)
    a.update(kw)
    lib = kv.load()
    head = [ctypes.byref(g), n, a["ks"], a["vs"], a["ts"], a["hs"], a["kc"], a["vc"], a["ksc"],
            a["vsc"], a["bt"], a["cu"], a["ctx"]]
    tail = [a["ko"], a["vo"], a["rows"], a["ots"], a["ohs"], a["ws"], a["wsb"], None, None]
    if fn == "kvc8_append_gather":
        return lib.kvc8_append_gather(*head, a["off"], *tail)
    return lib.kvc8_append_gather_planned(*head, *tail)


@pytest.mark.parametrize("fn", ["kvc8_append_gather", "kvc8_append_gather_planned"])
def test_append_gather_rejects_bad_arguments(fn):
    g = kv.Geom(2, 8, 128, 16, 64, 8, 0)
    for name in ("ks", "vs", "kc", "vc", "ksc", "vsc", "bt", "ctx", "ko", "vo"):
        assert _append(g, fn, **{name: None}) == kv.ERR_INVALID_ARG, name
    assert _append(g, fn, ts=1028) == kv.ERR_INVALID_ARG
    assert _append(g, fn, ks=FAKE + 2) == kv.ERR_INVALID_ARG
    assert _append(g, fn, ohs=4) == kv.ERR_INVALID_ARG
    assert _append(g, fn, rows=-1) == kv.ERR_INVALID_ARG
    assert _append(g, fn, n=3, cu=None) == kv.ERR_INVALID_ARG  # decode form: one per sequence
    assert _append(g, fn, n=-1) == kv.ERR_INVALID_ARG
    assert _append(g, fn, n=1 << 31) == kv.ERR_UNSUPPORTED
    assert _append(g, fn, n=1 << 27) == kv.ERR_UNSUPPORTED  # 2^27 tokens x 16 rows
    assert _append(kv.Geom(1 << 20, 8, 128, 16, 64, 1 << 8, 0), fn) == kv.ERR_UNSUPPORTED
    assert _append(g, fn, ws=None) == kv.ERR_WORKSPACE
    assert _append(g, fn, wsb=16) == kv.ERR_WORKSPACE
    assert _append(kv.Geom(2, 8, 128, 16, 64, 8, 3), fn) == kv.ERR_INVALID_ARG
    g0 = kv.Geom(0, 8, 128, 16, 64, 8, 0)
    assert _append(g0, fn, n=0, kc=None) == kv.OK  # empty batch: no-op
    assert _append(g0, fn, n=1) == kv.ERR_INVALID_ARG


def test_build_append_metadata_rejects_bad_arguments():
    g = kv.Geom(2, 8, 128, 16, 64, 8, 0)
    lib = kv.load()
    assert lib.kvc8_build_append_metadata(ctypes.byref(g), None, None, None, None, FAKE, 1 << 20,
                                          None, None) == kv.ERR_INVALID_ARG
    assert lib.kvc8_build_append_metadata(ctypes.byref(g), None, FAKE, None, None, FAKE, 8,
                                          None, None) == kv.ERR_WORKSPACE


def test_attention_rejects_bad_arguments():
    lib = kv.load()
    g = kv.Geom(2, 8, 128, 16, 64, 8, 0)
    ws_bytes = kv.kvc8_attention_workspace_bytes(g, 32)
    assert ws_bytes > 0 and kv.kvc8_attention_workspace_bytes(g, 4) == 0

    def call(g=g, hq=32, q=FAKE, qs=32 * 128, qh=128, scale=0.088, out=FAKE, ws=FAKE,
             wsb=ws_bytes, **kw):
        a = dict(kc=FAKE, vc=FAKE, ks=FAKE, vs=FAKE, bt=FAKE, lens=FAKE)
        a.update(kw)
        return lib.kvc8_paged_decode_attention(ctypes.byref(g), hq, q, qs, qh, a["kc"], a["vc"],
                                               a["ks"], a["vs"], a["bt"], a["lens"], scale, out,
                                               qs, qh, ws, wsb, None, None)
    for name in ("kc", "vc", "ks", "vs", "bt", "lens"):
        assert call(**{name: None}) == kv.ERR_INVALID_ARG, name
    assert call(q=None) == kv.ERR_INVALID_ARG
    assert call(out=None) == kv.ERR_INVALID_ARG
    assert call(hq=30) == kv.ERR_INVALID_ARG           # not a multiple of the kv heads
    assert call(hq=72) == kv.ERR_UNSUPPORTED            # group of 9
    assert call(qs=100) == kv.ERR_INVALID_ARG
    assert call(q=FAKE + 8) == kv.ERR_INVALID_ARG
    assert call(scale=float("inf")) == kv.ERR_INVALID_ARG
    assert call(ws=None) == kv.ERR_WORKSPACE
    assert call(wsb=ws_bytes - 1) == kv.ERR_WORKSPACE
    assert call(g=kv.Geom(2, 8, 96, 16, 64, 8, 0), qh=96, qs=32 * 96) == kv.ERR_UNSUPPORTED
    assert call(g=kv.Geom(2, 8, 128, 8, 64, 8, 0)) == kv.ERR_UNSUPPORTED  # block of 8
    assert call(g=kv.Geom(0, 8, 128, 16, 64, 8, 0), q=None) == kv.OK  # empty batch
